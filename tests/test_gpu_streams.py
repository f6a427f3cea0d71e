"""The operators on a caller's stream and inside CUDA graphs.

Every entry point enqueues its work on the stream it is given (the current
PyTorch stream by default) and makes no synchronising call, so (a) work the
caller queued on a side stream just before the call is ordered before it,
and (b) after one eager call on the device, a sequence of operators can be
captured into a CUDA graph and replayed: the replay must give the eager
results bit for bit, and again after new data is copied into the graph's
input buffers."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from tensor_matmul_collective_gb300 import coc
from tensor_matmul_collective_gb300 import workloads as wl

from gpu_util import assert_close, bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
BF16, F16 = torch.bfloat16, torch.float16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_matmul_collective_gb300 import build
    build.build()
    coc.lib()
    yield
    coc.sync_status()


def _rp(R, m, n, ks, dt, seed):
    return wl.RowParallel(R=R, m=m, n=n, k_shard=ks, dtype=dt, x_dist="normal(0,1)", w_dist="normal(0,0.02)",
                          seed=seed).make()


def test_side_stream_orders_after_the_callers_work():
    R, m, n, ks = 4, 512, 384, 256
    xs, ws = _rp(R, m, n, ks, BF16, 31)
    ref = orc.matmul_all_reduce(orc.BF16, bits(xs), bits(ws))
    src = [x.to(DEV) for x in xs]
    wd = [w.to(DEV) for w in ws]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        # the inputs are produced on the side stream immediately before the call
        xd = [torch.empty_like(x) for x in src]
        for a, b in zip(xd, src):
            a.copy_(b)
        outs = coc.matmul_all_reduce(xd, wd, chunks=2)
        got = [o.clone() for o in outs]
        routs = [torch.full((m // R, n), float("nan"), dtype=BF16, device=DEV) for _ in range(R)]
    # explicit stream argument, called from the default stream
    coc.matmul_reduce_scatter(xd, wd, routs, stream=s)
    s.synchronize()
    coc.sync_status(s)
    for r in range(R):
        assert_close(got[r], ref, R * ks, f"AR rank {r}")
        assert torch.equal(routs[r], got[0][r * (m // R):(r + 1) * (m // R)])


def _graph_suite():
    """Static buffers for AR, RS, AG-V2, w8A16 (pre-pass and fused paths),
    MoE top-2 with the gated combine and a decode-sized AR, and a function
    that runs all of them."""
    R = 4
    xs, ws = _rp(R, 512, 384, 256, BF16, 32)
    ar_x, ar_w = [x.to(DEV) for x in xs], [w.to(DEV) for w in ws]
    ar_out = [torch.empty(512, 384, dtype=BF16, device=DEV) for _ in range(R)]
    rs_out = [torch.empty(128, 384, dtype=BF16, device=DEV) for _ in range(R)]
    cs = wl.ColumnParallelSP(R=R, m_shard=128, n_shard=320, k=256, dtype=BF16, x_dist="normal(0,1)",
                             w_dist="normal(0,0.02)", seed=33)
    cxs, cws = cs.make()
    ag_x, ag_w = [x.to(DEV) for x in cxs], [w.to(DEV) for w in cws]
    ag_out = [torch.empty(512, 320, dtype=BF16, device=DEV) for _ in range(R)]
    ag_g = [torch.empty(512, 256, dtype=BF16, device=DEV) for _ in range(R)]
    w8 = {}
    for m in (2048, 256):   # from 2048 rows the pre-pass path, below it the fused one
        s8 = wl.W8A16(R=R, m=m, n=256, k_shard=128, group=64, seed=34 + m)
        x8, q8, c8 = s8.make("group")
        w8[m] = ([x.to(DEV) for x in x8], [q.to(DEV) for q in q8], [c.to(DEV) for c in c8],
                 [torch.empty(m, 256, dtype=F16, device=DEV) for _ in range(R)])
    ms = wl.MoEDispatch(R=R, T=200, h=128, f=136, e_loc=2, seed=35)
    mxs, _, mws = ms.make()
    ti, tg = ms.routing_topk(2)
    mo_x = [x.to(DEV) for x in mxs]
    mo_i, mo_g = [i.to(DEV) for i in ti], [g.to(DEV) for g in tg]
    mo_w = torch.stack(mws).to(DEV)
    mo = list(coc.moe_topk_grouped_matmul_combine(mo_x, mo_i, mo_g, mo_w, ms.e_loc))   # buffers
    dxs, dws = _rp(R, 16, 512, 128, BF16, 39)   # decode-sized: the rank-split path and its scratch
    dec_x, dec_w = [x.to(DEV) for x in dxs], [w.to(DEV) for w in dws]
    dec_out = [torch.empty(16, 512, dtype=BF16, device=DEV) for _ in range(R)]
    inputs = ar_x + ag_x + [t for m in w8 for t in w8[m][0]] + mo_x + dec_x
    outputs = ar_out + rs_out + ag_out + ag_g + [t for m in w8 for t in w8[m][3]] + mo[0] + [mo[3]] + dec_out

    def run():
        coc.matmul_all_reduce(ar_x, ar_w, ar_out, chunks=2)
        coc.matmul_reduce_scatter(ar_x, ar_w, rs_out, chunks=4)
        coc.all_gather_matmul_v2(ag_x, ag_w, ag_out, ag_g, chunks=2)
        for m in w8:
            x8, q8, c8, o8 = w8[m]
            coc.matmul_all_reduce_w8a16(x8, q8, c8, "group", 64, o8)
        coc.moe_topk_grouped_matmul_combine(mo_x, mo_i, mo_g, mo_w, ms.e_loc, xd=mo[2], y=mo[1], y_tok=mo[0],
                                            counts=mo[3], offsets=mo[4])
        coc.matmul_all_reduce(dec_x, dec_w, dec_out)
    return run, inputs, outputs


def test_cuda_graph_capture_and_replay():
    run, inputs, outputs = _graph_suite()
    run()                                   # eager: device state, pools, kernel attributes
    torch.cuda.synchronize()
    coc.sync_status()
    eager = [o.clone() for o in outputs]

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for o in outputs:
        o.fill_(-7)                         # nothing stale can pass for a result
    g.replay()
    torch.cuda.synchronize()
    coc.sync_status()
    for i, (a, b) in enumerate(zip(outputs, eager)):
        assert torch.equal(a, b), f"replay output {i} differs from the eager call"

    # new activations in the same buffers: replay == eager on the new data
    gen = torch.Generator(device="cpu").manual_seed(36)
    for t in inputs:
        t.copy_(torch.randn(t.shape, generator=gen).to(t.dtype))
    g.replay()
    torch.cuda.synchronize()
    coc.sync_status()
    replayed = [o.clone() for o in outputs]
    run()
    torch.cuda.synchronize()
    coc.sync_status()
    for i, (a, b) in enumerate(zip(replayed, outputs)):
        assert torch.equal(a, b), f"replay on new inputs: output {i} differs from the eager call"
    assert not all(torch.equal(a, b) for a, b in zip(replayed, eager))
    del g


def test_graph_replay_matches_oracle():
    """A captured AllReduce on fresh inputs against the fp64 oracle (the replay
    computes, it does not return a stored result)."""
    R, m, n, ks = 2, 256, 136, 200
    xs, ws = _rp(R, m, n, ks, BF16, 37)
    xd, wd = [x.to(DEV) for x in xs], [w.to(DEV) for w in ws]
    outs = [torch.empty(m, n, dtype=BF16, device=DEV) for _ in range(R)]
    coc.matmul_all_reduce(xd, wd, outs)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        coc.matmul_all_reduce(xd, wd, outs)
    xs2, _ = _rp(R, m, n, ks, BF16, 38)
    for a, b in zip(xd, xs2):
        a.copy_(b.to(DEV))
    g.replay()
    torch.cuda.synchronize()
    coc.sync_status()
    ref = orc.matmul_all_reduce(orc.BF16, bits(xs2), bits(ws))
    for r in range(R):
        assert_close(outs[r], ref, R * ks, f"rank {r}")
    assert np.isfinite(ref).all()
    del g
