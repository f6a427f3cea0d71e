"""No device allocation on the hot path.

The operators own no per-call memory: the status block is created by the
first call on a device, and the scratch some calls need (the rank-split fp32
parts, the MoE routing tables, the w8A16 pre-pass weight, the stacked X of a
decode-sized AllGather) lives in a workspace the library keeps per stream,
sized by the first call that needs it.  The library counts every device allocation it makes
(coc_debug_alloc_count); after one warm-up call of every operator, further
calls of the same shapes on the same stream must leave the count unchanged,
and so must replays of a CUDA graph that captured them."""
import os

import pytest
import torch

from tensor_matmul_collective_gb300 import coc
from tensor_matmul_collective_gb300 import workloads as wl

from gpu_util import DEV, to_dev

pytestmark = pytest.mark.gpu
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


def _calls():
    """One closure per operator and schedule (each with its outputs preallocated)."""
    calls = {}
    rp = lambda R, m, n, ks, dt=BF16, seed=1: wl.RowParallel(  # noqa: E731
        R=R, m=m, n=n, k_shard=ks, dtype=dt, x_dist="uniform[-1,1]", w_dist="uniform[-1,1]", seed=seed).make()
    # AllReduce: 2-SM tiles, single-CTA tiles, the rank split (decode-sized m)
    for name, (R, m, n, ks) in {"ar_pair": (8, 512, 512, 128), "ar_single": (4, 128, 520, 64),
                                "ar_split": (8, 16, 1024, 256)}.items():
        xs, ws = map(to_dev, rp(R, m, n, ks))
        outs = [torch.empty(m, n, dtype=BF16, device=DEV) for _ in range(R)]
        calls[name] = lambda xs=xs, ws=ws, o=outs: coc.matmul_all_reduce(xs, ws, o, chunks=2)
    # the column-slab kernel (decode-sized m), unsplit and split over clusters
    for name, plan in (("ar_slab", (2, 1, 2)), ("ar_slab_split", (2, 2, 2))):
        xs, ws = map(to_dev, rp(8, 16, 2048, 256))
        outs = [torch.empty(16, 2048, dtype=BF16, device=DEV) for _ in range(8)]

        def slab_call(xs=xs, ws=ws, o=outs, plan=plan):
            env = {"COC_SLAB": "1", "COC_SLAB_BOXES": str(plan[0]), "COC_SLAB_SPLIT": str(plan[1]),
                   "COC_SLAB_KPS": str(plan[2])}
            prev = {k: os.environ.get(k) for k in env}
            os.environ.update(env)
            try:
                coc.matmul_all_reduce(xs, ws, o)
            finally:
                for k, v in prev.items():
                    if v is None:
                        del os.environ[k]
                    else:
                        os.environ[k] = v
        calls[name] = slab_call
    xs, ws = map(to_dev, rp(8, 64, 1024, 256))
    rso = [torch.empty(8, 1024, dtype=BF16, device=DEV) for _ in range(8)]
    calls["rs_split"] = lambda: coc.matmul_reduce_scatter(xs, ws, rso)
    xs2, ws2 = map(to_dev, rp(4, 512, 264, 128, seed=2))
    rso2 = [torch.empty(128, 264, dtype=BF16, device=DEV) for _ in range(4)]
    calls["rs"] = lambda: coc.matmul_reduce_scatter(xs2, ws2, rso2, chunks=4)
    plain = torch.empty(512, 264, dtype=BF16, device=DEV)
    calls["plain"] = lambda: coc.matmul(xs2, ws2, plain)
    wnk = [w.t().contiguous() for w in ws2]
    nko = [torch.empty(512, 264, dtype=BF16, device=DEV) for _ in range(4)]
    calls["ar_nk"] = lambda: coc.fused_matmul("all_reduce", xs2, wnk, w_layout="nk", outs=nko)
    # AllGather, AllGather-V2, weight gradient
    s = wl.ColumnParallelSP(R=4, m_shard=64, n_shard=264, k=192, dtype=BF16, x_dist="uniform[-1,1]",
                            w_dist="uniform[-1,1]", seed=3)
    ax, aw = map(to_dev, s.make())
    ago = [torch.empty(256, 264, dtype=BF16, device=DEV) for _ in range(4)]
    agg = [torch.empty(256, 192, dtype=BF16, device=DEV) for _ in range(4)]
    calls["ag"] = lambda: coc.all_gather_matmul(ax, aw, ago)
    calls["ag_v2"] = lambda: coc.all_gather_matmul_v2(ax, aw, ago, agg)
    # decode-sized AllGather (column-slab kernel): V1 stacks X in the stream's workspace
    s8 = wl.ColumnParallelSP(R=8, m_shard=8, n_shard=1024, k=512, dtype=BF16, x_dist="uniform[-1,1]",
                             w_dist="uniform[-1,1]", seed=6)
    dx8, dw8 = map(to_dev, s8.make())
    do8 = [torch.empty(64, 1024, dtype=BF16, device=DEV) for _ in range(8)]
    dg8 = [torch.empty(64, 512, dtype=BF16, device=DEV) for _ in range(8)]
    calls["ag_slab"] = lambda: coc.all_gather_matmul(dx8, dw8, do8)
    calls["ag_slab_v2"] = lambda: coc.all_gather_matmul_v2(dx8, dw8, do8, dg8)
    dws = [torch.empty(264, 192, dtype=BF16, device=DEV) for _ in range(4)]
    calls["wgrad"] = lambda: coc.weight_grad(ago, agg, dws)
    # w8A16: the schedules without scratch (in-kernel dequantisation to shared
    # or to tensor memory) and the pre-pass schedule, whose dequantised weight
    # lives in the stream's workspace
    for name, m, path in (("w8_fused", 256, "fused"), ("w8_ts", 256, "ts"), ("w8_prepass", 2048, "prepass")):
        w8 = wl.W8A16(R=4, m=m, n=256, k_shard=256, group=128, seed=4)
        x8, q8, sc8 = w8.make("group")
        x8, q8, sc8 = to_dev(x8), to_dev(q8), to_dev(sc8)
        o8 = [torch.empty(m, 256, dtype=F16, device=DEV) for _ in range(4)]

        def w8call(x8=x8, q8=q8, sc8=sc8, o8=o8, path=path):
            prev = os.environ.get("COC_W8_PATH")
            if path is not None:
                os.environ["COC_W8_PATH"] = path
            try:
                coc.matmul_all_reduce_w8a16(x8, q8, sc8, "group", 128, o8)
            finally:
                if path is not None:
                    if prev is None:
                        del os.environ["COC_W8_PATH"]
                    else:
                        os.environ["COC_W8_PATH"] = prev
        calls[name] = w8call
    # MoE: dispatch + GroupedMatMul, the fused top-1 combine, top-2 with the gated combine
    moe = wl.MoEDispatch(R=4, T=200, h=128, f=264, e_loc=2, seed=5)
    mx, mi, mw = moe.make()
    mx, mi, mw = to_dev(mx), to_dev(mi), torch.stack(mw).to(DEV)
    y, xd, cnt, off = coc.moe_dispatch_grouped_matmul(mx, mi, mw, moe.e_loc)
    calls["moe"] = lambda: coc.moe_dispatch_grouped_matmul(mx, mi, mw, moe.e_loc, xd=xd, y=y, counts=cnt, offsets=off)
    ytok = [torch.empty(200, 264, dtype=BF16, device=DEV) for _ in range(4)]
    calls["moe_combine"] = lambda: coc.moe_dispatch_grouped_matmul(mx, mi, mw, moe.e_loc, xd=xd, y=ytok, counts=cnt,
                                                                   offsets=off, combine=True)
    ti, tg = moe.routing_topk(2)
    ti, tg = to_dev(ti), to_dev(tg)
    yt2, y2, xd2, c2, o2 = coc.moe_topk_grouped_matmul_combine(mx, ti, tg, mw, moe.e_loc)
    calls["moe_top2"] = lambda: coc.moe_topk_grouped_matmul_combine(mx, ti, tg, mw, moe.e_loc, xd=xd2, y=y2, y_tok=yt2,
                                                                    counts=c2, offsets=o2)
    return calls


def test_steady_state_calls_allocate_nothing():
    calls = _calls()
    for fn in calls.values():       # warm-up: sizes the stream's workspace
        fn()
    coc.sync_status()
    n0 = coc.alloc_count()
    for _ in range(3):
        for name, fn in calls.items():
            fn()
            assert coc.alloc_count() == n0, f"{name} allocated device memory in a steady-state call"
    coc.sync_status()
    assert coc.alloc_count() == n0


def test_other_stream_gets_its_own_workspace_then_allocates_nothing():
    calls = _calls()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        calls["ar_split"]()
        calls["moe"]()
        n0 = coc.alloc_count()
        for _ in range(3):
            calls["ar_split"]()
            calls["moe"]()
    torch.cuda.current_stream().wait_stream(s)
    coc.sync_status(s)
    assert coc.alloc_count() == n0


def test_graph_replays_allocate_nothing():
    calls = _calls()
    calls["ar_split"]()
    calls["w8_prepass"]()
    calls["ag_slab"]()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        calls["ar_split"]()
        calls["w8_prepass"]()
        calls["moe"]()
        calls["ag_slab"]()
    n0 = coc.alloc_count()
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    coc.sync_status()
    assert coc.alloc_count() == n0
    del g
