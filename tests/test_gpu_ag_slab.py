"""ALL_GATHER_MATMUL and ALL_GATHER_MATMUL_V2 at decode-sized gathered m
(R m_shard <= 128) through the column-slab kernel: a unit is one column slab
of one rank's output, summed over the full k in one CTA or in a cluster of 2
or 4 CTAs that add their parts in part order.  A copy kernel first stacks
the R shards of X into V2's gathered outputs (or, for V1 and for V2 with
every copy skipped, into the call's scratch), and the slab kernel reads A
from the first of them.

COC_SLAB=1 with COC_SLAB_BOXES / COC_SLAB_SPLIT / COC_SLAB_KPS pins the
schedule.  Checked against the fp64 oracle element by element (ragged n_shard
and k, an m_shard that is not a power of two, one rank, k x n and n x k
weight storage, both 16-bit types), plus: the V1 and V2 products
bit-identical, the gathered copies bit-exact, the unsplit slab bit-identical
to the persistent kernel (the same accumulation order: k ascending, 16 k per
MMA), one-hot weights reproducing gathered X columns bit for bit, skipped
gathered copies (A from a later rank's copy, or from scratch) left alone,
an injected timeout reported, and the default schedule at the decode
layer's shapes."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from tensor_matmul_collective_gb300 import coc
from tensor_matmul_collective_gb300 import workloads as wl

from gpu_util import assert_close, bits, to_dev

pytestmark = pytest.mark.gpu
BF16, F16 = torch.bfloat16, torch.float16
CODE = {F16: orc.F16, BF16: orc.BF16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_matmul_collective_gb300 import build
    build.build()
    coc.lib()
    yield
    coc.sync_status()


def _plan(monkeypatch, plan):
    b, sp, kps = plan
    for k, v in (("COC_SLAB", 1), ("COC_SLAB_BOXES", b), ("COC_SLAB_SPLIT", sp), ("COC_SLAB_KPS", kps)):
        monkeypatch.setenv(k, str(v))


def _data(R, ms, ns, k, dt, seed):
    return wl.ColumnParallelSP(R=R, m_shard=ms, n_shard=ns, k=k, dtype=dt, x_dist="normal(0,1)",
                               w_dist="normal(0,0.02)", seed=seed).make()


CASES = [
    # R, m_shard, n_shard, k, dtype, (boxes, split, kps)
    (8, 8, 7168, 1024, BF16, (2, 1, 2)),     # the decode layer's 8 rows per rank: 448 slabs, several per CTA
    (8, 16, 1024, 512, F16, (2, 2, 2)),      # 64 slabs in clusters of 2
    (4, 8, 1000, 200, BF16, (1, 2, 2)),      # k ends inside a k-block; 64-column slabs split in two, ragged last slab
    (2, 64, 2048, 512, F16, (2, 4, 1)),      # 128 rows (four row quadrants), clusters of 4
    (8, 16, 512, 4096, BF16, (2, 4, 2)),     # long k, clusters of 4
    (4, 24, 1104, 64, F16, (1, 1, 1)),       # m_shard 24, one k-block, 64-column slabs
    (2, 8, 20000, 64, BF16, (2, 1, 1)),      # several slabs per CTA (both accumulator buffers)
    (1, 128, 520, 256, BF16, (2, 2, 2)),     # one rank
]


@pytest.mark.parametrize("R,ms,ns,k,dt,plan", CASES)
def test_ag_slab_parity(R, ms, ns, k, dt, plan, monkeypatch):
    _plan(monkeypatch, plan)
    xs, ws = _data(R, ms, ns, k, dt, 17 * ms + ns)
    dx, dw = to_dev(xs), to_dev(ws)
    v1 = coc.all_gather_matmul(dx, dw)
    v2, gathered = coc.all_gather_matmul_v2(dx, dw)
    coc.sync_status()
    bx, bw = bits(xs), bits(ws)
    xg = orc.all_gather(bx)
    for r in range(R):
        assert_close(v1[r], orc.all_gather_matmul(CODE[dt], bx, bw, r), k, f"AG slab rank {r}")
        assert torch.equal(v1[r], v2[r]), f"V1 and V2 products differ on rank {r}"
        assert np.array_equal(wl.bits16(gathered[r].cpu()), xg), f"gathered copy {r} is not bit-exact"


@pytest.mark.parametrize("plan", [(2, 1, 2), (1, 2, 4), (2, 4, 1)])
def test_ag_slab_nk_weights_match_kn_bits(plan, monkeypatch):
    """n_shard x k weight storage (B read K-major) gives the k x n bits."""
    _plan(monkeypatch, plan)
    R, ms, ns, k = 8, 8, 1000, 512
    xs, ws = _data(R, ms, ns, k, BF16, 91)
    dx, dw = to_dev(xs), to_dev(ws)
    kn = coc.all_gather_matmul(dx, dw)
    nk, g = coc.fused_matmul("all_gather_v2", dx, [w.t().contiguous() for w in dw], w_layout="nk")
    coc.sync_status()
    for a, b in zip(kn, nk):
        assert torch.equal(a, b)
    xg = orc.all_gather(bits(xs))
    for t in g:
        assert np.array_equal(wl.bits16(t.cpu()), xg)
    assert_close(kn[5], orc.all_gather_matmul(orc.BF16, bits(xs), bits(ws), 5), k, "k x n")


@pytest.mark.parametrize("R,ms,ns,k", [(8, 8, 4096, 512), (4, 24, 1000, 200), (2, 64, 2048, 128)])
def test_unsplit_ag_slab_gives_the_persistent_kernels_bits(R, ms, ns, k, monkeypatch):
    """One CTA per slab adds the MMAs in the persistent kernel's order (k
    ascending, 16 k each) into one accumulator: the same bits."""
    xs, ws = _data(R, ms, ns, k, BF16, 5 * ms + k)
    dx, dw = to_dev(xs), to_dev(ws)
    _plan(monkeypatch, (2, 1, 2))
    slab = [t.clone() for t in coc.all_gather_matmul(dx, dw)]
    monkeypatch.setenv("COC_SLAB", "0")
    tile = coc.all_gather_matmul(dx, dw)
    coc.sync_status()
    for a, b in zip(slab, tile):
        assert torch.equal(a, b)


@pytest.mark.parametrize("plan", [(2, 1, 2), (2, 4, 1), (1, 2, 1)])
def test_ag_slab_one_hot_is_exact(plan, monkeypatch):
    """Weight 1.0 at one k per column of each rank's W: rank r's output must
    be the gathered X's columns sel_r bit for bit (a misplaced source rank
    row block, k-block, column or rank output shows)."""
    _plan(monkeypatch, plan)
    R, ms, ns, k = 8, 16, 1000, 256
    gen = torch.Generator().manual_seed(4)
    xs = [torch.randn(ms, k, generator=gen).to(BF16) for _ in range(R)]
    xg = torch.cat(xs, 0)
    ws, sels = [], []
    for r in range(R):
        sel = np.random.default_rng(40 + r).integers(0, k, ns)
        W = torch.zeros(k, ns)
        W[sel, torch.arange(ns)] = 1.0
        ws.append(W.to(BF16))
        sels.append(sel)
    outs = coc.all_gather_matmul(to_dev(xs), to_dev(ws))
    coc.sync_status()
    for r in range(R):
        assert torch.equal(outs[r].cpu(), xg[:, sels[r]]), f"rank {r}"


@pytest.mark.parametrize("keep", [(3,), (), (1, 6)], ids=["one", "none", "two"])
def test_ag_slab_skipped_copies(keep, monkeypatch):
    """V2 with some gathered entries None: the kept copies are exact, the
    skipped buffers untouched, and the products those of V1 (A read from
    the first kept copy, or from scratch when none is kept)."""
    _plan(monkeypatch, (2, 2, 2))
    R, ms, ns, k = 8, 8, 1000, 512
    xs, ws = _data(R, ms, ns, k, BF16, 47)
    dx, dw = to_dev(xs), to_dev(ws)
    canary = torch.full((R * ms, k), 7.0, dtype=BF16, device=dx[0].device)
    bufs = [canary.clone() for _ in range(R)]
    outs, _ = coc.all_gather_matmul_v2(dx, dw, gathered=[bufs[r] if r in keep else None for r in range(R)])
    v1 = coc.all_gather_matmul(dx, dw)
    coc.sync_status()
    xg = orc.all_gather(bits(xs))
    for r in range(R):
        assert torch.equal(outs[r], v1[r])
        if r in keep:
            assert np.array_equal(wl.bits16(bufs[r].cpu()), xg)
        else:
            assert torch.equal(bufs[r], canary), f"skipped copy {r} was written"
    assert_close(outs[2], orc.all_gather_matmul(orc.BF16, bits(xs), bits(ws), 2), k, "skipped copies")


def test_ag_slab_injected_timeout_is_reported_and_device_stays_usable(monkeypatch):
    _plan(monkeypatch, (2, 2, 2))
    R, ms, ns, k = 8, 8, 1024, 256
    xs, ws = _data(R, ms, ns, k, BF16, 43)
    dx, dw = to_dev(xs), to_dev(ws)
    coc.inject_timeout(True)
    try:
        coc.all_gather_matmul_v2(dx, dw)
        with pytest.raises(coc.CocError) as ei:
            coc.sync_status()
        assert ei.value.status == coc.ERR_TIMEOUT
    finally:
        coc.inject_timeout(False)
    coc.sync_status()
    outs, g = coc.all_gather_matmul_v2(dx, dw)
    coc.sync_status()
    assert_close(outs[6], orc.all_gather_matmul(orc.BF16, bits(xs), bits(ws), 6), k, "after timeout")
    assert np.array_equal(wl.bits16(g[2].cpu()), orc.all_gather(bits(xs)))


@pytest.mark.parametrize("ms,ns,k", [(8, 7168, 8192), (16, 1536, 4096)])
def test_ag_decode_default_schedule(ms, ns, k, monkeypatch):
    """The default schedule at the decode layer's shapes (8 ranks) gives the
    oracle's values on the first and last rank, for sampled rows."""
    for v in ("COC_SLAB", "COC_SLAB_BOXES", "COC_SLAB_SPLIT", "COC_SLAB_KPS"):
        monkeypatch.delenv(v, raising=False)
    R = 8
    xs, ws = _data(R, ms, ns, k, BF16, ms + k)
    outs, g = coc.all_gather_matmul_v2(to_dev(xs), to_dev(ws))
    coc.sync_status()
    bx, bw = bits(xs), bits(ws)
    rows = np.array([0, ms - 1, ms, 3 * ms + 5, R * ms - 1])
    for r in (0, R - 1):
        ref = orc.all_gather_matmul(orc.BF16, bx, bw, r, rows=rows)
        assert_close(outs[r][torch.as_tensor(rows)], ref, k, f"decode AG rank {r}")
    assert np.array_equal(wl.bits16(g[3].cpu()), orc.all_gather(bx))
