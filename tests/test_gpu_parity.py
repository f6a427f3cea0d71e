"""GPU parity of the fused kernels against the fp64 CPU oracle (element by
element), on small seeded shapes that span several tiles and ragged tails,
plus the exact special inputs (one-hot weights, small integers, zeros) that
are checked bitwise.  Every call goes through the C ABI."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from tensor_matmul_collective_gb300 import coc
from tensor_matmul_collective_gb300 import workloads as wl

from gpu_util import DEV, assert_close, bits, to_dev

pytestmark = pytest.mark.gpu

F16, BF16 = torch.float16, torch.bfloat16
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


def _row_parallel(R, m, n, ks, dt, seed, dist="uniform[-1,1]"):
    return wl.RowParallel(R=R, m=m, n=n, k_shard=ks, dtype=dt, x_dist=dist, w_dist=dist, seed=seed).make()


# ------------------------------------------------------------- AllReduce ---

@pytest.mark.parametrize("det", [0, 1])
def test_tiny_allreduce_config(det):
    """R = 2, fp16 64 x 128 per rank (k = 256), chunks 2, U[-1, 1], seed 0."""
    s = wl.TINY_AR
    xs, ws = s.make()
    outs = coc.matmul_all_reduce(to_dev(xs), to_dev(ws), chunks=2, deterministic=bool(det))
    coc.sync_status()
    ref = orc.matmul_all_reduce(orc.F16, bits(xs), bits(ws))
    for r, o in enumerate(outs):
        assert_close(o, ref, s.K, f"rank {r}")
        assert torch.equal(o, outs[0])


AR_CASES = [
    # R, m, n, k_shard, dtype, chunks
    (4, 200, 136, 72, BF16, 1),      # ragged m, n and k (k tail inside one k-block)
    (2, 384, 520, 200, F16, 2),      # 3 m-tiles, 3 n-tiles with tail
    (8, 256, 512, 128, BF16, 8),     # chunks smaller than a tile
    (1, 130, 264, 64, BF16, 1),      # R = 1: plain GEMM
    (8, 1024, 256, 96, BF16, 4),     # chunk-major order (2 m-tiles per chunk)
    (2, 64, 8, 8, F16, 1),           # one tiny tile
]


@pytest.mark.parametrize("R,m,n,ks,dt,chunks", AR_CASES)
def test_allreduce_parity(R, m, n, ks, dt, chunks):
    xs, ws = _row_parallel(R, m, n, ks, dt, seed=R * 1000 + m)
    outs = coc.matmul_all_reduce(to_dev(xs), to_dev(ws), chunks=chunks)
    coc.sync_status()
    ref = orc.matmul_all_reduce(CODE[dt], bits(xs), bits(ws))
    for r, o in enumerate(outs):
        assert_close(o, ref, R * ks, f"AR rank {r}")
        assert torch.equal(o, outs[0]), "AllReduce copies must be bit-identical"


def test_plain_matmul_is_allreduce_copy():
    xs, ws = _row_parallel(4, 300, 264, 72, BF16, seed=7)
    dx, dw = to_dev(xs), to_dev(ws)
    outs = coc.matmul_all_reduce(dx, dw, chunks=1, deterministic=True)
    plain = coc.matmul(dx, dw)
    coc.sync_status()
    assert torch.equal(plain, outs[0])


def test_chunk_count_does_not_change_bits():
    xs, ws = _row_parallel(8, 1024, 512, 64, BF16, seed=11, dist="normal(0,1)")
    dx, dw = to_dev(xs), to_dev(ws)
    base = coc.matmul_all_reduce(dx, dw, chunks=1, deterministic=True)[0].clone()
    for c in (2, 4, 8):
        for det in (True, False):
            o = coc.matmul_all_reduce(dx, dw, chunks=c, deterministic=det)
            assert all(torch.equal(t, base) for t in o), (c, det)
    coc.sync_status()


def test_zero_k_writes_zeros():
    R, m, n = 2, 96, 136
    xs = [torch.empty(m, 0, dtype=BF16, device=DEV) for _ in range(R)]
    ws = [torch.empty(0, n, dtype=BF16, device=DEV) for _ in range(R)]
    outs = [torch.full((m, n), 7.0, dtype=BF16, device=DEV) for _ in range(R)]
    coc.matmul_all_reduce(xs, ws, outs)
    coc.sync_status()
    assert all(torch.count_nonzero(o).item() == 0 for o in outs)


@pytest.mark.parametrize("dt,lim", [(F16, 4), (BF16, 1)])
def test_small_integers_bitwise(dt, lim):
    # Integer inputs with K = 512: every partial sum is an integer far below
    # 2^24 (exact in fp32) and the results stay inside the range where the
    # output type holds every integer (2048 for fp16, 256 for bf16).
    g = torch.Generator().manual_seed(5)
    R, m, n, ks = 4, 160, 264, 128
    xs = [torch.randint(-lim, lim + 1, (m, ks), generator=g).to(dt) for _ in range(R)]
    ws = [torch.randint(-lim, lim + 1, (ks, n), generator=g).to(dt) for _ in range(R)]
    ref = orc.matmul_all_reduce(CODE[dt], bits(xs), bits(ws))
    assert np.abs(ref).max() < (2048 if dt == F16 else 256)
    outs = coc.matmul_all_reduce(to_dev(xs), to_dev(ws))
    coc.sync_status()
    for o in outs:
        assert np.array_equal(o.cpu().double().numpy(), ref)


def _one_hot_weights(R, ks, n, perm_seed):
    """W_0 = column-permuted one-hot block (column j selects row perm[j] of X_0);
    W_r = 0 for r > 0.  Every output element receives exactly one product."""
    rng = np.random.default_rng(perm_seed)
    sel = rng.integers(0, ks, n)
    W0 = torch.zeros(ks, n)
    W0[sel, torch.arange(n)] = 1.0
    return sel, [W0] + [torch.zeros(ks, n) for _ in range(R - 1)]


@pytest.mark.parametrize("dt", [F16, BF16])
def test_one_hot_routing_allreduce_and_reduce_scatter(dt):
    R, m, n, ks = 4, 256, 392, 136
    xs, _ = _row_parallel(R, m, n, ks, dt, seed=21, dist="normal(0,1)")
    sel, Ws = _one_hot_weights(R, ks, n, 3)
    ws = [w.to(dt) for w in Ws]
    expect = xs[0][:, sel]                               # exact: one product per element
    outs = coc.matmul_all_reduce(to_dev(xs), to_dev(ws), chunks=2)
    rs = coc.matmul_reduce_scatter(to_dev(xs), to_dev(ws), chunks=2)
    coc.sync_status()
    for o in outs:
        assert torch.equal(o.cpu(), expect)
    for r, o in enumerate(rs):
        assert torch.equal(o.cpu(), expect[r * (m // R):(r + 1) * (m // R)])


# --------------------------------------------------------- ReduceScatter ---

RS_CASES = [
    # R, m, n, k_shard, dtype, chunks     (m / R rows per rank)
    (2, 48, 136, 72, BF16, 2),       # 24 rows per rank: 8-row store boxes
    (4, 512, 264, 136, F16, 4),      # 128 rows per rank
    (8, 1024, 256, 64, BF16, 8),     # tiles aligned with rank blocks
    (8, 320, 72, 24, BF16, 1),       # 40 rows per rank, one ragged n-tile
]


@pytest.mark.parametrize("R,m,n,ks,dt,chunks", RS_CASES)
def test_reduce_scatter_parity(R, m, n, ks, dt, chunks):
    xs, ws = _row_parallel(R, m, n, ks, dt, seed=R * 77 + m)
    outs = coc.matmul_reduce_scatter(to_dev(xs), to_dev(ws), chunks=chunks)
    coc.sync_status()
    for r, o in enumerate(outs):
        ref = orc.matmul_reduce_scatter(CODE[dt], bits(xs), bits(ws), r)
        assert_close(o, ref, R * ks, f"RS rank {r}")


def test_reduce_scatter_concat_equals_allreduce_bits():
    xs, ws = _row_parallel(8, 1024, 264, 72, BF16, seed=31, dist="normal(0,1)")
    dx, dw = to_dev(xs), to_dev(ws)
    ar = coc.matmul_all_reduce(dx, dw, chunks=4, deterministic=True)
    rs = coc.matmul_reduce_scatter(dx, dw, chunks=4, deterministic=True)
    coc.sync_status()
    assert torch.equal(torch.cat(rs, 0), ar[0])


# ------------------------------------------------------------- AllGather ---

AG_CASES = [
    # R, m_shard, n_shard, k, dtype, chunks
    (2, 40, 72, 136, BF16, 1),       # 80 gathered rows: the column-slab kernel on the stacked X
    (4, 128, 264, 64, F16, 2),       # aligned shards read in place, ragged n
    (8, 24, 256, 72, BF16, 8),       # 192 gathered rows from 24-row shards (X stacked), 8 chunks
    (1, 136, 40, 200, BF16, 1),      # R = 1
    (8, 136, 248, 136, BF16, 2),     # 1088 rows, X stacked: the last pair tile's second CTA starts past m
    (4, 200, 136, 72, F16, 1),       # 800 rows of 200-row shards, ragged k
]


@pytest.mark.parametrize("R,ms,ns,k,dt,chunks", AG_CASES)
def test_all_gather_matmul_v2_parity(R, ms, ns, k, dt, chunks):
    shape = wl.ColumnParallelSP(R=R, m_shard=ms, n_shard=ns, k=k, dtype=dt, x_dist="uniform[-1,1]",
                                w_dist="uniform[-1,1]", seed=R * 13 + ms)
    xs, ws = shape.make()
    outs, gathered = coc.all_gather_matmul_v2(to_dev(xs), to_dev(ws), chunks=chunks)
    outs1 = coc.all_gather_matmul(to_dev(xs), to_dev(ws), chunks=chunks)
    coc.sync_status()
    xg = orc.all_gather(bits(xs))
    for r in range(R):
        ref = orc.all_gather_matmul(CODE[dt], bits(xs), bits(ws), r)
        assert_close(outs[r], ref, k, f"AG rank {r}")
        assert torch.equal(outs[r], outs1[r])
        assert np.array_equal(wl.bits16(gathered[r].cpu()), xg), f"gathered copy {r} is not bit-exact"


def test_all_gather_v2_skips_null_entries():
    shape = wl.ColumnParallelSP(R=4, m_shard=64, n_shard=136, k=72, dtype=BF16, x_dist="normal(0,1)",
                                w_dist="normal(0,1)", seed=5)
    xs, ws = shape.make()
    keep = torch.full((256, 72), 3.0, dtype=BF16, device=DEV)
    g = [None, keep, None, torch.empty(256, 72, dtype=BF16, device=DEV)]
    coc.all_gather_matmul_v2(to_dev(xs), to_dev(ws), gathered=g)
    coc.sync_status()
    xg = torch.cat(xs, 0)
    assert torch.equal(keep.cpu(), xg) and torch.equal(g[3].cpu(), xg)


def test_all_gather_one_hot_exact():
    R, ms, ns, k = 4, 48, 136, 96
    shape = wl.ColumnParallelSP(R=R, m_shard=ms, n_shard=ns, k=k, dtype=BF16, x_dist="normal(0,1)",
                                w_dist="normal(0,1)", seed=8)
    xs, _ = shape.make()
    ws = []
    sels = []
    for r in range(R):
        sel = np.random.default_rng(r).integers(0, k, ns)
        W = torch.zeros(k, ns)
        W[sel, torch.arange(ns)] = 1.0
        ws.append(W.to(BF16))
        sels.append(sel)
    outs = coc.all_gather_matmul(to_dev(xs), to_dev(ws), chunks=4)
    coc.sync_status()
    xg = torch.cat(xs, 0)
    for r in range(R):
        assert torch.equal(outs[r].cpu(), xg[:, sels[r]])


# ----------------------------------------------------------------- w8A16 ---

W8_CASES = [
    # R, m, n, k_shard, group, chunks
    (2, 136, 272, 256, 128, 1),
    (4, 256, 512, 128, 64, 2),
    (8, 128, 256, 64, 64, 8),
]


@pytest.mark.parametrize("gran", ["tensor", "channel", "group"])
@pytest.mark.parametrize("R,m,n,ks,group,chunks", W8_CASES)
def test_w8a16_parity(gran, R, m, n, ks, group, chunks):
    shape = wl.W8A16(R=R, m=m, n=n, k_shard=ks, group=group, seed=R + m)
    xs, wqs, scales = shape.make(gran)
    outs = coc.matmul_all_reduce_w8a16(to_dev(xs), to_dev(wqs), to_dev(scales), gran, group, chunks=chunks)
    coc.sync_status()
    code = {"tensor": 0, "channel": 1, "group": 2}[gran]
    ref = orc.matmul_all_reduce_w8a16(bits(xs), [w.numpy() for w in wqs], bits(scales), code, group)
    for r, o in enumerate(outs):
        assert_close(o, ref, shape.K, f"w8A16 {gran} rank {r}")
        assert torch.equal(o, outs[0])


@pytest.mark.parametrize("gran", ["tensor", "channel", "group"])
def test_w8a16_dequant_bitwise(gran):
    """X = one-hot rows selecting single k rows of rank 0's weight, zero on the
    other ranks: the output is then the dequantised weight itself, so the
    in-kernel int8 -> fp16 dequantisation is compared bit for bit."""
    R, n, ks, group = 2, 256, 128, 64
    m = ks
    shape = wl.W8A16(R=R, m=m, n=n, k_shard=ks, group=group, seed=3)
    _, wqs, scales = shape.make(gran)
    X0 = torch.eye(ks, dtype=F16)
    xs = [X0] + [torch.zeros(m, ks, dtype=F16) for _ in range(R - 1)]
    outs = coc.matmul_all_reduce_w8a16(to_dev(xs), to_dev(wqs), to_dev(scales), gran, group)
    coc.sync_status()
    code = {"tensor": 0, "channel": 1, "group": 2}[gran]
    wd = orc.dequant_w8a16(wqs[0].numpy(), wl.bits16(scales[0]), code, group)
    assert np.array_equal(wl.bits16(outs[0].cpu()), wd)


# ------------------------------------------------------------- failures ---

def test_injected_timeout_is_reported_and_device_stays_usable():
    xs, ws = _row_parallel(2, 256, 264, 64, BF16, seed=40)
    dx, dw = to_dev(xs), to_dev(ws)
    coc.inject_timeout(True)
    try:
        coc.matmul_all_reduce(dx, dw)
        with pytest.raises(coc.CocError) as ei:
            coc.sync_status()
        assert ei.value.status == coc.ERR_TIMEOUT
    finally:
        coc.inject_timeout(False)
    coc.sync_status()   # status was cleared
    outs = coc.matmul_all_reduce(dx, dw)
    coc.sync_status()
    assert_close(outs[1], orc.matmul_all_reduce(orc.BF16, bits(xs), bits(ws)), 128, "after timeout")
