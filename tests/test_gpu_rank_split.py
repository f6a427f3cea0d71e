"""AllReduce and ReduceScatter at decode-sized m, where the library cuts each
output tile's R shards into parts run as separate work units (rank split)
and the last part of each row slab adds the parts in a fixed order.

Checked against the fp64 oracle element by element, plus the properties that
must survive the split: the R AllReduce copies bit-identical, concat(RS) equal
to the AllReduce bits, results bit-identical across repeated calls and chunk
counts, the plain single-output GEMM equal to the AllReduce, R = 1 unsplit."""
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


@pytest.fixture(autouse=True)
def _no_slab(monkeypatch):
    # decode-sized shapes whose column slabs cover the SMs would otherwise go
    # to the column-slab kernel, which needs no split
    monkeypatch.setenv("COC_SLAB", "0")


def _data(R, m, n, ks, dt, seed):
    return wl.RowParallel(R=R, m=m, n=n, k_shard=ks, dtype=dt, x_dist="normal(0,1)", w_dist="normal(0,0.02)",
                          seed=seed).make()


CASES = [
    # R, m, n, k_shard, dtype: few output tiles (split), ragged m / n / k
    (8, 1, 4096, 256, BF16),
    (8, 16, 8192, 128, BF16),
    (8, 64, 1000, 72, F16),
    (4, 100, 520, 200, BF16),
    (2, 128, 256, 64, F16),
    (8, 200, 2048, 96, BF16),
    (8, 256, 4096, 128, BF16),
    (4, 384, 8192, 64, F16),
]


@pytest.mark.parametrize("R,m,n,ks,dt", CASES)
def test_split_allreduce_parity(R, m, n, ks, dt):
    xs, ws = _data(R, m, n, ks, dt, 7 * m + n)
    outs = coc.matmul_all_reduce(to_dev(xs), to_dev(ws))
    coc.sync_status()
    ref = orc.matmul_all_reduce(CODE[dt], bits(xs), bits(ws))
    for r in range(R):
        assert_close(outs[r], ref, R * ks, f"AR rank {r}")
        assert torch.equal(outs[r], outs[0])
    plain = coc.matmul(to_dev(xs), to_dev(ws))
    coc.sync_status()
    assert torch.equal(plain, outs[0])


@pytest.mark.parametrize("R,m,n,ks,dt", [c for c in CASES if c[1] % (8 * c[0]) == 0])   # m / R: 8-row blocks
def test_split_reduce_scatter_parity_and_concat(R, m, n, ks, dt):
    xs, ws = _data(R, m, n, ks, dt, 11 * m + n)
    dx, dw = to_dev(xs), to_dev(ws)
    rs = coc.matmul_reduce_scatter(dx, dw)
    ar = coc.matmul_all_reduce(dx, dw)
    coc.sync_status()
    ref = orc.matmul_all_reduce(CODE[dt], bits(xs), bits(ws))
    per = m // R
    for r in range(R):
        assert_close(rs[r], ref[r * per:(r + 1) * per], R * ks, f"RS rank {r}")
    assert torch.equal(torch.cat(rs, 0), ar[0])


def test_split_is_reproducible_across_runs_and_chunks():
    R, m, n, ks = 8, 128, 4096, 256
    xs, ws = _data(R, m, n, ks, BF16, 5)
    dx, dw = to_dev(xs), to_dev(ws)
    first = coc.matmul_all_reduce(dx, dw, chunks=1, deterministic=True)[0].clone()
    for _ in range(10):
        assert torch.equal(coc.matmul_all_reduce(dx, dw, chunks=1, deterministic=True)[0], first)
    for c in (2, 4, 8):
        assert torch.equal(coc.matmul_all_reduce(dx, dw, chunks=c, deterministic=True)[0], first)
        assert torch.equal(coc.matmul_all_reduce(dx, dw, chunks=c, deterministic=False)[0], first)
    coc.sync_status()


def test_split_one_hot_is_exact():
    """Each output element receives exactly one nonzero product, from one rank
    chosen per column: the parts of the other ranks are exact zeros, so the
    sum of parts must reproduce X columns bit for bit."""
    R, m, n, ks = 8, 64, 512, 64
    gen = torch.Generator().manual_seed(3)
    xs = [torch.randn(m, ks, generator=gen).to(BF16) for _ in range(R)]
    ws = [torch.zeros(ks, n, dtype=BF16) for _ in range(R)]
    expect = torch.empty(m, n, dtype=BF16)
    for j in range(n):
        r, t = j % R, (j * 7) % ks
        ws[r][t, j] = 1.0
        expect[:, j] = xs[r][:, t]
    outs = coc.matmul_all_reduce(to_dev(xs), to_dev(ws))
    rs = coc.matmul_reduce_scatter(to_dev(xs), to_dev(ws))
    coc.sync_status()
    for o in outs:
        assert torch.equal(o.cpu(), expect)
    assert torch.equal(torch.cat(rs, 0).cpu(), expect)


@pytest.mark.parametrize("R,m,n,ks,forced", [(8, 200, 2048, 96, 2), (8, 256, 1024, 128, 4), (4, 64, 1000, 72, 4),
                                             (8, 100, 4096, 64, 8)])
def test_forced_part_counts(R, m, n, ks, forced, monkeypatch):
    """Part counts the shape would not choose (the 256-row pair tiles are never
    split by default): the same parity and reproducibility."""
    xs, ws = _data(R, m, n, ks, BF16, 13 * m + forced)
    dx, dw = to_dev(xs), to_dev(ws)
    ref = orc.matmul_all_reduce(orc.BF16, bits(xs), bits(ws))
    monkeypatch.setenv("COC_KSPLIT", str(forced))
    outs = coc.matmul_all_reduce(dx, dw)
    again = coc.matmul_all_reduce(dx, dw, chunks=4 if m % 4 == 0 else 1)
    coc.sync_status()
    for r in range(R):
        assert_close(outs[r], ref, R * ks, f"AR rank {r}, {forced} parts")
        assert torch.equal(outs[r], outs[0])
    assert torch.equal(again[0], outs[0])
    if m % (8 * R) == 0:
        rs = coc.matmul_reduce_scatter(dx, dw)
        coc.sync_status()
        assert torch.equal(torch.cat(rs, 0), outs[0])


def test_split_nk_weights_match_kn_bits():
    """Megatron's n x k weight storage takes the same split and gives the
    same bits as k x n (the B operand read K-major instead of MN-major)."""
    R, m, n, ks = 8, 16, 2048, 128
    xs, ws = _data(R, m, n, ks, BF16, 17)
    dx, dw = to_dev(xs), to_dev(ws)
    wnk = [w.t().contiguous() for w in dw]
    kn = coc.matmul_all_reduce(dx, dw)
    nk = coc.fused_matmul("all_reduce", dx, wnk, w_layout="nk")
    coc.sync_status()
    for a, b in zip(kn, nk):
        assert torch.equal(a, b)
    m2 = 128   # ReduceScatter needs m / R in 8-row blocks
    xs2, ws2 = _data(R, m2, n, ks, BF16, 18)
    dx2, dw2 = to_dev(xs2), to_dev(ws2)
    rs = coc.matmul_reduce_scatter(dx2, dw2)
    rs_nk = coc.fused_matmul("reduce_scatter", dx2, [w.t().contiguous() for w in dw2], w_layout="nk")
    coc.sync_status()
    for a, b in zip(rs, rs_nk):
        assert torch.equal(a, b)


def test_r1_and_zero_k_are_not_split():
    xs, ws = _data(1, 16, 256, 64, BF16, 9)
    out = coc.matmul_all_reduce(to_dev(xs), to_dev(ws))
    coc.sync_status()
    assert_close(out[0], orc.matmul_all_reduce(orc.BF16, bits(xs), bits(ws)), 64, "R = 1")
    z = coc.matmul_all_reduce([torch.empty(16, 0, dtype=BF16, device="cuda")] * 4,
                              [torch.empty(0, 256, dtype=BF16, device="cuda")] * 4)
    coc.sync_status()
    assert all(torch.count_nonzero(o) == 0 for o in z)


@pytest.mark.parametrize("R,m,n,ks,dt", [(8, 16, 8192, 128, BF16), (8, 64, 1000, 72, F16), (4, 100, 520, 200, BF16),
                                         (2, 128, 256, 64, F16), (8, 128, 4096, 64, BF16)])
def test_cluster_and_scratch_split_give_the_same_bits(R, m, n, ks, dt, monkeypatch):
    """The rank split runs its parts as one cluster that adds them through
    distributed shared memory, or (COC_SPLIT_PATH=scratch) through a global
    workspace with arrival counters: the same parts added in the same order,
    so the same bits, for AllReduce and ReduceScatter."""
    xs, ws = _data(R, m, n, ks, dt, 19 * m + n)
    dx, dw = to_dev(xs), to_dev(ws)
    a = [t.clone() for t in coc.matmul_all_reduce(dx, dw)]
    rs_ok = m % (8 * R) == 0
    ra = [t.clone() for t in coc.matmul_reduce_scatter(dx, dw)] if rs_ok else None
    monkeypatch.setenv("COC_SPLIT_PATH", "scratch")
    b = coc.matmul_all_reduce(dx, dw)
    rb = coc.matmul_reduce_scatter(dx, dw) if rs_ok else None
    coc.sync_status()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    if rs_ok:
        for x, y in zip(ra, rb):
            assert torch.equal(x, y)
    assert_close(a[0], orc.matmul_all_reduce(CODE[dt], bits(xs), bits(ws)), R * ks, "cluster split")
