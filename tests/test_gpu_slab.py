"""AllReduce and ReduceScatter at decode-sized m through the column-slab
kernel: each output slab of 64 or 128 columns (all m rows) is summed over the
contraction in one CTA, or in a cluster of 2 or 4 CTAs that each sum a
contiguous range of it and add the parts in part order through distributed
shared memory.

COC_SLAB=1 takes the kernel for every m <= 128 whatever the SM count, and
COC_SLAB_BOXES / COC_SLAB_SPLIT / COC_SLAB_KPS pin the slab width, the
cluster size and the k-blocks per stage, so the cases below reach every
schedule on any device.  Checked against the fp64 oracle element by element
(ragged m, n and k_shard; 2-D and 3-D operand maps; several slabs per CTA;
k x n and n x k weight storage; both 16-bit types), plus: the R AllReduce
copies bit-identical, concat(RS) equal to the AllReduce bits, the plain GEMM
equal to the AllReduce, bit-identical results across calls and chunk
counts, an unsplit slab equal to the persistent kernel's unsplit tile bits,
and an injected timeout reported."""
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
def _slab(monkeypatch):
    monkeypatch.setenv("COC_SLAB", "1")


def _data(R, m, n, ks, dt, seed):
    return wl.RowParallel(R=R, m=m, n=n, k_shard=ks, dtype=dt, x_dist="normal(0,1)", w_dist="normal(0,0.02)",
                          seed=seed).make()


CASES = [
    # R, m, n, k_shard, dtype, (boxes, split, kps)
    (8, 1, 5000, 256, BF16, (2, 2, 2)),      # one row; 40 slabs, the last 8 columns wide; 3-D X map
    (8, 16, 8192, 128, BF16, (2, 2, 2)),     # the decode layer's m and n
    (8, 5, 9792, 200, F16, (1, 1, 4)),       # k_shard ends inside a k-block: 2-D X boxes
    (4, 33, 6000, 72, BF16, (2, 4, 1)),      # rows in two TMEM lane quadrants, clusters of 4
    (8, 64, 4864, 64, F16, (1, 2, 1)),       # 64-column slabs split in two (32 columns per part)
    (2, 128, 4096, 64, BF16, (2, 1, 1)),     # all four epilogue warps, unsplit
    (4, 100, 6000, 128, BF16, (2, 2, 1)),    # four row quadrants pushed between two parts
    (8, 128, 4096, 256, F16, (2, 4, 1)),     # four row quadrants, clusters of 4
    (2, 16, 40000, 64, BF16, (2, 1, 1)),     # several slabs per CTA (both accumulator buffers)
    (8, 16, 4096, 1024, BF16, (2, 4, 2)),    # the 4096-column decode layer: clusters of 4
    (8, 48, 8192, 256, F16, (2, 2, 4)),      # four k-blocks per stage with 128-column slabs
]


def _plan(monkeypatch, plan):
    b, sp, kps = plan
    monkeypatch.setenv("COC_SLAB_BOXES", str(b))
    monkeypatch.setenv("COC_SLAB_SPLIT", str(sp))
    monkeypatch.setenv("COC_SLAB_KPS", str(kps))


@pytest.mark.parametrize("R,m,n,ks,dt,plan", CASES)
def test_slab_allreduce_parity(R, m, n, ks, dt, plan, monkeypatch):
    _plan(monkeypatch, plan)
    xs, ws = _data(R, m, n, ks, dt, 23 * m + n)
    dx, dw = to_dev(xs), to_dev(ws)
    outs = coc.matmul_all_reduce(dx, dw)
    coc.sync_status()
    ref = orc.matmul_all_reduce(CODE[dt], bits(xs), bits(ws))
    for r in range(R):
        assert_close(outs[r], ref, R * ks, f"AR rank {r}")
        assert torch.equal(outs[r], outs[0])
    plain = coc.matmul(dx, dw)
    coc.sync_status()
    assert torch.equal(plain, outs[0])


@pytest.mark.parametrize("R,m,n,ks,dt,plan", [c for c in CASES if c[1] % (8 * c[0]) == 0])
def test_slab_reduce_scatter_parity_and_concat(R, m, n, ks, dt, plan, monkeypatch):
    _plan(monkeypatch, plan)
    xs, ws = _data(R, m, n, ks, dt, 29 * m + n)
    dx, dw = to_dev(xs), to_dev(ws)
    rs = coc.matmul_reduce_scatter(dx, dw)
    ar = coc.matmul_all_reduce(dx, dw)
    coc.sync_status()
    ref = orc.matmul_all_reduce(CODE[dt], bits(xs), bits(ws))
    per = m // R
    for r in range(R):
        assert_close(rs[r], ref[r * per:(r + 1) * per], R * ks, f"RS rank {r}")
    assert torch.equal(torch.cat(rs, 0), ar[0])


@pytest.mark.parametrize("n,plan", [(5000, (2, 2, 2)), (9792, (1, 1, 2)), (6000, (2, 4, 1)), (4096, (1, 2, 4))])
def test_slab_nk_weights_match_kn_bits(n, plan, monkeypatch):
    """n x k weight storage (the B operand read K-major, as 3-D boxes when a
    stage holds several k-blocks) gives the k x n bits."""
    _plan(monkeypatch, plan)
    R, m, ks = 8, 16, 128
    xs, ws = _data(R, m, n, ks, BF16, n + 1)
    dx, dw = to_dev(xs), to_dev(ws)
    kn = coc.matmul_all_reduce(dx, dw)
    nk = coc.fused_matmul("all_reduce", dx, [w.t().contiguous() for w in dw], w_layout="nk")
    coc.sync_status()
    for a, b in zip(kn, nk):
        assert torch.equal(a, b)
    assert_close(kn[0], orc.matmul_all_reduce(orc.BF16, bits(xs), bits(ws)), R * ks, "k x n")


def test_slab_is_reproducible_across_runs_and_chunks():
    R, m, n, ks = 8, 16, 8192, 256
    xs, ws = _data(R, m, n, ks, BF16, 5)
    dx, dw = to_dev(xs), to_dev(ws)
    first = coc.matmul_all_reduce(dx, dw, chunks=1)[0].clone()
    for _ in range(5):
        assert torch.equal(coc.matmul_all_reduce(dx, dw, chunks=1)[0], first)
    for c in (2, 4, 8):
        assert torch.equal(coc.matmul_all_reduce(dx, dw, chunks=c, deterministic=True)[0], first)
    coc.sync_status()


@pytest.mark.parametrize("R,m,n,ks", [(8, 16, 8192, 256), (4, 64, 5000, 200), (2, 100, 4096, 64)])
def test_unsplit_slab_gives_the_persistent_kernels_bits(R, m, n, ks, monkeypatch):
    """One CTA per slab adds the same MMAs into one accumulator in the same
    order (rank 0..R-1, k ascending) as the persistent kernel's unsplit tile,
    so the bits agree."""
    xs, ws = _data(R, m, n, ks, BF16, 31 * m + ks)
    dx, dw = to_dev(xs), to_dev(ws)
    _plan(monkeypatch, (2, 1, 2))
    slab = [t.clone() for t in coc.matmul_all_reduce(dx, dw)]
    monkeypatch.setenv("COC_SLAB", "0")
    monkeypatch.setenv("COC_KSPLIT", "1")
    tile = coc.matmul_all_reduce(dx, dw)
    coc.sync_status()
    for a, b in zip(slab, tile):
        assert torch.equal(a, b)


@pytest.mark.parametrize("plan", [(2, 1, 2), (2, 4, 2)])
def test_slab_one_hot_is_exact(plan, monkeypatch):
    """Each output element receives exactly one nonzero product (weight 1.0
    at one k of one rank per column): the output must reproduce X columns bit
    for bit, and any misplaced k, rank or column shows."""
    _plan(monkeypatch, plan)
    R, m, n, ks = 8, 16, 5000, 64
    gen = torch.Generator().manual_seed(3)
    xs = [torch.randn(m, ks, generator=gen).to(BF16) for _ in range(R)]
    ws = [torch.zeros(ks, n, dtype=BF16) for _ in range(R)]
    expect = torch.empty(m, n, dtype=BF16)
    for j in range(n):
        r, t = (j * 5) % R, (j * 7) % ks
        ws[r][t, j] = 1.0
        expect[:, j] = xs[r][:, t]
    outs = coc.matmul_all_reduce(to_dev(xs), to_dev(ws))
    coc.sync_status()
    for o in outs:
        assert torch.equal(o.cpu(), expect)


@pytest.mark.parametrize("plan", [(2, 1, 2), (2, 2, 2)])
def test_slab_injected_timeout_is_reported_and_device_stays_usable(plan, monkeypatch):
    _plan(monkeypatch, plan)
    xs, ws = _data(8, 16, 5000, 64, BF16, 41)
    dx, dw = to_dev(xs), to_dev(ws)
    coc.inject_timeout(True)
    try:
        coc.matmul_all_reduce(dx, dw)
        with pytest.raises(coc.CocError) as ei:
            coc.sync_status()
        assert ei.value.status == coc.ERR_TIMEOUT
    finally:
        coc.inject_timeout(False)
    coc.sync_status()
    outs = coc.matmul_all_reduce(dx, dw)
    coc.sync_status()
    assert_close(outs[3], orc.matmul_all_reduce(orc.BF16, bits(xs), bits(ws)), 8 * 64, "after timeout")
