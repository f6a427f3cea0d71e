"""w8A16 MATMUL_ALL_REDUCE at decode-sized m through the column-slab kernel:
the int8 weight streamed over all SMs in slabs of 64, 128 or 256 columns, each
stage dequantised in shared memory by the kernel's own warps (the fused
kernel's conversion), and, with the split, each slab's contraction shared by
a cluster of 2 or 4 CTAs whose fp32 parts add in part order.

COC_W8_PATH=slab with COC_SLAB=1 takes the kernel whatever the SM count;
COC_SLAB_BOXES / COC_SLAB_SPLIT / COC_SLAB_KPS pin the schedule.  Checked
against the fp64 oracle element by element (per-tensor / per-channel /
per-group scales, zero points, fp16 and bf16 activations, ragged m, n and
k_shard), plus: the R copies bit-identical, the unsplit slab bit-identical
to the fused / pre-pass / tensor-memory schedules, and one-hot activations
reproducing the dequantised weight bit for bit."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from tensor_matmul_collective_gb300 import coc
from tensor_matmul_collective_gb300 import workloads as wl

from gpu_util import assert_close, bits, to_dev

pytestmark = pytest.mark.gpu

GRAN = {"tensor": 0, "channel": 1, "group": 2}
CODE = {torch.float16: orc.F16, torch.bfloat16: orc.BF16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_matmul_collective_gb300 import build
    build.build()
    coc.lib()
    yield
    coc.sync_status()


def _slab(monkeypatch, plan):
    b, sp, kps = plan
    for k, v in (("COC_W8_PATH", "slab"), ("COC_SLAB", "1"), ("COC_SLAB_BOXES", b), ("COC_SLAB_SPLIT", sp),
                 ("COC_SLAB_KPS", kps)):
        monkeypatch.setenv(k, str(v))


def _ref(shape, xs, wqs, scales, zs, gran, group, dt):
    return orc.matmul_all_reduce_w8a16(bits(xs), [w.numpy() for w in wqs], bits(scales), GRAN[gran], group,
                                      zeros=[z.numpy() for z in zs] if zs is not None else None, dtype=CODE[dt])


CASES = [
    # R, m, n, k_shard, group, (boxes, split, kps)
    (8, 16, 2048, 256, 128, (2, 2, 2)),     # the decode layer's m, clusters of 2
    (4, 5, 1008, 192, 64, (2, 4, 1)),       # ragged last slab, clusters of 4, group 64
    (2, 100, 528, 128, 128, (1, 2, 2)),     # four row quadrants, 64-column slabs split in two
    (8, 128, 4096, 256, 256, (2, 1, 2)),    # unsplit, group 256
    (2, 33, 20000, 64, 64, (2, 1, 1)),      # several slabs per CTA
    # 256-column slabs (one k-block per stage)
    (8, 16, 4000, 128, 64, (4, 4, 1)),      # clusters of 4, the last slab 160 columns wide
    (2, 100, 2064, 192, 64, (4, 2, 1)),     # clusters of 2, k_shard of three k-blocks, ragged m
    (4, 33, 4352, 256, 128, (4, 1, 1)),     # unsplit, several slabs per CTA
]


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16], ids=["fp16", "bf16"])
@pytest.mark.parametrize("zero", [False, True], ids=["sym", "zp"])
@pytest.mark.parametrize("gran", ["tensor", "channel", "group"])
@pytest.mark.parametrize("R,m,n,ks,group,plan", CASES)
def test_w8a16_slab_parity(monkeypatch, dt, zero, gran, R, m, n, ks, group, plan):
    _slab(monkeypatch, plan)
    shape = wl.W8A16(R=R, m=m, n=n, k_shard=ks, group=group, seed=61 + m, dtype=dt)
    xs, wqs, scales = shape.make(gran)
    zs = shape.zeros(gran) if zero else None
    outs = coc.matmul_all_reduce_w8a16(to_dev(xs), to_dev(wqs), to_dev(scales), gran, group,
                                       zeros=to_dev(zs) if zs is not None else None)
    coc.sync_status()
    ref = _ref(shape, xs, wqs, scales, zs, gran, group, dt)
    for r in range(R):
        assert_close(outs[r], ref, shape.K, f"w8 slab rank {r} {dt} zero={zero} {gran}")
        assert torch.equal(outs[r], outs[0])


@pytest.mark.parametrize("plan", [(2, 1, 2), (4, 1, 1)], ids=["128col", "256col"])
@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16], ids=["fp16", "bf16"])
@pytest.mark.parametrize("gran", ["tensor", "channel", "group"])
def test_unsplit_slab_gives_the_other_schedules_bits(monkeypatch, dt, gran, plan):
    """One CTA per slab: the same conversion and the same accumulation order
    (rank 0..R-1, k ascending, 16 k per MMA) as the fused, pre-pass and
    tensor-memory schedules, so the same bits."""
    shape = wl.W8A16(R=4, m=100, n=1040, k_shard=192, group=64, seed=71, dtype=dt)
    xs, wqs, scales = shape.make(gran)
    zs = shape.zeros(gran)
    args = (to_dev(xs), to_dev(wqs), to_dev(scales), gran, 64)
    kw = dict(zeros=to_dev(zs))
    _slab(monkeypatch, plan)
    a = [t.clone() for t in coc.matmul_all_reduce_w8a16(*args, **kw)]
    outs = {}
    for path in ("fused", "prepass", "ts"):
        monkeypatch.setenv("COC_W8_PATH", path)
        outs[path] = [t.clone() for t in coc.matmul_all_reduce_w8a16(*args, **kw)]
    coc.sync_status()
    for path, o in outs.items():
        for x, y in zip(a, o):
            assert torch.equal(x, y), f"slab differs from the {path} schedule"


@pytest.mark.parametrize("plan", [(2, 1, 2), (2, 2, 2), (1, 2, 4), (4, 4, 1)])
def test_w8a16_slab_dequant_bitwise(monkeypatch, plan):
    """One-hot activations (X_r = e_i rows of one rank, the others zero):
    output row i is the dequantised weight row i of that rank, bit for bit."""
    _slab(monkeypatch, plan)
    R, m, n, ks, group = 4, 16, 1024, 128, 64
    shape = wl.W8A16(R=R, m=m, n=n, k_shard=ks, group=group, seed=73, dtype=torch.float16)
    _, wqs, scales = shape.make("group")
    zs = shape.zeros("group")
    xs = [torch.zeros(m, ks, dtype=torch.float16) for _ in range(R)]
    rows = []
    for i in range(m):
        r, k = i % R, (i * 7) % ks
        xs[r][i, k] = 1.0
        rows.append((r, k))
    outs = coc.matmul_all_reduce_w8a16(to_dev(xs), to_dev(wqs), to_dev(scales), "group", group, zeros=to_dev(zs))
    coc.sync_status()
    got = outs[0].cpu()
    for i, (r, k) in enumerate(rows):
        wd = orc.dequant_w8a16_ex(wqs[r].numpy(), wl.bits16(scales[r]), GRAN["group"], group, 0, zs[r].numpy(),
                                  orc.F16)
        assert np.array_equal(wl.bits16(got[i:i + 1])[0], wd[k]), f"row {i} (rank {r}, k {k})"


@pytest.mark.parametrize("m", [1, 16, 64, 128])
def test_w8a16_decode_default_takes_the_slab(monkeypatch, m):
    """The default schedule at the decode layer's shape gives the oracle's
    values (on a 152-SM GB300 it is the slab kernel split in clusters, with
    the slab width and stage depth the library picks for m)."""
    monkeypatch.delenv("COC_W8_PATH", raising=False)
    shape = wl.W8A16(R=8, m=m, n=8192, k_shard=1024, group=128, seed=75 + m, dtype=torch.float16)
    xs, wqs, scales = shape.make("channel")
    outs = coc.matmul_all_reduce_w8a16(to_dev(xs), to_dev(wqs), to_dev(scales), "channel", 128)
    coc.sync_status()
    ref = _ref(shape, xs, wqs, scales, None, "channel", 128, torch.float16)
    assert_close(outs[5], ref, shape.K, "decode w8A16")
