"""w8A16 extensions on the GPU against the oracle: int8 zero points
(asymmetric quantisation) and bf16 activations, with group sizes 64/128/256.

Wd = rne_dt((q - z) * s), Y = sum_r X_r @ Wd_r (oracle: fp64, the product
exact and rounded once).  The dequantisation is also compared bit for bit
(one-hot activations make the output the dequantised weight itself)."""
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

CASES = [
    # R, m, n, k_shard, group, chunks
    (2, 136, 272, 256, 128, 1),     # ragged rows (pair tile half empty) and columns
    (4, 256, 512, 256, 256, 2),     # group 256
    (8, 128, 256, 64, 64, 8),       # group 64, one k-block per rank
]


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16], ids=["fp16", "bf16"])
@pytest.mark.parametrize("zero", [False, True], ids=["sym", "zp"])
@pytest.mark.parametrize("gran", ["tensor", "channel", "group"])
@pytest.mark.parametrize("R,m,n,ks,group,chunks", CASES)
def test_w8a16_ext_parity(dt, zero, gran, R, m, n, ks, group, chunks):
    shape = wl.W8A16(R=R, m=m, n=n, k_shard=ks, group=group, seed=R + m + n, dtype=dt)
    xs, wqs, scales = shape.make(gran)
    zs = shape.zeros(gran) if zero else None
    outs = coc.matmul_all_reduce_w8a16(to_dev(xs), to_dev(wqs), to_dev(scales), gran, group, chunks=chunks,
                                       zeros=to_dev(zs) if zs is not None else None)
    coc.sync_status()
    assert all(o.dtype == dt for o in outs)
    ref = orc.matmul_all_reduce_w8a16(bits(xs), [w.numpy() for w in wqs], bits(scales), GRAN[gran], group,
                                      zeros=[z.numpy() for z in zs] if zs is not None else None, dtype=CODE[dt])
    for r, o in enumerate(outs):
        assert_close(o, ref, shape.K, f"w8A16 {dt} zero={zero} {gran} rank {r}")
        assert torch.equal(o, outs[0])


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16], ids=["fp16", "bf16"])
@pytest.mark.parametrize("zero", [False, True], ids=["sym", "zp"])
@pytest.mark.parametrize("gran", ["tensor", "channel", "group"])
def test_w8a16_ext_dequant_bitwise(dt, zero, gran):
    """One-hot rows of X on rank 0 (zeros elsewhere) select single k rows of
    rank 0's weight: the output is the dequantised weight, bit for bit."""
    R, n, ks, group = 2, 256, 128, 64
    m = ks
    shape = wl.W8A16(R=R, m=m, n=n, k_shard=ks, group=group, seed=5, dtype=dt)
    _, wqs, scales = shape.make(gran)
    zs = shape.zeros(gran) if zero else None
    xs = [torch.eye(ks, dtype=dt)] + [torch.zeros(m, ks, dtype=dt) for _ in range(R - 1)]
    outs = coc.matmul_all_reduce_w8a16(to_dev(xs), to_dev(wqs), to_dev(scales), gran, group,
                                       zeros=to_dev(zs) if zs is not None else None)
    coc.sync_status()
    wd = orc.dequant_w8a16_ex(wqs[0].numpy(), wl.bits16(scales[0]), GRAN[gran], group, 0,
                              zs[0].numpy() if zs is not None else None, CODE[dt])
    assert np.array_equal(wl.bits16(outs[0].cpu()), wd)


def test_zero_point_zero_matches_symmetric_bits():
    """An all-zero zero-point tensor gives the symmetric result bit for bit,
    through the pages' fp16 entry point and the extended one."""
    shape = wl.W8A16(R=4, m=256, n=256, k_shard=128, group=64, seed=9)
    xs, wqs, scales = shape.make("group")
    z0 = [torch.zeros_like(z) for z in shape.zeros("group")]
    a = coc.matmul_all_reduce_w8a16(to_dev(xs), to_dev(wqs), to_dev(scales), "group", 64)
    b = coc.matmul_all_reduce_w8a16(to_dev(xs), to_dev(wqs), to_dev(scales), "group", 64, zeros=to_dev(z0))
    coc.sync_status()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_zero_point_equal_to_weight_gives_zero():
    """q == z in every column: the dequantised weight is exactly zero."""
    shape = wl.W8A16(R=2, m=128, n=256, k_shard=128, group=64, seed=12, dtype=torch.bfloat16)
    xs, wqs, scales = shape.make("channel")
    z = shape.zeros("channel")[0]
    wq_eq = [z.view(1, -1).expand(128, -1).contiguous() for _ in range(2)]
    outs = coc.matmul_all_reduce_w8a16(to_dev(xs), to_dev(wq_eq), to_dev(scales), "channel", 64,
                                       zeros=to_dev([z, z]))
    coc.sync_status()
    assert not torch.any(outs[0])


def _force_path(monkeypatch, path):
    monkeypatch.setenv("COC_W8_PATH", path)


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16], ids=["fp16", "bf16"])
@pytest.mark.parametrize("zero", [False, True], ids=["sym", "zp"])
@pytest.mark.parametrize("gran", ["tensor", "channel", "group"])
def test_all_schedules_give_the_same_bits(monkeypatch, dt, zero, gran):
    """Three schedules of the same operator: the default kernel with the
    dequantised weight in tensor memory (Y^T = Wd^T X^T), the fused kernel
    with dequant warps writing the weight tile to shared memory, and the
    pre-pass that dequantises once before the fp16 AllReduce kernel.  All
    use the same conversion and the same accumulation order (rank 0..R-1, k
    ascending, 16 k per MMA): identical outputs."""
    shape = wl.W8A16(R=4, m=512, n=272, k_shard=192, group=64, seed=31, dtype=dt)
    xs, wqs, scales = shape.make(gran)
    zs = shape.zeros(gran) if zero else None
    args = (to_dev(xs), to_dev(wqs), to_dev(scales), gran, 64)
    kw = dict(zeros=to_dev(zs) if zs is not None else None, chunks=2)
    _force_path(monkeypatch, "fused")
    a = coc.matmul_all_reduce_w8a16(*args, **kw)
    _force_path(monkeypatch, "prepass")
    b = coc.matmul_all_reduce_w8a16(*args, **kw)
    _force_path(monkeypatch, "ts")
    c = coc.matmul_all_reduce_w8a16(*args, **kw)
    coc.sync_status()
    for x, y, z in zip(a, b, c):
        assert torch.equal(x, y)
        assert torch.equal(z, y), "tensor-memory schedule differs from the pre-pass schedule"
    ref = orc.matmul_all_reduce_w8a16(bits(xs), [w.numpy() for w in wqs], bits(scales), GRAN[gran], 64,
                                      zeros=[z.numpy() for z in zs] if zs is not None else None, dtype=CODE[dt])
    assert_close(b[0], ref, shape.K, f"pre-pass {dt} zero={zero} {gran}")


def test_prepass_dequant_bitwise(monkeypatch):
    """The pre-pass's dequantised weight, read back through one-hot rows."""
    R, n, ks, group = 2, 256, 128, 64
    shape = wl.W8A16(R=R, m=ks, n=n, k_shard=ks, group=group, seed=6, dtype=torch.bfloat16)
    _, wqs, scales = shape.make("group")
    zs = shape.zeros("group")
    xs = [torch.eye(ks, dtype=torch.bfloat16)] + [torch.zeros(ks, ks, dtype=torch.bfloat16)]
    _force_path(monkeypatch, "prepass")
    outs = coc.matmul_all_reduce_w8a16(to_dev(xs), to_dev(wqs), to_dev(scales), "group", group, zeros=to_dev(zs))
    coc.sync_status()
    wd = orc.dequant_w8a16_ex(wqs[0].numpy(), wl.bits16(scales[0]), 2, group, 0, zs[0].numpy(), orc.BF16)
    assert np.array_equal(wl.bits16(outs[0].cpu()), wd)
