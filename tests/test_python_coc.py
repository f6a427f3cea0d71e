"""The Python-script CoC comparison path (CoC page, Python脚本层面实现)
against the fp64 oracle: AllReduce, ReduceScatter and AllGather(+V2) cut into
1/2/4/8 chunks along m.  On the CPU the steps run in program order; on the
GPU on a compute and a communication stream, and there the results are also
compared with the fused kernels'."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from tensor_matmul_collective_gb300 import python_coc as pc
from tensor_matmul_collective_gb300 import workloads as wl

from gpu_util import assert_close, bits

BF16, F16 = torch.bfloat16, torch.float16
CODE = {F16: orc.F16, BF16: orc.BF16}


def _rp(R, m, n, ks, dt, seed):
    return wl.RowParallel(R=R, m=m, n=n, k_shard=ks, dtype=dt, x_dist="normal(0,1)", w_dist="normal(0,0.02)",
                          seed=seed).make()


def _cp(R, ms, ns, k, dt, seed):
    return wl.ColumnParallelSP(R=R, m_shard=ms, n_shard=ns, k=k, dtype=dt, x_dist="normal(0,1)",
                               w_dist="normal(0,0.02)", seed=seed).make()


def _run_all(xs, ws, dev, streams, R, m, n, k_total, dt):
    code = CODE[dt]
    xd, wd = [x.to(dev) for x in xs], [w.to(dev) for w in ws]
    ref = orc.matmul_all_reduce(code, bits(xs), bits(ws))
    for C in (1, 2, 4, 8):
        outs = [torch.full((m, n), float("nan"), dtype=dt, device=dev) for _ in range(R)]
        pc.all_reduce(xd, wd, outs, C, *streams)
        if dev.type == "cuda":
            torch.cuda.synchronize()
        for r in range(R):
            assert_close(outs[r], ref, k_total, f"AR chunks {C} rank {r}")
            assert torch.equal(outs[r], outs[0])
        routs = [torch.full((m // R, n), float("nan"), dtype=dt, device=dev) for _ in range(R)]
        pc.reduce_scatter(xd, wd, routs, C, *streams)
        if dev.type == "cuda":
            torch.cuda.synchronize()
        for r in range(R):
            assert_close(routs[r], ref[r * (m // R):(r + 1) * (m // R)], k_total, f"RS chunks {C} rank {r}")
    return ref


@pytest.mark.parametrize("dt", [BF16, F16])
def test_row_parallel_chunks_cpu(dt):
    R, m, n, ks = 4, 64, 48, 40
    xs, ws = _rp(R, m, n, ks, dt, 11)
    _run_all(xs, ws, torch.device("cpu"), (None, None), R, m, n, R * ks, dt)


@pytest.mark.parametrize("dt", [BF16, F16])
def test_all_gather_chunks_cpu(dt):
    R, ms, ns, k = 4, 16, 40, 72
    xs, ws = _cp(R, ms, ns, k, dt, 12)
    xg_ref = orc.all_gather(bits(xs))
    for C in (1, 2, 4, 8):
        outs = [torch.full((R * ms, ns), float("nan"), dtype=dt) for _ in range(R)]
        gath = [torch.zeros(R * ms, k, dtype=dt) for _ in range(R)]
        pc.all_gather(xs, ws, outs, C, gathered=gath)
        for r in range(R):
            assert_close(outs[r], orc.all_gather_matmul(CODE[dt], bits(xs), bits(ws), r), k, f"AG chunks {C} rank {r}")
            assert np.array_equal(wl.bits16(gath[r]), xg_ref)     # the gathered input, bit-exact


def test_chunk_count_must_divide():
    R, m, n, ks = 2, 12, 8, 8
    xs, ws = _rp(R, m, n, ks, BF16, 13)
    outs = [torch.empty(m, n, dtype=BF16) for _ in range(R)]
    with pytest.raises(ValueError):
        pc.all_reduce(xs, ws, outs, 8)
    with pytest.raises(ValueError):
        pc.reduce_scatter(xs, ws, [torch.empty(m // R, n, dtype=BF16)] * R, 8)
    with pytest.raises(ValueError):
        pc.all_gather([torch.empty(3, 8, dtype=BF16)] * 2, [torch.empty(8, 4, dtype=BF16)] * 2,
                      [torch.empty(6, 4, dtype=BF16)] * 2, 4)


def test_reduce_scatter_chunks_straddle_ranks_cpu():
    """Chunk boundaries that cut through a rank's row block (m/C not a
    multiple of m/R) still land every row at its owner."""
    R, m, n, ks = 4, 48, 16, 24
    xs, ws = _rp(R, m, n, ks, BF16, 14)
    ref = orc.matmul_all_reduce(orc.BF16, bits(xs), bits(ws))
    routs = [torch.full((m // R, n), float("nan"), dtype=BF16) for _ in range(R)]
    pc.reduce_scatter(xs, ws, routs, 8)          # 6-row chunks, 12-row rank blocks
    for r in range(R):
        assert_close(routs[r], ref[r * 12:(r + 1) * 12], R * ks, f"rank {r}")
    routs3 = [torch.full((m // R, n), float("nan"), dtype=BF16) for _ in range(R)]
    pc.reduce_scatter(xs, ws, routs3, 3)         # 16-row chunks across 12-row blocks
    for r in range(R):
        assert_close(routs3[r], ref[r * 12:(r + 1) * 12], R * ks, f"3 chunks, rank {r}")


@pytest.mark.gpu
def test_streams_gpu_against_oracle_and_fused():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_matmul_collective_gb300 import build, coc
    build.build()
    dev = torch.device("cuda:0")
    streams = (torch.cuda.Stream(), torch.cuda.Stream())
    R, m, n, ks = 8, 512, 384, 256
    xs, ws = _rp(R, m, n, ks, BF16, 15)
    ref = _run_all(xs, ws, dev, streams, R, m, n, R * ks, BF16)
    fused = coc.matmul_all_reduce([x.to(dev) for x in xs], [w.to(dev) for w in ws], chunks=4)
    coc.sync_status()
    assert_close(fused[0], ref, R * ks, "fused AR")
    R, ms, ns, k = 8, 64, 320, 256
    xs, ws = _cp(R, ms, ns, k, BF16, 16)
    xd, wd = [x.to(dev) for x in xs], [w.to(dev) for w in ws]
    xg_ref = orc.all_gather(bits(xs))
    for C in (1, 2, 4, 8):
        outs = [torch.full((R * ms, ns), float("nan"), dtype=BF16, device=dev) for _ in range(R)]
        gath = [torch.zeros(R * ms, k, dtype=BF16, device=dev) for _ in range(R)]
        pc.all_gather(xd, wd, outs, C, gath, *streams)
        torch.cuda.synchronize()
        for r in range(R):
            assert_close(outs[r], orc.all_gather_matmul(orc.BF16, bits(xs), bits(ws), r), k, f"AG chunks {C} rank {r}")
            assert np.array_equal(wl.bits16(gath[r].cpu()), xg_ref)
