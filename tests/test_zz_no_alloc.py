"""The allocation-free MATMUL_ALL_REDUCE entry point.

Some callers cannot allocate device memory at the point where they run the
operator: runtimes that pre-carve all device memory into their own pools,
latency-critical paths that cannot take cudaMalloc's implicit
synchronisation, processes whose allocations must all go through their own
allocator.  coc_matmul_all_reduce_noalloc serves them: its kernel scratch
(the status block of the bounded waits) lives in a fixed static device array
instead of a buffer the library allocates.

This file calls it through the C ABI and checks every result against the fp64
oracle and against the allocating entry point's output, within the tolerance
the parity tests use, with two calls in a row per shape.  It also checks that
the chunk count never changes a bit, that an injected timeout is reported by
coc_sync_status (and the next call is correct), and that the library's
allocation counter does not move.  It builds the library itself, so it passes
alone in a fresh process as well as after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from tensor_matmul_collective_gb300 import coc
from tensor_matmul_collective_gb300 import workloads as wl

from gpu_util import DEV, assert_close, bits

pytestmark = pytest.mark.gpu

CODE = {torch.float16: orc.F16, torch.bfloat16: orc.BF16}


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_matmul_collective_gb300 import build
    build.build()
    return coc.lib()


def _ptrs(ts):
    a = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        a[i] = t.data_ptr()
    return a


def _call(L, dx, dw, outs, chunks):
    R, (m, ks), n = len(dx), dx[0].shape, dw[0].shape[1]
    code = coc.BF16 if dx[0].dtype == torch.bfloat16 else coc.FP16
    st = L.coc_matmul_all_reduce_noalloc(R, m, n, ks, _ptrs(dx), _ptrs(dw), _ptrs(outs), code, chunks, 1,
                                         torch.cuda.current_stream().cuda_stream)
    assert st == coc.OK, L.coc_last_error()


CASES = [
    # R, m, n, k_shard, dtype, chunks
    (1, 16, 264, 128, torch.bfloat16, 1),     # R = 1, decode-sized m (no rank split here)
    (2, 100, 72, 64, torch.float16, 2),       # partial row tile, one narrow column tile
    (8, 200, 136, 0, torch.bfloat16, 1),      # k_shard = 0: zeros
    (4, 384, 520, 136, torch.bfloat16, 2),    # several tiles, ragged n and k
    (8, 1024, 264, 72, torch.float16, 4),     # chunk-major order
]


@pytest.mark.parametrize("R,m,n,ks,dt,chunks", CASES)
def test_noalloc_allreduce_against_oracle_twice(L, R, m, n, ks, dt, chunks):
    for call in range(2):   # two calls in a row, on different inputs
        xs, ws = wl.RowParallel(R=R, m=m, n=n, k_shard=ks, dtype=dt, x_dist="normal(0,1)",
                                w_dist="normal(0,1)", seed=100 + 10 * call + R).make()
        dx = [x.to(DEV) for x in xs]
        dw = [w.to(DEV) for w in ws]
        outs = [torch.full((m, n), float("nan"), dtype=dt, device=DEV) for _ in range(R)]
        _call(L, dx, dw, outs, chunks)
        coc.sync_status()
        ref = orc.matmul_all_reduce(CODE[dt], bits(xs), bits(ws))
        for r in range(R):
            assert_close(outs[r], ref, max(R * ks, 1), f"no-alloc call {call} rank {r}")
            assert torch.equal(outs[r], outs[0])
        if ks == 0:
            assert not outs[0].any()
        # and against the allocating entry point, within the same tolerance
        alloc_out = coc.matmul_all_reduce(dx, dw, chunks=chunks)
        coc.sync_status()
        assert_close(outs[0], alloc_out[0].double().cpu().numpy(), max(R * ks, 1), "vs allocating entry point")
    # no-alloc calls leave the library's allocation counter where it was
    xs, ws = wl.RowParallel(R=R, m=m, n=n, k_shard=ks, dtype=dt, x_dist="normal(0,1)",
                            w_dist="normal(0,1)", seed=999).make()
    dx, dw = [x.to(DEV) for x in xs], [w.to(DEV) for w in ws]
    outs = [torch.empty((m, n), dtype=dt, device=DEV) for _ in range(R)]
    n0 = coc.alloc_count()
    for _ in range(3):
        _call(L, dx, dw, outs, chunks)
    torch.cuda.synchronize()
    assert coc.alloc_count() == n0


def test_noalloc_chunk_count_never_changes_a_bit(L):
    R, m, n, ks, dt = 8, 1024, 264, 200, torch.bfloat16
    xs, ws = wl.RowParallel(R=R, m=m, n=n, k_shard=ks, dtype=dt, x_dist="normal(0,1)",
                            w_dist="normal(0,1)", seed=77).make()
    dx, dw = [x.to(DEV) for x in xs], [w.to(DEV) for w in ws]
    res = {}
    for chunks in (1, 2, 4, 8):
        outs = [torch.empty((m, n), dtype=dt, device=DEV) for _ in range(R)]
        _call(L, dx, dw, outs, chunks)
        coc.sync_status()
        res[chunks] = outs[0].clone()
        assert all(torch.equal(o, outs[0]) for o in outs)
    for chunks in (2, 4, 8):
        assert torch.equal(res[chunks], res[1]), f"chunks = {chunks}"
    rows = wl.sample_rows(m, 64)
    ref = orc.matmul_all_reduce(CODE[dt], bits(xs), bits(ws), rows)
    assert_close(res[1].index_select(0, torch.from_numpy(rows).to(DEV)), ref, R * ks, "chunk sweep")


def test_noalloc_timeout_is_reported(L):
    """A bounded wait that runs out in the allocation-free kernel is reported
    by coc_sync_status (the static status block), and the next call works."""
    R, m, n, ks, dt = 2, 256, 264, 64, torch.bfloat16
    xs, ws = wl.RowParallel(R=R, m=m, n=n, k_shard=ks, dtype=dt, x_dist="normal(0,1)",
                            w_dist="normal(0,1)", seed=55).make()
    dx, dw = [x.to(DEV) for x in xs], [w.to(DEV) for w in ws]
    outs = [torch.empty((m, n), dtype=dt, device=DEV) for _ in range(R)]
    coc.sync_status()
    coc.inject_timeout(True)
    try:
        _call(L, dx, dw, outs, 1)
        with pytest.raises(coc.CocError) as ei:
            coc.sync_status()
        assert ei.value.status == coc.ERR_TIMEOUT
        assert "allocation-free" in ei.value.detail
    finally:
        coc.inject_timeout(False)
    coc.sync_status()   # reported once, then cleared
    _call(L, dx, dw, outs, 1)
    coc.sync_status()
    assert_close(outs[1], orc.matmul_all_reduce(orc.BF16, bits(xs), bits(ws)), R * ks, "after the timeout")
