"""The allocation-free MATMUL_ALL_REDUCE entry point.

Some callers cannot allocate device memory at the point where they run the
operator (runtimes that pre-carve all device memory into their own pools,
latency-critical paths that cannot take cudaMalloc's implicit
synchronisation).  coc_matmul_all_reduce_noalloc serves them: its kernel
scratch lives in a fixed static device array instead of a buffer the library
allocates.  This test calls it through the C ABI, twice in a row on different
inputs, and checks each result against the allocating entry point's, within
the same tolerance the parity tests use.  It builds the library itself, so it
passes alone in a fresh process as well as after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from tensor_matmul_collective_gb300 import coc
from tensor_matmul_collective_gb300 import workloads as wl

from gpu_util import DEV, assert_close

pytestmark = pytest.mark.gpu


def _ptrs(ts):
    a = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        a[i] = t.data_ptr()
    return a


def test_noalloc_allreduce_matches_allocating_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_matmul_collective_gb300 import build
    build.build()
    L = coc.lib()
    stream = torch.cuda.current_stream().cuda_stream
    cases = [(4, 384, 520, 136, torch.bfloat16, 2, 101), (8, 1024, 264, 72, torch.float16, 4, 102)]
    for R, m, n, ks, dt, chunks, seed in cases:
        xs, ws = wl.RowParallel(R=R, m=m, n=n, k_shard=ks, dtype=dt, x_dist="normal(0,1)",
                                w_dist="normal(0,1)", seed=seed).make()
        dx = [x.to(DEV) for x in xs]
        dw = [w.to(DEV) for w in ws]
        ref = coc.matmul_all_reduce(dx, dw, chunks=chunks)
        outs = [torch.full((m, n), float("nan"), dtype=dt, device=DEV) for _ in range(R)]
        code = coc.BF16 if dt == torch.bfloat16 else coc.FP16
        st = L.coc_matmul_all_reduce_noalloc(R, m, n, ks, _ptrs(dx), _ptrs(dw), _ptrs(outs), code,
                                             chunks, 1, stream)
        assert st == coc.OK, L.coc_last_error()
        torch.cuda.synchronize()
        expect = ref[0].double().cpu().numpy()
        for r in range(R):
            assert_close(outs[r], expect, R * ks, f"no-alloc rank {r}")
            assert torch.equal(outs[r], outs[0])
    coc.sync_status()
