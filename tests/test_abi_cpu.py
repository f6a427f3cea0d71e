"""C-ABI checks that need no GPU: the library loads, exports every entry point
include/coc.h declares, and rejects bad arguments with the documented status
before making any CUDA call.  Only argument combinations that fail host-side
validation (or are documented no-ops) are passed here: nothing reaches a kernel.
"""
import ctypes
import json
import os
import re

import pytest

from tensor_matmul_collective_gb300 import coc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "coc.h")


@pytest.fixture(scope="module")
def L():
    from tensor_matmul_collective_gb300 import build
    build.build()
    return coc.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(coc_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_match_binding():
    assert _declared() == sorted(coc.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_status_strings_and_version(L):
    names = [L.coc_status_string(i).decode() for i in range(7)]
    assert names == ["COC_OK", "COC_ERR_INVALID_ARG", "COC_ERR_SHAPE", "COC_ERR_ALIGN",
                     "COC_ERR_UNSUPPORTED", "COC_ERR_CUDA", "COC_ERR_TIMEOUT"]
    assert coc.version() == (1, 0)


# Fake, never-dereferenced device addresses: aligned and misaligned.
A = 0x7f0000000000
MIS = A + 2


def _arr(vals):
    a = (ctypes.c_void_p * len(vals))()
    for i, v in enumerate(vals):
        a[i] = v
    return a


def ar(L, R=2, m=64, n=128, ks=128, x=None, w=None, out=None, dt=1, chunks=1, fn="coc_matmul_all_reduce"):
    x = _arr([A] * R) if x is None else x
    w = _arr([A] * R) if w is None else w
    out = _arr([A] * R) if out is None else out
    return getattr(L, fn)(R, m, n, ks, x, w, out, dt, chunks, 0, None)


CONSTRAINTS = json.load(open(os.path.join(ROOT, "tests", "golden", "page_constraints.json")))


def test_rank_and_chunk_counts(L):
    # The pages split into 2/4/8 chunks and run the fused kernel at TP8;
    # 1 (no chunking / one rank) is the added degenerate value.
    assert CONSTRAINTS["chunk_counts"]["value"] == [2, 4, 8]
    for bad in (0, 3, 5, 6, 7, 16, -1):
        assert ar(L, R=bad if bad > 0 else 2, chunks=1 if bad > 0 else bad) == coc.ERR_INVALID_ARG
        assert ar(L, chunks=bad) == coc.ERR_INVALID_ARG


def test_m_must_divide_by_chunks(L):
    assert CONSTRAINTS["m_divisible_by_chunk_count"]["value"] is True
    assert ar(L, m=66, chunks=4) == coc.ERR_SHAPE
    assert ar(L, m=100, chunks=8) == coc.ERR_SHAPE
    # AllGather: m_shard % 8 == 0 already makes the gathered m divisible by
    # every allowed chunk count.


def test_bad_dtype_and_null_pointers(L):
    assert ar(L, dt=2) == coc.ERR_INVALID_ARG
    assert ar(L, x=_arr([A, None])) == coc.ERR_INVALID_ARG
    assert ar(L, out=_arr([None, A])) == coc.ERR_INVALID_ARG
    assert L.coc_matmul_all_reduce(2, 64, 128, 128, None, _arr([A] * 2), _arr([A] * 2), 1, 1, 0, None) \
        == coc.ERR_INVALID_ARG


def test_alignment(L):
    assert ar(L, x=_arr([A, MIS])) == coc.ERR_ALIGN
    assert ar(L, w=_arr([MIS, A])) == coc.ERR_ALIGN
    assert ar(L, out=_arr([A, MIS])) == coc.ERR_ALIGN
    assert ar(L, ks=100) == coc.ERR_ALIGN      # 200-byte X rows
    assert ar(L, n=132) == coc.ERR_ALIGN       # 264-byte W rows


def test_size_limits(L):
    assert ar(L, m=-64) == coc.ERR_SHAPE
    assert ar(L, n=1 << 31, chunks=1) == coc.ERR_SHAPE


def test_reduce_scatter_rows(L):
    fn = "coc_matmul_reduce_scatter"
    assert ar(L, R=4, m=66, fn=fn) == coc.ERR_SHAPE      # m % R
    assert ar(L, R=4, m=4 * 12, fn=fn) == coc.ERR_SHAPE  # (m / R) % 8


def test_all_gather_constraints(L):
    x = _arr([A] * 2)
    assert L.coc_all_gather_matmul(2, 12, 64, 64, x, x, x, 1, 1, 0, None) == coc.ERR_SHAPE   # m_shard % 8
    assert L.coc_all_gather_matmul(2, 16, 60, 64, x, x, x, 1, 1, 0, None) == coc.ERR_ALIGN   # n_shard rows
    assert L.coc_all_gather_matmul_v2(2, 16, 64, 64, x, x, x, None, 1, 1, 0, None) == coc.ERR_INVALID_ARG
    assert L.coc_all_gather_matmul_v2(2, 16, 0, 64, x, x, x, _arr([A, None]), 1, 1, 0, None) == coc.ERR_SHAPE
    assert L.coc_all_gather_matmul_v2(2, 16, 64, 64, x, x, x, _arr([A, MIS]), 1, 1, 0, None) == coc.ERR_ALIGN


def test_w8a16_constraints(L):
    x = _arr([A] * 2)
    f = L.coc_matmul_all_reduce_w8a16
    assert f(2, 64, 136, 128, x, x, x, 0, 0, x, 1, 0, None) == coc.ERR_ALIGN        # n % 16 (int8 rows)
    assert f(2, 64, 128, 128, x, x, x, 3, 0, x, 1, 0, None) == coc.ERR_INVALID_ARG  # granularity
    assert f(2, 64, 128, 128, x, x, None, 0, 0, x, 1, 0, None) == coc.ERR_INVALID_ARG
    assert f(2, 64, 128, 256, x, x, x, 2, 96, x, 1, 0, None) == coc.ERR_SHAPE       # group % 64
    assert f(2, 64, 128, 192, x, x, x, 2, 128, x, 1, 0, None) == coc.ERR_SHAPE     # k_shard % group
    assert f(2, 64, 128, 128, x, x, _arr([A, MIS]), 1, 0, x, 1, 0, None) == coc.ERR_ALIGN


def test_w8a16_ex_constraints(L):
    # extended entry point: argument order (R, m, n, k_shard, x, w, scale, zero, gran,
    # group, out, dt, chunks, det, stream); every call below fails host validation
    x = _arr([A] * 2)
    f = L.coc_matmul_all_reduce_w8a16_ex
    assert f(2, 64, 128, 128, x, x, x, None, 0, 0, x, 7, 1, 0, None) == coc.ERR_INVALID_ARG    # dtype
    assert f(2, 64, 128, 128, x, x, x, _arr([A, None]), 1, 0, x, 1, 1, 0, None) == coc.ERR_INVALID_ARG
    assert f(2, 64, 128, 128, x, x, x, _arr([A, MIS]), 1, 0, x, 0, 1, 0, None) == coc.ERR_ALIGN  # zero, channel
    assert f(2, 64, 128, 128, x, x, x, _arr([A, MIS]), 2, 64, x, 1, 1, 0, None) == coc.ERR_ALIGN  # zero, group
    assert f(2, 64, 136, 128, x, x, x, x, 0, 0, x, 1, 1, 0, None) == coc.ERR_ALIGN        # n % 16
    assert f(2, 64, 128, 128, x, x, x, x, 3, 0, x, 1, 1, 0, None) == coc.ERR_INVALID_ARG  # granularity
    assert f(2, 64, 128, 192, x, x, x, x, 2, 128, x, 0, 1, 0, None) == coc.ERR_SHAPE      # k_shard % group
    assert f(2, 0, 128, 128, x, x, x, x, 1, 0, x, 1, 1, 0, None) == coc.OK                # empty: no-op


def test_moe_constraints(L):
    # (R, tokens, h, f, experts_per_rank, x, idx, w, xd, y, capacity, counts, offsets, dt, stream);
    # every call below fails host validation before any CUDA call
    f = L.coc_moe_dispatch_grouped_matmul
    x = _arr([A] * 2)
    cap = L.coc_moe_capacity(2, 100, 2)
    assert cap == 768                                   # 2 x 100 + 2 x 255 = 710, rounded up to 256
    assert L.coc_moe_capacity(0, 100, 1) == -1 and L.coc_moe_capacity(2, -1, 1) == -1

    def call(R=2, T=100, h=128, fo=136, el=2, xp=x, ip=x, w=A, xd=x, y=x, cap=cap, cnt=A, off=A, dt=1):
        return f(R, T, h, fo, el, xp, ip, w, xd, y, cap, cnt, off, dt, None)
    assert call(R=0) == coc.ERR_INVALID_ARG
    assert call(R=9) == coc.ERR_INVALID_ARG
    assert call(dt=5) == coc.ERR_INVALID_ARG
    assert call(el=0) == coc.ERR_INVALID_ARG
    assert call(el=129) == coc.ERR_INVALID_ARG          # 2 x 129 > 256 experts
    assert call(h=100) == coc.ERR_SHAPE                 # h % 64
    assert call(fo=100) == coc.ERR_ALIGN                # f * 2 % 16
    assert call(cap=cap - 1) == coc.ERR_SHAPE           # capacity too small
    assert call(cnt=None) == coc.ERR_INVALID_ARG
    assert call(off=A + 2) == coc.ERR_ALIGN
    assert call(w=A + 8) == coc.ERR_ALIGN
    assert call(xd=_arr([A, MIS])) == coc.ERR_ALIGN
    assert call(y=_arr([MIS, A])) == coc.ERR_ALIGN
    assert call(xp=_arr([A, MIS])) == coc.ERR_ALIGN
    assert call(y=_arr([A, None])) == coc.ERR_INVALID_ARG
    assert call(ip=_arr([A, None])) == coc.ERR_INVALID_ARG
    assert call(ip=_arr([A, A + 2])) == coc.ERR_ALIGN


def test_empty_problems_are_noops(L):
    # m == 0 or n == 0: documented no-op, returns before any CUDA call
    assert ar(L, m=0) == coc.OK
    assert ar(L, n=0) == coc.OK
    assert ar(L, m=0, fn="coc_matmul_reduce_scatter") == coc.OK
    x = _arr([A] * 2)
    assert L.coc_all_gather_matmul(2, 0, 64, 64, x, x, x, 1, 1, 0, None) == coc.OK
    assert L.coc_matmul(2, 0, 64, 64, x, x, A, 1, None) == coc.OK


def test_last_error_names_the_problem(L):
    assert ar(L, m=66, chunks=4) == coc.ERR_SHAPE
    assert b"chunks" in L.coc_last_error()


def test_binding_rejects_cpu_tensors():
    import torch
    xs = [torch.zeros(8, 8, dtype=torch.bfloat16)] * 2
    with pytest.raises(ValueError):
        coc.matmul_all_reduce(xs, xs)


def test_fused_matmul_rejects_bad_enums(L):
    x = _arr([A] * 2)
    # unknown weight layout / operator: rejected before any CUDA call
    assert L.coc_fused_matmul(0, 2, 64, 128, 128, x, x, 2, x, None, 1, 1, 0, None) == coc.ERR_INVALID_ARG
    assert L.coc_fused_matmul(7, 2, 64, 128, 128, x, x, 0, x, None, 1, 1, 0, None) == coc.ERR_INVALID_ARG
    # the named operators' checks apply: m % chunks, RS rows, V2 needs `gathered`
    assert L.coc_fused_matmul(0, 2, 66, 128, 128, x, x, 1, x, None, 1, 4, 0, None) == coc.ERR_SHAPE
    assert L.coc_fused_matmul(1, 4, 48, 128, 128, _arr([A] * 4), _arr([A] * 4), 1, _arr([A] * 4), None, 1, 1, 0,
                              None) == coc.ERR_SHAPE
    assert L.coc_fused_matmul(3, 2, 16, 64, 64, x, x, 1, x, None, 1, 1, 0, None) == coc.ERR_INVALID_ARG
    assert L.coc_fused_matmul(0, 2, 0, 128, 128, x, x, 1, x, None, 1, 1, 0, None) == coc.OK   # empty: no-op


def test_weight_grad_argument_checks(L):
    x = _arr([A] * 2)
    # (rows, cols, inner) = (out_features, in_features, tokens)
    assert L.coc_fused_matmul(4, 2, 64, 128, 256, x, x, 1, x, None, 1, 1, 0, None) == coc.ERR_INVALID_ARG  # n x k
    assert L.coc_fused_matmul(4, 2, 60, 128, 256, x, x, 0, x, None, 1, 1, 0, None) == coc.ERR_ALIGN        # dY rows
    assert L.coc_fused_matmul(4, 2, 64, 132, 256, x, x, 0, x, None, 1, 1, 0, None) == coc.ERR_ALIGN        # X rows
    assert L.coc_fused_matmul(4, 2, 64, 128, 256, x, x, 0, x, None, 1, 3, 0, None) == coc.ERR_INVALID_ARG  # chunks
    assert L.coc_fused_matmul(4, 2, 0, 128, 256, x, x, 0, x, None, 1, 1, 0, None) == coc.OK                # empty
