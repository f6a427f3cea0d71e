"""fp64 CPU oracle for the fused tensor-parallel matmul + collective operators.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference legs may import this module.  It shares
no code with the CUDA path (``tensor_matmul_collective_gb300``) and the CUDA path
never imports it.

Every operator is written out from its definition.  The pages are the MindSpeed
developer guide page on compute-communication parallelism ("CoC"), sections
问题分析 (problem analysis) and 融合算子实现 (fused-operator implementation),
and the blog "MindSpeed LLM通信计算重叠与MC2如何榨干昇腾芯片算力", section
第三层CoC.  They name the operators and the Megatron layers they fuse; the
layouts are the standard Megatron tensor-parallel ones:

* RowParallelLinear splits the contraction dimension: rank r holds
  X_r (m x k_r) and W_r (k_r x n).  Without sequence parallelism the matmul is
  followed by AllReduce, with it by ReduceScatter along the rows.
* ColumnParallelLinear with sequence parallelism splits the rows of the input
  (rank r holds X_r, m_s x k) and the columns of the weight (W_r, k x n_s); the
  input is AllGathered along the rows before the matmul.

Inputs are 16-bit bit patterns (numpy uint16) tagged F16 or BF16, int8 arrays
for the quantised weight.  Results are fp64 arrays, except the AllGather
intermediate (a bit-exact copy) and the dequantised weight (binary16 bits).

Parity pins (tests/test_oracle_pins.py): exact rational brute force on tiny
inputs, R=1 and unsharded equivalence with numpy.matmul in float64, the
shard invariants, and numpy's own binary16 conversion for the rounding helper.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F16 = 0
BF16 = 1

SCALE_TENSOR = 0
SCALE_CHANNEL = 1
SCALE_GROUP = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O3", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-shared", "-fPIC", _SRC, "-o", _LIB, "-lm"]
        subprocess.run(cmd, check=True)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_f16_to_f64.restype = ctypes.c_double
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_f64_to_f16_rne.restype = ctypes.c_uint16
            lib.oracle_f64_to_f16_rne.argtypes = [ctypes.c_double]
            lib.oracle_decode16.argtypes = [ctypes.c_int, p, p, i64]
            lib.oracle_encode_f16.argtypes = [p, p, i64]
            lib.oracle_accumulate_partial.argtypes = [
                ctypes.c_int, p, i64, p, i64, i64, i64, p, i64, p, ctypes.c_int]
            lib.oracle_dequant_w8.argtypes = [p, i64, i64, p, ctypes.c_int, i64, i64, p]
            lib.oracle_dequant_w8_ex.argtypes = [p, i64, i64, p, p, ctypes.c_int, i64, i64, ctypes.c_int, p]
            lib.oracle_encode_bf16.argtypes = [p, p, i64]
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bit patterns, got {a.dtype}")
    return a


# ---------------------------------------------------------------- formats ---

def decode16(bits, dtype: int) -> np.ndarray:
    """Exact widening of binary16 (F16) or bfloat16 (BF16) bit patterns to fp64."""
    b = _c16(bits)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_decode16(int(dtype), _ptr(b), _ptr(out), b.size)
    return out


def encode_f16(values) -> np.ndarray:
    """Round fp64 values to binary16 (ties to even, overflow to inf); returns bits."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_encode_f16(_ptr(v), _ptr(out), v.size)
    return out


def encode_bf16(values) -> np.ndarray:
    """Round fp64 values to bfloat16 (ties to even, overflow to inf); returns bits."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_encode_bf16(_ptr(v), _ptr(out), v.size)
    return out


# ------------------------------------------------------ partial products ---

def partial_sum(dtype: int, xs, ws, rows, nthreads: int | None = None) -> np.ndarray:
    """sum_r X_r[rows, :] @ W_r in fp64, summed r ascending then t ascending.

    xs[r]: (m x k_r) bits, ws[r]: (k_r x n) bits; rows: int64 row indices.
    """
    if len(xs) != len(ws) or len(xs) == 0:
        raise ValueError("need one W per X and at least one rank")
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = ws[0].shape[1]
    acc = np.zeros((rows.size, n), dtype=np.float64)
    nth = nthreads or max_threads()
    lib = _load()
    for x, w in zip(xs, ws):
        x = _c16(x)
        w = _c16(w)
        if x.shape[1] != w.shape[0] or w.shape[1] != n:
            raise ValueError("shard shapes do not chain")
        if rows.size and (rows.min() < 0 or rows.max() >= x.shape[0]):
            raise IndexError("row outside X")
        lib.oracle_accumulate_partial(int(dtype), _ptr(x), x.shape[1], _ptr(w), w.shape[1],
                                      w.shape[0], n, _ptr(rows), rows.size, _ptr(acc), nth)
    return acc


def _all_rows(m: int) -> np.ndarray:
    return np.arange(m, dtype=np.int64)


# -------------------------------------------------------------- operators ---

def matmul_all_reduce(dtype: int, xs, ws, rows=None, nthreads=None) -> np.ndarray:
    """MATMUL_ALL_REDUCE (CoC page, 融合算子实现, first bullet).

    Row-parallel matmul then AllReduce: every rank ends with
    Y = sum_r X_r @ W_r.  Returns Y[rows] (fp64); each of the R rank outputs
    must equal it.
    """
    m = xs[0].shape[0]
    rows = _all_rows(m) if rows is None else rows
    return partial_sum(dtype, xs, ws, rows, nthreads)


def matmul_reduce_scatter(dtype: int, xs, ws, rank: int, local_rows=None, nthreads=None) -> np.ndarray:
    """MATMUL_REDUCE_SCATTER (same section, second bullet).

    Row-parallel matmul then ReduceScatter along the rows (sequence
    parallelism): rank `rank` receives rows [rank*m/R, (rank+1)*m/R) of
    Y = sum_r X_r @ W_r.  Returns out_rank[local_rows].
    """
    R = len(xs)
    m = xs[0].shape[0]
    if m % R:
        raise ValueError("ReduceScatter needs m divisible by the rank count")
    ms = m // R
    local_rows = _all_rows(ms) if local_rows is None else np.asarray(local_rows, dtype=np.int64)
    return partial_sum(dtype, xs, ws, rank * ms + local_rows, nthreads)


def all_gather(xs) -> np.ndarray:
    """The AllGather intermediate: X_0, ..., X_{R-1} stacked along rows, rank order."""
    return np.concatenate([_c16(x) for x in xs], axis=0)


def all_gather_matmul(dtype: int, xs, ws, rank: int, rows=None, nthreads=None) -> np.ndarray:
    """ALL_GATHER_MATMUL (same section, third bullet): out_rank = AllGather(X) @ W_rank.

    Returns out_rank[rows] (rows index the gathered m = R * m_s).
    """
    xg = all_gather(xs)
    rows = _all_rows(xg.shape[0]) if rows is None else rows
    return partial_sum(dtype, [xg], [ws[rank]], rows, nthreads)


def all_gather_matmul_v2(dtype: int, xs, ws, rank: int, rows=None, nthreads=None):
    """ALL_GATHER_MATMUL_V2: as ALL_GATHER_MATMUL, and the AllGather result is
    also returned (the V2 form gives the caller the gathered input as well).
    Returns (out_rank[rows], gathered bits)."""
    return all_gather_matmul(dtype, xs, ws, rank, rows, nthreads), all_gather(xs)


def dequant_w8a16(wq, scale_bits, gran: int, group: int = 0, k_offset: int = 0) -> np.ndarray:
    """Pseudo-quantised weight of one rank: binary16 bits of RNE(q * s).

    wq: (k x n) int8 slab; scale_bits: binary16 bits of the scale tensor —
    shape (1,) per tensor, (n,) per channel, (K/group, n) per group indexed by
    global row (k_offset + t) / group.
    """
    q = np.ascontiguousarray(wq, dtype=np.int8)
    s = _c16(scale_bits)
    k, n = q.shape
    if gran == SCALE_TENSOR:
        need = 1
    elif gran == SCALE_CHANNEL:
        need = n
    elif gran == SCALE_GROUP:
        if group <= 0:
            raise ValueError("group size must be positive")
        need = ((k_offset + k - 1) // group + 1) * n if k else 0
    else:
        raise ValueError("unknown scale granularity")
    if s.size < need:
        raise ValueError("scale tensor too small for this granularity")
    out = np.empty((k, n), dtype=np.uint16)
    _load().oracle_dequant_w8(_ptr(q), k, n, _ptr(s), int(gran), int(group), int(k_offset), _ptr(out))
    return out


def dequant_w8a16_ex(wq, scale_bits, gran: int, group: int = 0, k_offset: int = 0, zero=None,
                     dtype: int = F16) -> np.ndarray:
    """Extended w8A16 weight of one rank: bits (in `dtype`) of RNE((q - z) * s).

    The zero point `zero` (int8, laid out like the scale; None = symmetric)
    and the bfloat16 activation type are the plain reading of the pages'
    antiquant-offset and bf16-activation extensions; the scale is in `dtype`
    too.  With zero=None and dtype=F16 this is dequant_w8a16.
    """
    q = np.ascontiguousarray(wq, dtype=np.int8)
    s = _c16(scale_bits)
    k, n = q.shape
    if gran == SCALE_TENSOR:
        need = 1
    elif gran == SCALE_CHANNEL:
        need = n
    elif gran == SCALE_GROUP:
        if group <= 0:
            raise ValueError("group size must be positive")
        need = ((k_offset + k - 1) // group + 1) * n if k else 0
    else:
        raise ValueError("unknown scale granularity")
    if s.size < need:
        raise ValueError("scale tensor too small for this granularity")
    z = None
    if zero is not None:
        z = np.ascontiguousarray(zero, dtype=np.int8)
        if z.size < need:
            raise ValueError("zero-point tensor too small for this granularity")
    out = np.empty((k, n), dtype=np.uint16)
    _load().oracle_dequant_w8_ex(_ptr(q), k, n, _ptr(s), _ptr(z) if z is not None else None, int(gran), int(group),
                                 int(k_offset), int(dtype), _ptr(out))
    return out


def matmul_all_reduce_w8a16(xs, wqs, scales, gran: int, group: int = 0, rows=None, nthreads=None, zeros=None,
                            dtype: int = F16):
    """w8A16 MATMUL_ALL_REDUCE (same section, last bullet).

    xs[r]: activation bits (m x k_r) in `dtype` (the page's fp16, or the
    bfloat16 extension); wqs[r]: int8 (k_r x n); scales[r]: this rank's scale
    view in `dtype` (the shared scalar, the shared per-column vector, or this
    rank's rows of the per-group table, so k_offset is 0 within the view);
    zeros[r]: optional int8 zero points laid out like scales[r].
    Y = sum_r X_r @ Wd_r with Wd_r the dequantised weight.
    """
    if zeros is None and dtype == F16:
        wds = [dequant_w8a16(wq, s, gran, group, 0) for wq, s in zip(wqs, scales)]
    else:
        zs = zeros if zeros is not None else [None] * len(wqs)
        wds = [dequant_w8a16_ex(wq, s, gran, group, 0, z, dtype) for wq, s, z in zip(wqs, scales, zs)]
    return matmul_all_reduce(dtype, xs, wds, rows, nthreads)


# ------------------------------------------- MoE dispatch + GroupedMatMul ---
#
# The MindSpeed-LLM overlap blog (section 第二层MC2) names an expert-parallel
# form of the fused operators: the MoE token all-to-all fused with the
# experts' GroupedMatMul.  It gives no formula; the reading used here is the
# plain one of expert parallelism with top-1 routing:
#
# * R expert-parallel ranks, E = R * E_loc experts, expert e held by rank
#   e // E_loc; rank r holds tokens X_r (T x h) and their expert ids idx_r.
# * Dispatch (the all-to-all): destination rank q receives every token routed
#   to one of its experts, grouped by expert (ascending), inside an expert by
#   source rank (ascending), inside a source rank by token index (ascending).
# * GroupedMatMul: each expert's group of rows times that expert's weight
#   W_e (h x f).

def moe_dispatch_order(idxs, E: int):
    """For every expert e (0..E-1): the list of (source rank, token) pairs in
    dispatch order, as an (n_e x 2) int64 array."""
    R = len(idxs)
    out = []
    for e in range(E):
        pairs = []
        for r in range(R):
            t = np.nonzero(np.asarray(idxs[r]) == e)[0]
            pairs.append(np.stack([np.full(t.size, r, dtype=np.int64), t.astype(np.int64)], axis=1))
        out.append(np.concatenate(pairs, axis=0) if pairs else np.zeros((0, 2), np.int64))
    return out


def moe_dispatch_grouped_matmul(dtype: int, xs, idxs, ws, nthreads=None):
    """Dispatch + GroupedMatMul.  xs[r]: token bits (T x h) in `dtype`;
    idxs[r]: int expert ids (T); ws[e]: expert weight bits (h x f), E = len(ws).
    Returns, per expert e, (pairs_e, Xd_e, Y_e): the dispatch order, the
    dispatched token bits (n_e x h, a bit-exact copy) and Y_e = Xd_e @ W_e in
    fp64 (n_e x f)."""
    E = len(ws)
    res = []
    for e, pairs in enumerate(moe_dispatch_order(idxs, E)):
        h = xs[0].shape[1]
        Xd = np.empty((pairs.shape[0], h), dtype=np.uint16)
        for i, (r, t) in enumerate(pairs):
            Xd[i] = xs[r][t]
        f = ws[e].shape[1]
        Y = matmul_all_reduce(dtype, [Xd], [ws[e]], None, nthreads) if pairs.shape[0] else np.zeros((0, f))
        res.append((pairs, Xd, Y))
    return res


def moe_token_outputs(dtype: int, xs, idxs, ws, nthreads=None):
    """The combine (all-to-all back) written per token, without any dispatch
    order: Y_r[t] = X_r[t] @ W_{idx_r[t]} (fp64), rows of ids outside [0, E)
    left NaN.  Returns one (T x f) array per rank."""
    E = len(ws)
    f = ws[0].shape[1]
    out = []
    for x, idx in zip(xs, idxs):
        idx = np.asarray(idx)
        Y = np.full((x.shape[0], f), np.nan)
        for e in range(E):
            rows = np.nonzero(idx == e)[0]
            if rows.size:
                Y[rows] = matmul_all_reduce(dtype, [x], [ws[e]], rows, nthreads)
        out.append(Y)
    return out


def moe_topk_combine(dtype: int, xs, idxs, gates, ws, nthreads=None):
    """Top-k combine: out_r[t] = sum_j g[t, j] * rne_dtype(X_r[t] @ W_{idx[t, j]})
    (the expert outputs in the activation type, as the GroupedMatMul
    produces them, weighted and summed in fp64).  idxs[r] / gates[r]: T x k.
    Entries with an id outside [0, E) contribute nothing."""
    E = len(ws)
    f = ws[0].shape[1]
    enc = encode_bf16 if dtype == BF16 else encode_f16
    out = []
    for x, idx, g in zip(xs, idxs, gates):
        idx = np.asarray(idx).reshape(x.shape[0], -1)
        g = np.asarray(g, dtype=np.float64).reshape(idx.shape)
        acc = np.zeros((x.shape[0], f))
        for j in range(idx.shape[1]):
            for e in range(E):
                rows = np.nonzero(idx[:, j] == e)[0]
                if rows.size:
                    Y = decode16(enc(matmul_all_reduce(dtype, [x], [ws[e]], rows, nthreads)), dtype)
                    acc[rows] += g[rows, j:j + 1] * Y
        out.append(acc)
    return out
