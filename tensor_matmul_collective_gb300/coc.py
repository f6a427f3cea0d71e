"""Python binding of the C ABI in include/coc.h (ctypes; argument marshalling only).

Every operator runs in the library's CUDA kernels.  PyTorch is used for device
memory (tensors, optional output allocation) and for the current stream.  If
libcoc.so is missing or cannot be loaded the binding raises: there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcoc.so")

OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_ALIGN, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = range(7)
FP16, BF16 = 0, 1
SCALE_TENSOR, SCALE_CHANNEL, SCALE_GROUP = 0, 1, 2
_GRAN = {"tensor": SCALE_TENSOR, "channel": SCALE_CHANNEL, "group": SCALE_GROUP}
MAX_RANKS = 8

# Every symbol include/coc.h declares (checked by the CPU test suite).
EXPORTS = (
    "coc_matmul_all_reduce", "coc_matmul_reduce_scatter", "coc_all_gather_matmul",
    "coc_all_gather_matmul_v2", "coc_matmul_all_reduce_w8a16", "coc_matmul",
    "coc_sync_status", "coc_status_string", "coc_last_error", "coc_version",
    "coc_debug_inject_timeout", "coc_shutdown", "coc_matmul_all_reduce_noalloc",
    "coc_fused_matmul", "coc_matmul_all_reduce_w8a16_ex", "coc_moe_dispatch_grouped_matmul", "coc_moe_capacity",
    "coc_moe_dispatch_grouped_matmul_combine", "coc_moe_topk_grouped_matmul_combine", "coc_debug_alloc_count",
    "coc_debug_clock_probe", "coc_debug_clock_read",
)

OP_ALL_REDUCE, OP_REDUCE_SCATTER, OP_ALL_GATHER, OP_ALL_GATHER_V2, OP_WEIGHT_GRAD = range(5)
_OPS = {"all_reduce": OP_ALL_REDUCE, "reduce_scatter": OP_REDUCE_SCATTER,
        "all_gather": OP_ALL_GATHER, "all_gather_v2": OP_ALL_GATHER_V2}
W_KN, W_NK = 0, 1


class CocError(RuntimeError):
    def __init__(self, status: int, name: str, detail: str):
        super().__init__(f"{name}: {detail}" if detail else name)
        self.status = status
        self.name = name
        self.detail = detail


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Load libcoc.so (built by __graft_entry__.build() or build.py)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(LIB_PATH)
            i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            pp = ctypes.POINTER(ctypes.c_void_p)
            row = [i32, i64, i64, i64, pp, pp, pp, i32, i32, i32, vp]
            for name in ("coc_matmul_all_reduce", "coc_matmul_reduce_scatter", "coc_all_gather_matmul",
                         "coc_matmul_all_reduce_noalloc"):
                getattr(L, name).argtypes = row
                getattr(L, name).restype = i32
            L.coc_all_gather_matmul_v2.argtypes = [i32, i64, i64, i64, pp, pp, pp, pp, i32, i32, i32, vp]
            L.coc_all_gather_matmul_v2.restype = i32
            L.coc_matmul_all_reduce_w8a16.argtypes = [i32, i64, i64, i64, pp, pp, pp, i32, i64, pp, i32, i32, vp]
            L.coc_matmul_all_reduce_w8a16.restype = i32
            L.coc_matmul_all_reduce_w8a16_ex.argtypes = [i32, i64, i64, i64, pp, pp, pp, pp, i32, i64, pp, i32, i32,
                                                         i32, vp]
            L.coc_matmul_all_reduce_w8a16_ex.restype = i32
            L.coc_moe_dispatch_grouped_matmul.argtypes = [i32, i64, i64, i64, i32, pp, pp, vp, pp, pp, i64, vp, vp,
                                                          i32, vp]
            L.coc_moe_dispatch_grouped_matmul.restype = i32
            L.coc_moe_dispatch_grouped_matmul_combine.argtypes = L.coc_moe_dispatch_grouped_matmul.argtypes
            L.coc_moe_dispatch_grouped_matmul_combine.restype = i32
            L.coc_moe_topk_grouped_matmul_combine.argtypes = [i32, i64, i32, i64, i64, i32, pp, pp, pp, vp, pp, pp, pp,
                                                              i64, vp, vp, i32, vp]
            L.coc_moe_topk_grouped_matmul_combine.restype = i32
            L.coc_moe_capacity.argtypes = [i32, i64, i32]
            L.coc_moe_capacity.restype = i64
            L.coc_fused_matmul.argtypes = [i32, i32, i64, i64, i64, pp, pp, i32, pp, pp, i32, i32, i32, vp]
            L.coc_fused_matmul.restype = i32
            L.coc_matmul.argtypes = [i32, i64, i64, i64, pp, pp, vp, i32, vp]
            L.coc_matmul.restype = i32
            L.coc_sync_status.argtypes = [vp]
            L.coc_sync_status.restype = i32
            L.coc_status_string.argtypes = [i32]
            L.coc_status_string.restype = ctypes.c_char_p
            L.coc_last_error.argtypes = []
            L.coc_last_error.restype = ctypes.c_char_p
            L.coc_version.restype = i32
            L.coc_debug_inject_timeout.argtypes = [i32]
            L.coc_debug_inject_timeout.restype = i32
            L.coc_shutdown.restype = i32
            L.coc_debug_alloc_count.argtypes = []
            L.coc_debug_alloc_count.restype = i64
            L.coc_debug_clock_probe.argtypes = [i32]
            L.coc_debug_clock_probe.restype = i32
            L.coc_debug_clock_read.argtypes = [i32, ctypes.POINTER(i64), ctypes.POINTER(i64)]
            L.coc_debug_clock_read.restype = i32
            _lib = L
    return _lib


def _check(status: int) -> None:
    if status != OK:
        L = lib()
        raise CocError(status, L.coc_status_string(status).decode(), L.coc_last_error().decode())


def _ptrs(ts) -> ctypes.Array:
    arr = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = None if t is None else t.data_ptr()
    return arr


# The current stream's handle without building a torch.cuda.Stream object
# (a few microseconds per call on the host); the public query where this
# PyTorch lacks the raw one.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int:
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float16:
        return FP16
    if dt == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {dt}; expected float16 or bfloat16")


def _check_list(ts, name, shape, dtype, device):
    if not isinstance(ts, (list, tuple)) or len(ts) == 0:
        raise ValueError(f"{name} must be a non-empty list of tensors")
    # one combined test per tensor; the checks below only word the error
    shape = tuple(shape)
    for t in ts:
        if (not isinstance(t, torch.Tensor) or t.dtype is not dtype or t.shape != shape or t.device != device
                or not t.is_contiguous()):
            break
    else:
        return
    for i, t in enumerate(ts):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name}[{i}] is not a tensor")
        if t.device != device:
            raise ValueError(f"{name}[{i}] is on {t.device}, expected {device}")
        if t.dtype != dtype:
            raise TypeError(f"{name}[{i}] has dtype {t.dtype}, expected {dtype}")
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name}[{i}] has shape {tuple(t.shape)}, expected {tuple(shape)}")
        if not t.is_contiguous():
            raise ValueError(f"{name}[{i}] is not contiguous")


def _prep(xs, ws):
    if not xs or not ws or len(xs) != len(ws):
        raise ValueError("xs and ws must be lists of equal length (one tensor per rank)")
    R = len(xs)
    if R > MAX_RANKS:
        raise ValueError(f"at most {MAX_RANKS} ranks")
    x0, w0 = xs[0], ws[0]
    if x0.dim() != 2 or w0.dim() != 2:
        raise ValueError("X and W shards must be 2-D")
    _check_device(x0)
    return R, x0, w0


def _check_device(t):
    """The library works on the current CUDA device: tensors of another one
    would be addressed from the wrong context, so they are rejected here."""
    if t.device.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    cur = torch.cuda.current_device()
    if t.device.index is not None and t.device.index != cur:
        raise ValueError(f"inputs are on {t.device} but the current device is cuda:{cur}; "
                         f"call inside `with torch.cuda.device({t.device}):`")


def _outs(outs, R, shape, dtype, device):
    if outs is None:
        return [torch.empty(shape, dtype=dtype, device=device) for _ in range(R)]
    _check_list(outs, "outs", shape, dtype, device)
    if len(outs) != R:
        raise ValueError("need one output per rank")
    return list(outs)


def matmul_all_reduce(xs, ws, outs=None, chunks: int = 1, deterministic: bool = False, stream=None):
    """MATMUL_ALL_REDUCE: outs[r] = sum_q xs[q] @ ws[q] for every rank r."""
    R, x0, w0 = _prep(xs, ws)
    m, ks = x0.shape
    n = w0.shape[1]
    _check_list(xs, "xs", (m, ks), x0.dtype, x0.device)
    _check_list(ws, "ws", (ks, n), x0.dtype, x0.device)
    outs = _outs(outs, R, (m, n), x0.dtype, x0.device)
    _check(lib().coc_matmul_all_reduce(R, m, n, ks, _ptrs(xs), _ptrs(ws), _ptrs(outs), _dtype_code(x0.dtype),
                                       int(chunks), int(bool(deterministic)), _stream(stream)))
    return outs


def matmul_all_reduce_noalloc(xs, ws, outs=None, chunks: int = 1, deterministic: bool = False, stream=None):
    """MATMUL_ALL_REDUCE through the allocation-free entry point (the library
    allocates no device memory for this call; `outs` None allocates the
    outputs here, through PyTorch)."""
    R, x0, w0 = _prep(xs, ws)
    m, ks = x0.shape
    n = w0.shape[1]
    _check_list(xs, "xs", (m, ks), x0.dtype, x0.device)
    _check_list(ws, "ws", (ks, n), x0.dtype, x0.device)
    outs = _outs(outs, R, (m, n), x0.dtype, x0.device)
    _check(lib().coc_matmul_all_reduce_noalloc(R, m, n, ks, _ptrs(xs), _ptrs(ws), _ptrs(outs), _dtype_code(x0.dtype),
                                               int(chunks), int(bool(deterministic)), _stream(stream)))
    return outs


def matmul_reduce_scatter(xs, ws, outs=None, chunks: int = 1, deterministic: bool = False, stream=None):
    """MATMUL_REDUCE_SCATTER: outs[r] = rows [r*m/R, (r+1)*m/R) of sum_q xs[q] @ ws[q]."""
    R, x0, w0 = _prep(xs, ws)
    m, ks = x0.shape
    n = w0.shape[1]
    _check_list(xs, "xs", (m, ks), x0.dtype, x0.device)
    _check_list(ws, "ws", (ks, n), x0.dtype, x0.device)
    if m % R:
        raise CocError(ERR_SHAPE, "COC_ERR_SHAPE", f"m = {m} is not a multiple of R = {R}")
    outs = _outs(outs, R, (m // R, n), x0.dtype, x0.device)
    _check(lib().coc_matmul_reduce_scatter(R, m, n, ks, _ptrs(xs), _ptrs(ws), _ptrs(outs), _dtype_code(x0.dtype),
                                           int(chunks), int(bool(deterministic)), _stream(stream)))
    return outs


def _ag_common(xs, ws, outs):
    R, x0, w0 = _prep(xs, ws)
    ms, k = x0.shape
    ns = w0.shape[1]
    _check_list(xs, "xs", (ms, k), x0.dtype, x0.device)
    _check_list(ws, "ws", (k, ns), x0.dtype, x0.device)
    outs = _outs(outs, R, (R * ms, ns), x0.dtype, x0.device)
    return R, x0, ms, k, ns, outs


def all_gather_matmul(xs, ws, outs=None, chunks: int = 1, deterministic: bool = False, stream=None):
    """ALL_GATHER_MATMUL: outs[r] = cat(xs, dim=0) @ ws[r]."""
    R, x0, ms, k, ns, outs = _ag_common(xs, ws, outs)
    _check(lib().coc_all_gather_matmul(R, ms, ns, k, _ptrs(xs), _ptrs(ws), _ptrs(outs), _dtype_code(x0.dtype),
                                       int(chunks), int(bool(deterministic)), _stream(stream)))
    return outs


def all_gather_matmul_v2(xs, ws, outs=None, gathered=None, chunks: int = 1, deterministic: bool = False,
                         stream=None):
    """ALL_GATHER_MATMUL_V2: as all_gather_matmul, and gathered[r] = cat(xs, dim=0).

    `gathered` entries may be None to skip that rank's copy."""
    R, x0, ms, k, ns, outs = _ag_common(xs, ws, outs)
    if gathered is None:
        gathered = [torch.empty((R * ms, k), dtype=x0.dtype, device=x0.device) for _ in range(R)]
    else:
        if len(gathered) != R:
            raise ValueError("need one gathered entry per rank (None to skip)")
        present = [g for g in gathered if g is not None]
        if present:
            _check_list(present, "gathered", (R * ms, k), x0.dtype, x0.device)
    _check(lib().coc_all_gather_matmul_v2(R, ms, ns, k, _ptrs(xs), _ptrs(ws), _ptrs(outs), _ptrs(gathered),
                                          _dtype_code(x0.dtype), int(chunks), int(bool(deterministic)),
                                          _stream(stream)))
    return outs, gathered


def matmul_all_reduce_w8a16(xs, wqs, scales, gran, group_size: int = 0, outs=None, chunks: int = 1,
                            deterministic: bool = False, stream=None, zeros=None):
    """w8A16 MATMUL_ALL_REDUCE: outs[r] = sum_q xs[q] @ rne((wqs[q] - z_q) * s_q) for every r.

    The activations xs set the type (fp16 as on the page, or bf16); scales
    are in that type.  gran: "tensor" | "channel" | "group" (or the SCALE_*
    codes); scales[q] is rank q's view of the scale tensor.  zeros: None
    (symmetric) or one int8 zero-point view per rank, laid out like scales."""
    R, x0, w0 = _prep(xs, wqs)
    gcode = _GRAN[gran] if isinstance(gran, str) else int(gran)
    m, ks = x0.shape
    n = w0.shape[1]
    if x0.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("w8A16 activations must be fp16 or bf16")
    dt = x0.dtype
    _check_list(xs, "xs", (m, ks), dt, x0.device)
    _check_list(wqs, "wqs", (ks, n), torch.int8, x0.device)
    need = 1 if gcode == SCALE_TENSOR else n if gcode == SCALE_CHANNEL else \
        (ks // group_size) * n if group_size > 0 else 0
    for name, views, want in (("scales", scales, dt), ("zeros", zeros, torch.int8)):
        if views is None:
            continue
        if len(views) != R:
            raise ValueError(f"need one {name} view per rank")
        for i, s in enumerate(views):
            if s.dtype != want or s.device != x0.device or not s.is_contiguous():
                raise ValueError(f"{name}[{i}] must be a contiguous {want} tensor on {x0.device}")
            if s.numel() < need:
                raise ValueError(f"{name}[{i}] has {s.numel()} values, needs {need}")
    outs = _outs(outs, R, (m, n), dt, x0.device)
    _check(lib().coc_matmul_all_reduce_w8a16_ex(R, m, n, ks, _ptrs(xs), _ptrs(wqs), _ptrs(scales),
                                                _ptrs(zeros) if zeros is not None else None, gcode,
                                                int(group_size), _ptrs(outs), BF16 if dt == torch.bfloat16 else FP16,
                                                int(chunks), int(bool(deterministic)), _stream(stream)))
    return outs


def fused_matmul(op, xs, ws, w_layout: str = "kn", outs=None, gathered=None, chunks: int = 1,
                 deterministic: bool = False, stream=None):
    """Any of the four fused operators with a choice of weight layout.

    op: "all_reduce" | "reduce_scatter" | "all_gather" | "all_gather_v2".
    w_layout: "kn" (W_r is inner x cols, as the named functions) or "nk"
    (W_r is cols x inner: Megatron's [out_features, in_features]).
    Returns outs, or (outs, gathered) for "all_gather_v2"."""
    code = _OPS[op] if isinstance(op, str) else int(op)
    nk = {"kn": False, "nk": True}[w_layout]
    R, x0, w0 = _prep(xs, ws)
    rows, inner = x0.shape
    cols = w0.shape[0] if nk else w0.shape[1]
    wshape = (cols, inner) if nk else (inner, cols)
    _check_list(xs, "xs", (rows, inner), x0.dtype, x0.device)
    _check_list(ws, "ws", wshape, x0.dtype, x0.device)
    if code == OP_REDUCE_SCATTER:
        if rows % R:
            raise CocError(ERR_SHAPE, "COC_ERR_SHAPE", f"m = {rows} is not a multiple of R = {R}")
        oshape = (rows // R, cols)
    elif code in (OP_ALL_GATHER, OP_ALL_GATHER_V2):
        oshape = (R * rows, cols)
    else:
        oshape = (rows, cols)
    outs = _outs(outs, R, oshape, x0.dtype, x0.device)
    if code == OP_ALL_GATHER_V2:
        if gathered is None:
            gathered = [torch.empty((R * rows, inner), dtype=x0.dtype, device=x0.device) for _ in range(R)]
        elif len(gathered) != R:
            raise ValueError("need one gathered entry per rank (None to skip)")
        else:
            present = [g for g in gathered if g is not None]
            if present:
                _check_list(present, "gathered", (R * rows, inner), x0.dtype, x0.device)
        gptr = _ptrs(gathered)
    else:
        gptr = None
    _check(lib().coc_fused_matmul(code, R, rows, cols, inner, _ptrs(xs), _ptrs(ws), W_NK if nk else W_KN,
                                  _ptrs(outs), gptr, _dtype_code(x0.dtype), int(chunks), int(bool(deterministic)),
                                  _stream(stream)))
    return (outs, gathered) if code == OP_ALL_GATHER_V2 else outs


def weight_grad(dys, xs, outs=None, chunks: int = 1, stream=None):
    """Weight gradient of a TP linear layer on every rank: outs[r] = dys[r]^T @ xs[r].

    dys[r]: tokens x out_features, xs[r]: tokens x in_features (for a
    ColumnParallel layer with sequence parallelism, the gathered input that
    all_gather_matmul_v2 returned), outs[r]: out_features x in_features."""
    R, d0, x0 = _prep(dys, xs)
    inner, rows = d0.shape
    cols = x0.shape[1]
    _check_list(dys, "dys", (inner, rows), d0.dtype, d0.device)
    _check_list(xs, "xs", (inner, cols), d0.dtype, d0.device)
    outs = _outs(outs, R, (rows, cols), d0.dtype, d0.device)
    _check(lib().coc_fused_matmul(OP_WEIGHT_GRAD, R, rows, cols, inner, _ptrs(dys), _ptrs(xs), W_KN, _ptrs(outs),
                                  None, _dtype_code(d0.dtype), int(chunks), 1, _stream(stream)))
    return outs


def moe_capacity(R: int, tokens: int, experts_per_rank: int) -> int:
    """Rows each destination buffer of moe_dispatch_grouped_matmul needs."""
    v = int(lib().coc_moe_capacity(int(R), int(tokens), int(experts_per_rank)))
    if v < 0:
        raise ValueError("bad MoE capacity arguments")
    return v


def moe_dispatch_grouped_matmul(xs, idxs, w, experts_per_rank: int, xd=None, y=None, counts=None, offsets=None,
                                stream=None, combine: bool = False):
    """MoE token dispatch (all-to-all) + expert GroupedMatMul on every rank.

    xs[r]: tokens x h (fp16/bf16); idxs[r]: int32 expert ids; w: experts x h x
    f stacked weights (expert e = rank e // experts_per_rank).  Returns
    (y, xd, counts, offsets): expert e's rows are offsets[e] ..
    offsets[e] + counts[e] - 1 of y[q] / xd[q] with q = e // experts_per_rank.
    combine=True adds the all-to-all back: y[r] is then tokens x f, row t the
    output of rank r's token t."""
    R = len(xs)
    if R < 1 or R > MAX_RANKS or len(idxs) != R:
        raise ValueError("need 1..8 ranks and one idx per rank")
    x0 = xs[0]
    T, h = x0.shape
    if x0.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("tokens must be fp16 or bf16")
    _check_device(x0)
    dt = x0.dtype
    _check_list(xs, "xs", (T, h), dt, x0.device)
    _check_list(idxs, "idxs", (T,), torch.int32, x0.device)
    E = R * int(experts_per_rank)
    if w.dim() != 3 or w.shape[0] != E or w.shape[1] != h or w.dtype != dt or w.device != x0.device \
            or not w.is_contiguous():
        raise ValueError(f"w must be a contiguous {dt} tensor of shape ({E}, {h}, f) on {x0.device}")
    f = w.shape[2]
    cap = moe_capacity(R, T, experts_per_rank)
    xd = _outs(xd, R, (cap, h), dt, x0.device)
    y = _outs(y, R, (T, f) if combine else (cap, f), dt, x0.device)
    if counts is None:
        counts = torch.empty(E, dtype=torch.int32, device=x0.device)
    if offsets is None:
        offsets = torch.empty(E, dtype=torch.int32, device=x0.device)
    _check_list([counts, offsets], "counts/offsets", (E,), torch.int32, x0.device)
    fn = lib().coc_moe_dispatch_grouped_matmul_combine if combine else lib().coc_moe_dispatch_grouped_matmul
    _check(fn(R, T, h, f, int(experts_per_rank), _ptrs(xs), _ptrs(idxs), w.data_ptr(), _ptrs(xd), _ptrs(y), cap,
              counts.data_ptr(), offsets.data_ptr(), _dtype_code(dt), _stream(stream)))
    return y, xd, counts, offsets


def moe_topk_grouped_matmul_combine(xs, idxs, gates, w, experts_per_rank: int, xd=None, y=None, y_tok=None,
                                    counts=None, offsets=None, stream=None):
    """Top-k MoE: dispatch every (token, slot) entry, GroupedMatMul, gated
    combine.  idxs[r] / gates[r]: tokens x k int32 / float32.  Returns
    (y_tok, y, xd, counts, offsets); y_tok[r] is tokens x f."""
    R = len(xs)
    if R < 1 or R > MAX_RANKS or len(idxs) != R or len(gates) != R:
        raise ValueError("need 1..8 ranks and one idx / gates tensor per rank")
    x0 = xs[0]
    T, h = x0.shape
    if x0.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("tokens must be fp16 or bf16")
    _check_device(x0)
    dt = x0.dtype
    k = idxs[0].shape[1] if idxs[0].dim() == 2 else 1
    _check_list(xs, "xs", (T, h), dt, x0.device)
    _check_list(idxs, "idxs", (T, k), torch.int32, x0.device)
    _check_list(gates, "gates", (T, k), torch.float32, x0.device)
    E = R * int(experts_per_rank)
    if w.dim() != 3 or w.shape[0] != E or w.shape[1] != h or w.dtype != dt or w.device != x0.device \
            or not w.is_contiguous():
        raise ValueError(f"w must be a contiguous {dt} tensor of shape ({E}, {h}, f) on {x0.device}")
    f = w.shape[2]
    cap = moe_capacity(R, T * k, experts_per_rank)
    xd = _outs(xd, R, (cap, h), dt, x0.device)
    y = _outs(y, R, (cap, f), dt, x0.device)
    y_tok = _outs(y_tok, R, (T, f), dt, x0.device)
    if counts is None:
        counts = torch.empty(E, dtype=torch.int32, device=x0.device)
    if offsets is None:
        offsets = torch.empty(E, dtype=torch.int32, device=x0.device)
    _check_list([counts, offsets], "counts/offsets", (E,), torch.int32, x0.device)
    _check(lib().coc_moe_topk_grouped_matmul_combine(R, T, k, h, f, int(experts_per_rank), _ptrs(xs), _ptrs(idxs),
                                                     _ptrs(gates), w.data_ptr(), _ptrs(xd), _ptrs(y), _ptrs(y_tok),
                                                     cap, counts.data_ptr(), offsets.data_ptr(), _dtype_code(dt),
                                                     _stream(stream)))
    return y_tok, y, xd, counts, offsets


def matmul(xs, ws, out=None, stream=None):
    """Plain sharded contraction into one buffer (the fused-overhead baseline)."""
    R, x0, w0 = _prep(xs, ws)
    m, ks = x0.shape
    n = w0.shape[1]
    _check_list(xs, "xs", (m, ks), x0.dtype, x0.device)
    _check_list(ws, "ws", (ks, n), x0.dtype, x0.device)
    if out is None:
        out = torch.empty((m, n), dtype=x0.dtype, device=x0.device)
    else:
        _check_list([out], "out", (m, n), x0.dtype, x0.device)
    _check(lib().coc_matmul(R, m, n, ks, _ptrs(xs), _ptrs(ws), out.data_ptr(), _dtype_code(x0.dtype),
                            _stream(stream)))
    return out


def sync_status(stream=None) -> None:
    """Wait for the stream and raise CocError if a kernel's bounded wait ran out."""
    _check(lib().coc_sync_status(_stream(stream)))


def inject_timeout(enable: bool) -> None:
    """Test hook: make subsequently launched kernels stop with COC_ERR_TIMEOUT."""
    _check(lib().coc_debug_inject_timeout(int(bool(enable))))


def alloc_count() -> int:
    """Device allocations the library has made in this process (an audit hook)."""
    return int(lib().coc_debug_alloc_count())


def clock_probe(slot: int) -> None:
    """Fused kernels launched from now on add their block-0 SM cycles and ns
    to clock slot `slot` (0..7); -1 stops recording."""
    _check(lib().coc_debug_clock_probe(int(slot)))


def clock_read(slot: int):
    """(cycles, ns) accumulated in a clock slot since its last read (waits for
    the device); cycles / ns * 1e3 is the SM clock in MHz."""
    c, n = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().coc_debug_clock_read(int(slot), ctypes.byref(c), ctypes.byref(n)))
    return c.value, n.value


def clock_mhz(slot: int):
    """The SM clock (MHz) the kernels recorded in `slot` ran at, None if none ran."""
    c, n = clock_read(slot)
    return round(1e3 * c / n, 1) if n > 0 else None


def shutdown() -> None:
    _check(lib().coc_shutdown())


def version() -> tuple:
    v = lib().coc_version()
    return (v >> 16, v & 0xFFFF)
