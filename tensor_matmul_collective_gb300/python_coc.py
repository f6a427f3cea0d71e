"""Python-script CoC: the comparison path for the fused operators.

CoC page, 解决思路 / Python脚本层面实现 (Python-side implementation): the
left matrix is cut along m into C chunks; each chunk's matmul runs on a
compute stream and its collective on a communication stream, so chunk c's
collective overlaps chunk c+1's matmul, and the chunks are concatenated at
the end.  The page notes that with many chunks the host issues so many
operations per layer that it becomes host bound; the fused operators in
``coc`` run the same schedule inside one persistent kernel instead.

This module is PyTorch only and is NOT the product path: it exists to be
measured against the fused kernels (the bench's context section) and is
checked against the oracle like them.  On one GPU the R ranks are R shard
buffers, so the "collective" of a chunk is a reduction of the ranks' partial
products (AllReduce / ReduceScatter) or a copy of the gathered rows
(AllGather) into the rank buffers:

* every per-rank matmul returns the activation dtype (what a framework's
  matmul hands to its collective), and the ranks' partials of a chunk are
  summed in fp32 in rank order 0..R-1 and rounded once;
* the copies into the R rank buffers run on the communication stream.

Pass ``comp`` / ``comm`` streams on a GPU; with None (CPU tensors) the same
steps run in program order.
"""
from __future__ import annotations

import contextlib

import torch


def _ctx(stream):
    return torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()


def _begin(comp, comm):
    if comp is None:
        return None
    cur = torch.cuda.current_stream()
    comp.wait_stream(cur)
    comm.wait_stream(cur)
    return cur


def _end(cur, comp, comm):
    if cur is not None:
        cur.wait_stream(comp)
        cur.wait_stream(comm)


def _handoff(t, comp, comm):
    """Make the communication stream wait for the compute stream's result t."""
    if comp is None:
        return
    ev = torch.cuda.Event()
    ev.record(comp)
    comm.wait_event(ev)
    t.record_stream(comm)


def _reduced_rows(xs, ws, sl):
    acc = torch.matmul(xs[0][sl], ws[0]).float()
    for r in range(1, len(xs)):
        acc += torch.matmul(xs[r][sl], ws[r]).float()
    return acc.to(xs[0].dtype)


def all_reduce(xs, ws, outs, chunks: int, comp=None, comm=None):
    """MATMUL_ALL_REDUCE by chunks: outs[r][rows of c] = sum_q xs[q][rows of c] @ ws[q].

    xs[r]: m x k_shard, ws[r]: k_shard x n, outs[r]: m x n; m % chunks == 0."""
    m = xs[0].shape[0]
    if chunks < 1 or m % chunks:
        raise ValueError(f"m={m} is not divisible into {chunks} chunks")
    rows = m // chunks
    cur = _begin(comp, comm)
    for c in range(chunks):
        sl = slice(c * rows, (c + 1) * rows)
        with _ctx(comp):
            red = _reduced_rows(xs, ws, sl)
        _handoff(red, comp, comm)
        with _ctx(comm):
            for o in outs:
                o[sl].copy_(red)
    _end(cur, comp, comm)
    return outs


def reduce_scatter(xs, ws, outs, chunks: int, comp=None, comm=None):
    """MATMUL_REDUCE_SCATTER by chunks: rank r keeps rows [r m/R, (r+1) m/R) of the sum.

    Chunk c covers rows [c m/C, (c+1) m/C) of the full product; its reduced
    rows are scattered to the ranks that own them.  outs[r]: (m/R) x n."""
    m, R = xs[0].shape[0], len(xs)
    if chunks < 1 or m % chunks or m % R:
        raise ValueError(f"m={m} must be divisible by chunks={chunks} and R={R}")
    rows, per_rank = m // chunks, m // R
    cur = _begin(comp, comm)
    for c in range(chunks):
        lo, hi = c * rows, (c + 1) * rows
        with _ctx(comp):
            red = _reduced_rows(xs, ws, slice(lo, hi))
        _handoff(red, comp, comm)
        with _ctx(comm):
            for r in range(R):
                a, b = max(lo, r * per_rank), min(hi, (r + 1) * per_rank)
                if a < b:
                    outs[r][a - r * per_rank:b - r * per_rank].copy_(red[a - lo:b - lo])
    _end(cur, comp, comm)
    return outs


def all_gather(xs, ws, outs, chunks: int, gathered=None, comp=None, comm=None):
    """ALL_GATHER_MATMUL by chunks: outs[r] = concat_q(xs[q]) @ ws[r].

    xs[q]: m_shard x k, ws[r]: k x n_shard, outs[r]: (R m_shard) x n_shard.
    The gathered rows of chunk c are assembled on the communication stream
    (the collective) and multiplied on the compute stream while chunk c+1 is
    gathered; ``gathered`` (R buffers of (R m_shard) x k, optional) receives
    the gathered input as ALL_GATHER_MATMUL_V2 returns it."""
    R, ms = len(xs), xs[0].shape[0]
    m = R * ms
    if chunks < 1 or m % chunks:
        raise ValueError(f"gathered m={m} is not divisible into {chunks} chunks")
    rows = m // chunks
    cur = _begin(comp, comm)
    for c in range(chunks):
        lo, hi = c * rows, (c + 1) * rows
        with _ctx(comm):
            parts = []
            for q in range(R):
                a, b = max(lo, q * ms), min(hi, (q + 1) * ms)
                if a < b:
                    parts.append(xs[q][a - q * ms:b - q * ms])
            xg = torch.cat(parts, 0)
            if gathered is not None:
                for g in gathered:
                    g[lo:hi].copy_(xg)
        if comp is not None:
            ev = torch.cuda.Event()
            ev.record(comm)
            comp.wait_event(ev)
            xg.record_stream(comp)
        with _ctx(comp):
            for r in range(R):
                torch.matmul(xg, ws[r], out=outs[r][lo:hi])
    _end(cur, comp, comm)
    return outs
