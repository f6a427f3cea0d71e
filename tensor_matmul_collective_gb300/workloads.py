"""Seeded synthetic inputs shaped like the tensor-parallel layers the CoC pages
measure on (BLOOM-7B, BLOOM-176B and LLaMA2-70B with TP8).

This module draws numbers and slices them into shards; it holds none of the
operators' arithmetic.  Both the CUDA path's tests/benchmark and the CPU oracle
consume the arrays it returns.

Recipe: a named workload fixes the shapes, the value distributions and a seed.
The full unsharded matrices are drawn in fp32 (int8 for quantised weights),
cast to the 16-bit type with round-to-nearest-even, and the rank shards are
slices of them.  Draws are made in fixed blocks of rows, each block from its
own PCG64 stream keyed by (seed, tensor id, block index), so generation runs in
parallel threads and gives the same bits on any host and thread count.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

_BLOCK_ROWS = 64
_THREADS = max(1, min(32, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1))


def _fill_blocks(out: np.ndarray, seed: int, tensor_id: int, draw) -> np.ndarray:
    rows = out.shape[0]
    nblk = (rows + _BLOCK_ROWS - 1) // _BLOCK_ROWS

    def job(b):
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor_id, b])))
        draw(g, out[b * _BLOCK_ROWS:(b + 1) * _BLOCK_ROWS])

    if nblk <= 1:
        for b in range(nblk):
            job(b)
    else:
        with ThreadPoolExecutor(min(_THREADS, nblk)) as ex:
            list(ex.map(job, range(nblk)))
    return out


def normal(shape, std: float, seed: int, tensor_id: int) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)

    def draw(g, blk):
        g.standard_normal(out=blk, dtype=np.float32)
        if std != 1.0:
            blk *= np.float32(std)
    return _fill_blocks(out, seed, tensor_id, draw)


def uniform(shape, lo: float, hi: float, seed: int, tensor_id: int) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)

    def draw(g, blk):
        g.random(out=blk, dtype=np.float32)
        blk *= np.float32(hi - lo)
        blk += np.float32(lo)
    return _fill_blocks(out, seed, tensor_id, draw)


def int8_uniform(shape, lo: int, hi: int, seed: int, tensor_id: int) -> np.ndarray:
    """Integers uniform on [lo, hi] inclusive."""
    out = np.empty(shape, dtype=np.int8)

    def draw(g, blk):
        blk[...] = g.integers(lo, hi + 1, size=blk.shape, dtype=np.int8)
    return _fill_blocks(out, seed, tensor_id, draw)


def to16(a: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    """fp32 -> fp16/bf16 with round-to-nearest-even (torch's cast)."""
    return torch.from_numpy(a).to(dtype)


def _draw(kind: str, shape, seed: int, tid: int) -> np.ndarray:
    if kind == "normal(0,1)":
        return normal(shape, 1.0, seed, tid)
    if kind == "normal(0,0.02)":
        return normal(shape, 0.02, seed, tid)
    if kind == "uniform[-1,1]":
        return uniform(shape, -1.0, 1.0, seed, tid)
    raise ValueError(kind)


# ------------------------------------------------------------- workloads ---

@dataclass
class RowParallel:
    """Row-parallel shapes (AllReduce / ReduceScatter): X_r m x k_shard, W_r k_shard x n."""
    R: int
    m: int
    n: int
    k_shard: int
    dtype: torch.dtype
    x_dist: str
    w_dist: str
    seed: int

    @property
    def K(self) -> int:
        return self.R * self.k_shard

    def flops(self) -> float:
        return 2.0 * self.m * self.n * self.K

    def make(self):
        """Returns (xs, ws): lists of R contiguous CPU tensors."""
        X = to16(_draw(self.x_dist, (self.m, self.K), self.seed, 0), self.dtype)
        W = to16(_draw(self.w_dist, (self.K, self.n), self.seed, 1), self.dtype)
        ks = self.k_shard
        xs = [X[:, r * ks:(r + 1) * ks].contiguous() for r in range(self.R)]
        ws = [W[r * ks:(r + 1) * ks, :].contiguous() for r in range(self.R)]
        return xs, ws


@dataclass
class ColumnParallelSP:
    """Column-parallel + sequence-parallel shapes (AllGather-matmul):
    X_r m_shard x k (row shards of the gathered input), W_r k x n_shard."""
    R: int
    m_shard: int
    n_shard: int
    k: int
    dtype: torch.dtype
    x_dist: str
    w_dist: str
    seed: int

    @property
    def m(self) -> int:
        return self.R * self.m_shard

    def flops(self) -> float:
        return 2.0 * self.m * (self.R * self.n_shard) * self.k

    def make(self):
        X = to16(_draw(self.x_dist, (self.m, self.k), self.seed, 0), self.dtype)
        W = to16(_draw(self.w_dist, (self.k, self.R * self.n_shard), self.seed, 1), self.dtype)
        ms, ns = self.m_shard, self.n_shard
        xs = [X[r * ms:(r + 1) * ms].contiguous() for r in range(self.R)]
        ws = [W[:, r * ns:(r + 1) * ns].contiguous() for r in range(self.R)]
        return xs, ws


SCALE_GRANS = ("tensor", "channel", "group")


@dataclass
class W8A16:
    """w8A16 AllReduce shapes: X_r m x k_shard and scales in `dtype` (the pages'
    fp16, or bf16), int8 W_r k_shard x n, optional int8 zero points."""
    R: int
    m: int
    n: int
    k_shard: int
    group: int
    seed: int
    x_dist: str = "normal(0,1)"
    dtype: torch.dtype = torch.float16

    @property
    def K(self) -> int:
        return self.R * self.k_shard

    def flops(self) -> float:
        return 2.0 * self.m * self.n * self.K

    def make(self, gran: str):
        """Returns (xs, wqs, scales): scales[r] is rank r's view of the scale
        tensor — the shared scalar (1,), the shared per-column vector (n,), or
        rank r's rows of the (K/group) x n per-group table."""
        dt = self.dtype
        X = to16(_draw(self.x_dist, (self.m, self.K), self.seed, 0), dt)
        Wq = torch.from_numpy(int8_uniform((self.K, self.n), -127, 127, self.seed, 1))
        if gran == "tensor":
            S = to16(uniform((1,), 0.001, 0.01, self.seed, 2), dt)
        elif gran == "channel":
            S = to16(uniform((self.n,), 0.001, 0.01, self.seed, 3), dt)
        elif gran == "group":
            S = to16(uniform((self.K // self.group, self.n), 0.001, 0.01, self.seed, 4), dt)
        else:
            raise ValueError(gran)
        ks = self.k_shard
        xs = [X[:, r * ks:(r + 1) * ks].contiguous() for r in range(self.R)]
        wqs = [Wq[r * ks:(r + 1) * ks, :].contiguous() for r in range(self.R)]
        return xs, wqs, self._views(S, gran)

    def _views(self, T: torch.Tensor, gran: str):
        """Rank views of a scale-shaped tensor: the shared scalar or per-column
        vector, or rank r's rows of the per-group table."""
        if gran != "group":
            return [T] * self.R
        gpr = self.k_shard // self.group
        return [T[r * gpr:(r + 1) * gpr].contiguous() for r in range(self.R)]

    def zeros(self, gran: str, lo: int = -128, hi: int = 127):
        """Rank views of int8 zero points laid out like the scales of `gran`
        (asymmetric quantisation; seeded independently of the scales)."""
        shape = {"tensor": (1,), "channel": (self.n,), "group": (self.K // self.group, self.n)}[gran]
        Z = torch.from_numpy(int8_uniform(shape, lo, hi, self.seed, 5))
        return self._views(Z, gran)


@dataclass
class MoEDispatch:
    """Expert-parallel MoE layer input: R ranks with T tokens each (T x h),
    top-1 expert ids in [0, E) with E = R * e_loc (expert e on rank
    e // e_loc), and one h x f weight per expert.  Expert popularity is
    skewed (weights (e + 1)^-skew, shuffled) so groups have unequal sizes."""
    R: int
    T: int
    h: int
    f: int
    e_loc: int
    seed: int
    dtype: torch.dtype = torch.bfloat16
    skew: float = 0.5

    @property
    def E(self) -> int:
        return self.R * self.e_loc

    def flops(self) -> float:
        return 2.0 * self.R * self.T * self.h * self.f

    def routing(self):
        g = np.random.Generator(np.random.PCG64(self.seed * 7919 + 11))
        w = (np.arange(self.E) + 1.0) ** (-self.skew)
        w = w[g.permutation(self.E)]
        p = w / w.sum()
        return [torch.from_numpy(g.choice(self.E, size=self.T, p=p).astype(np.int32)) for _ in range(self.R)]

    def routing_topk(self, k: int):
        """k distinct experts per token (Gumbel top-k over the skewed
        popularity) and fp32 gates: positive, summing to 1 per token.
        Returns (idxs, gates), each a list of (T x k) tensors."""
        g = np.random.Generator(np.random.PCG64(self.seed * 7919 + 13))
        w = (np.arange(self.E) + 1.0) ** (-self.skew)
        logp = np.log(w[g.permutation(self.E)] / w.sum())
        idxs, gates = [], []
        for _ in range(self.R):
            keys = logp[None, :] + g.gumbel(size=(self.T, self.E))
            top = np.argsort(-keys, axis=1)[:, :k].astype(np.int32)
            raw = g.random((self.T, k)).astype(np.float32) + np.float32(0.1)
            idxs.append(torch.from_numpy(np.ascontiguousarray(top)))
            gates.append(torch.from_numpy(raw / raw.sum(axis=1, keepdims=True)))
        return idxs, gates

    def make(self):
        """Returns (xs, idxs, ws)."""
        xs = [to16(normal((self.T, self.h), 1.0, self.seed, 20 + r), self.dtype) for r in range(self.R)]
        ws = [to16(normal((self.h, self.f), 0.02, self.seed, 40 + e), self.dtype) for e in range(self.E)]
        return xs, self.routing(), ws


@dataclass
class Workload:
    name: str
    op: str            # "ar", "rs", "ag_v2", "w8a16_ar"
    shape: object
    chunks: int = 1
    deterministic: bool = False
    grans: tuple = field(default_factory=tuple)


# The pages' TP8 layers (BLOOM-7B / LLaMA2-70B / BLOOM-176B) and the small R=2 case.
TINY_AR = RowParallel(R=2, m=64, n=128, k_shard=128, dtype=torch.float16,
                      x_dist="uniform[-1,1]", w_dist="uniform[-1,1]", seed=0)
BLOOM7B_AR = RowParallel(R=8, m=2048, n=4096, k_shard=2048, dtype=torch.bfloat16,
                         x_dist="normal(0,1)", w_dist="normal(0,0.02)", seed=1)
LLAMA70B_AG = ColumnParallelSP(R=8, m_shard=512, n_shard=7168, k=8192, dtype=torch.bfloat16,
                               x_dist="normal(0,1)", w_dist="normal(0,0.02)", seed=2)
LLAMA70B_RS = RowParallel(R=8, m=4096, n=8192, k_shard=3584, dtype=torch.bfloat16,
                          x_dist="normal(0,1)", w_dist="normal(0,0.02)", seed=2)
W8A16_AR = W8A16(R=8, m=4096, n=8192, k_shard=1024, group=128, seed=3)
BLOOM176B = RowParallel(R=8, m=2048, n=14336, k_shard=7168, dtype=torch.bfloat16,
                        x_dist="normal(0,1)", w_dist="normal(0,0.02)", seed=4)

# One pass over every step of the hot path: each fused operator once on its
# TP8 layer shape.  Chunk counts as the layer configurations give them
# (BLOOM-7B: 4); 1 where they give none, and 1 for the BLOOM-176B layer whose
# configuration sweeps 1/2/4/8 as a bitwise-reproducibility check.
TP8_SUITE = [
    Workload("bloom7b_ar", "ar", BLOOM7B_AR, chunks=4),
    Workload("llama70b_ag_v2", "ag_v2", LLAMA70B_AG, chunks=1),
    Workload("llama70b_rs", "rs", LLAMA70B_RS, chunks=1),
    Workload("w8a16_ar", "w8a16_ar", W8A16_AR, chunks=1, grans=SCALE_GRANS),
    Workload("bloom176b_det_ar", "ar", BLOOM176B, chunks=1, deterministic=True),
    Workload("bloom176b_det_rs", "rs", BLOOM176B, chunks=1, deterministic=True),
]


def sample_rows(m: int, count: int = 256, seed: int = 1234) -> np.ndarray:
    """The seeded row sample at which full-size outputs are checked."""
    perm = np.random.Generator(np.random.PCG64(seed)).permutation(m)
    return np.sort(perm[:min(count, m)]).astype(np.int64)


def bits16(t: torch.Tensor) -> np.ndarray:
    """View a CPU fp16/bf16 tensor as its uint16 bit patterns (no copy)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
