"""Out-of-bounds write checks (the stand-in for a memory sanitizer).

Every fused operator writes R rank buffers, and several of its store paths
compute their addresses by hand instead of going through a bounds-clipped TMA
store: the AllReduce replica stores, the rank-split slab stores, the
column-slab kernel's stores (AllReduce, ReduceScatter and AllGather), the
ALL_GATHER_MATMUL_V2 gather copies (persistent and column-slab kernels), the
MoE token permute and combine scatter, and the w8A16 and allocation-free
AllReduce paths.  A store that runs past a
buffer would land in the next rank's buffer, which only an element-wise
check of that row would notice.

Here all the output buffers of one call are views inside ONE device slab,
separated (and preceded and followed) by guard regions filled with a canary
bit pattern that no finite result can take (0x7FC1: a quiet NaN both as fp16
and as bf16).  After the call every guard region must still hold the canary,
every element the operator defines must have been written (no canary left
inside a buffer), and the values must match the fp64 oracle.  Shapes are
ragged (rows, columns and k not multiples of the tiles) and cover both kernel
variants (single-CTA tiles up to 128 rows, 2-SM pairs above) and the rank
split at decode-sized m.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from tensor_matmul_collective_gb300 import coc
from tensor_matmul_collective_gb300 import workloads as wl

from gpu_util import DEV, assert_close, bits, to_dev

pytestmark = pytest.mark.gpu

F16, BF16 = torch.float16, torch.bfloat16
CODE = {F16: orc.F16, BF16: orc.BF16}
CANARY = 0x7FC1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_matmul_collective_gb300 import build
    build.build()
    coc.lib()
    yield
    coc.sync_status()


class Slab:
    """Buffers carved out of one canary-filled int16 slab with a guard region
    of at least `guard` elements (and at least 256 rows of the widest buffer)
    before, between and after them.  Offsets are multiples of 64 elements so
    every view keeps the 16-byte alignment the library requires."""

    def __init__(self, shapes, dtypes, guard=8192):
        widest = max(int(s[-1]) if len(s) > 1 else 1 for s in shapes)
        self.guard = -(-max(guard, 256 * widest) // 64) * 64
        self.spans, off = [], self.guard
        for s in shapes:
            n = int(np.prod(s))
            self.spans.append((off, n))
            off += -(-n // 64) * 64 + self.guard
        self.slab = torch.full((off,), CANARY, dtype=torch.int16, device=DEV)
        self.views = [self.slab[o:o + n].view(dt).view(s) if n else
                      torch.empty(s, dtype=dt, device=DEV)
                      for (o, n), s, dt in zip(self.spans, shapes, dtypes)]

    def check_guards(self, what):
        torch.cuda.synchronize()
        host = self.slab.cpu().numpy().view(np.uint16)
        edges = [0] + [e for o, n in self.spans for e in (o, o + n)] + [host.size]
        for i in range(0, len(edges), 2):
            lo, hi = edges[i], edges[i + 1]
            bad = np.nonzero(host[lo:hi] != CANARY)[0]
            assert bad.size == 0, (f"{what}: {bad.size} guard elements overwritten between buffers "
                                   f"{i // 2 - 1} and {i // 2} (first at slab offset {lo + bad[0]})")

    @staticmethod
    def assert_written(t, what):
        raw = t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        left = np.count_nonzero(raw == CANARY)
        assert left == 0, f"{what}: {left} elements never written"


def _rp(R, m, n, ks, dt, seed):
    return wl.RowParallel(R=R, m=m, n=n, k_shard=ks, dtype=dt, x_dist="uniform[-1,1]",
                          w_dist="uniform[-1,1]", seed=seed).make()


# AllReduce: replica stores (single-CTA and 2-SM tiles) and the rank split
# (m <= 128 with few tiles: 8 parts for one 40 x 264 tile column).
AR_CASES = [
    # R, m, n, k_shard, dtype, chunks
    (8, 40, 264, 128, BF16, 1),      # rank split, ragged n
    (4, 100, 72, 200, F16, 2),       # rank split, one partial tile
    (8, 200, 136, 72, BF16, 1),      # 2-SM pair, ragged m/n/k
    (2, 520, 1000, 64, F16, 4),      # several pair tiles, ragged tail in both dimensions
    (1, 130, 264, 64, BF16, 1),      # R = 1
    # n a multiple of 16 (the cases above end 8 columns into a 16-column group)
    (8, 200, 144, 72, BF16, 1),      # one partial pair tile, 144 = two sub-tiles + 16 columns
    (2, 520, 1008, 64, F16, 4),      # the last sub-tile 48 columns wide
    (4, 300, 4096, 64, BF16, 2),     # whole tiles in n, ragged m
]


@pytest.mark.parametrize("R,m,n,ks,dt,chunks", AR_CASES)
def test_allreduce_guards(R, m, n, ks, dt, chunks):
    xs, ws = _rp(R, m, n, ks, dt, seed=500 + m)
    slab = Slab([(m, n)] * R, [dt] * R)
    coc.matmul_all_reduce(to_dev(xs), to_dev(ws), slab.views, chunks=chunks)
    coc.sync_status()
    slab.check_guards("AllReduce")
    ref = orc.matmul_all_reduce(CODE[dt], bits(xs), bits(ws))
    for r, o in enumerate(slab.views):
        Slab.assert_written(o, f"AllReduce rank {r}")
        assert_close(o, ref, R * ks, f"AllReduce rank {r}")


# The column-slab kernel (decode-sized m): plain 16-byte stores of every
# slab's rows to every rank output (AllReduce) or to the owning rank
# (ReduceScatter), slabs split over clusters of 2 and 4, ragged last slab.
SLAB_CASES = [
    # op, R, m, n, k_shard, dtype, (boxes, split, kps)
    ("ar", 8, 40, 1000, 200, BF16, (2, 2, 1)),    # k_shard ends inside a k-block
    ("ar", 4, 17, 520, 128, F16, (2, 4, 2)),      # clusters of 4, 3-D X boxes
    ("ar", 2, 100, 264, 64, BF16, (1, 1, 1)),     # 64-column slabs, unsplit
    ("ar", 4, 120, 1000, 128, BF16, (2, 2, 1)),   # four row quadrants pushed between two parts
    ("rs", 8, 64, 1000, 72, BF16, (2, 2, 1)),     # 8 rows per rank
    ("rs", 4, 32, 520, 128, F16, (1, 2, 2)),      # 64-column slabs split in two
]


@pytest.mark.parametrize("op,R,m,n,ks,dt,plan", SLAB_CASES)
def test_column_slab_guards(op, R, m, n, ks, dt, plan, monkeypatch):
    b, sp, kps = plan
    for k, v in (("COC_SLAB", 1), ("COC_SLAB_BOXES", b), ("COC_SLAB_SPLIT", sp), ("COC_SLAB_KPS", kps)):
        monkeypatch.setenv(k, str(v))
    xs, ws = _rp(R, m, n, ks, dt, seed=550 + m)
    rows = m if op == "ar" else m // R
    slab = Slab([(rows, n)] * R, [dt] * R)
    if op == "ar":
        coc.matmul_all_reduce(to_dev(xs), to_dev(ws), slab.views)
    else:
        coc.matmul_reduce_scatter(to_dev(xs), to_dev(ws), slab.views)
    coc.sync_status()
    slab.check_guards(f"column slab {op}")
    ref = orc.matmul_all_reduce(CODE[dt], bits(xs), bits(ws))
    for r, o in enumerate(slab.views):
        Slab.assert_written(o, f"column slab {op} rank {r}")
        assert_close(o, ref if op == "ar" else ref[r * rows:(r + 1) * rows], R * ks, f"column slab {op} rank {r}")


def test_allreduce_noalloc_guards():
    R, m, n, ks, dt = 4, 200, 264, 72, BF16
    xs, ws = _rp(R, m, n, ks, dt, seed=517)
    slab = Slab([(m, n)] * R, [dt] * R)
    coc.matmul_all_reduce_noalloc(to_dev(xs), to_dev(ws), slab.views, chunks=2)
    coc.sync_status()
    slab.check_guards("no-alloc AllReduce")
    ref = orc.matmul_all_reduce(CODE[dt], bits(xs), bits(ws))
    for r, o in enumerate(slab.views):
        Slab.assert_written(o, f"no-alloc rank {r}")
        assert_close(o, ref, R * ks, f"no-alloc rank {r}")


def test_plain_matmul_guards():
    R, m, n, ks, dt = 2, 300, 200, 136, F16
    xs, ws = _rp(R, m, n, ks, dt, seed=518)
    slab = Slab([(m, n)], [dt])
    coc.matmul(to_dev(xs), to_dev(ws), slab.views[0])
    coc.sync_status()
    slab.check_guards("plain matmul")
    Slab.assert_written(slab.views[0], "plain matmul")
    assert_close(slab.views[0], orc.matmul_all_reduce(CODE[dt], bits(xs), bits(ws)), R * ks, "plain matmul")


# ReduceScatter: per-rank row blocks of 8..32 rows, the rank split at small m.
RS_CASES = [
    (8, 64, 264, 128, BF16, 1),      # 8 rows per rank, rank split
    (4, 96, 520, 72, F16, 2),        # 24 rows per rank (8-row store boxes)
    (8, 1024, 200, 64, BF16, 4),     # pair tiles straddling rank blocks
]


@pytest.mark.parametrize("R,m,n,ks,dt,chunks", RS_CASES)
def test_reduce_scatter_guards(R, m, n, ks, dt, chunks):
    xs, ws = _rp(R, m, n, ks, dt, seed=600 + m)
    slab = Slab([(m // R, n)] * R, [dt] * R)
    coc.matmul_reduce_scatter(to_dev(xs), to_dev(ws), slab.views, chunks=chunks)
    coc.sync_status()
    slab.check_guards("ReduceScatter")
    for r, o in enumerate(slab.views):
        Slab.assert_written(o, f"ReduceScatter rank {r}")
        assert_close(o, orc.matmul_reduce_scatter(CODE[dt], bits(xs), bits(ws), r), R * ks, f"RS rank {r}")


# ALL_GATHER_MATMUL_V2: the products (TMA stores) and the gather copy (plain
# stores spread over all work units), shards that split a tile.
AG_CASES = [
    # R, m_shard, n_shard, k, dtype, chunks
    (8, 24, 136, 72, BF16, 1),
    (4, 40, 264, 200, F16, 2),
    (2, 200, 72, 64, BF16, 4),
]


@pytest.mark.parametrize("R,ms,ns,k,dt,chunks", AG_CASES)
def test_all_gather_v2_guards(R, ms, ns, k, dt, chunks):
    s = wl.ColumnParallelSP(R=R, m_shard=ms, n_shard=ns, k=k, dtype=dt, x_dist="uniform[-1,1]",
                            w_dist="uniform[-1,1]", seed=700 + ms)
    xs, ws = s.make()
    m = R * ms
    slab = Slab([(m, ns)] * R + [(m, k)] * R, [dt] * (2 * R))
    outs, gathered = slab.views[:R], slab.views[R:]
    coc.all_gather_matmul_v2(to_dev(xs), to_dev(ws), outs, gathered, chunks=chunks)
    coc.sync_status()
    slab.check_guards("AllGather-V2")
    bx, bw = bits(xs), bits(ws)
    xg = orc.all_gather(bx)
    for r in range(R):
        Slab.assert_written(outs[r], f"AG-V2 product rank {r}")
        assert np.array_equal(wl.bits16(gathered[r].cpu()), xg), f"gather copy rank {r}"
        assert_close(outs[r], orc.all_gather_matmul(CODE[dt], bx, bw, r), k, f"AG-V2 rank {r}")


# The column-slab kernel's AllGather (gathered m <= 128): plain 16-byte stores
# of each slab to its rank's output, the gathered copies from the epilogue
# warps, ragged last slab and k, clusters of 2 and 4.
AG_SLAB_CASES = [
    # R, m_shard, n_shard, k, dtype, (boxes, split, kps)
    (8, 8, 1000, 200, BF16, (2, 2, 1)),
    (4, 24, 520, 128, F16, (1, 2, 2)),
    (2, 64, 1104, 512, BF16, (2, 4, 1)),
    (8, 16, 136, 72, F16, (2, 1, 1)),
]


@pytest.mark.parametrize("R,ms,ns,k,dt,plan", AG_SLAB_CASES)
def test_all_gather_v2_column_slab_guards(R, ms, ns, k, dt, plan, monkeypatch):
    b, sp, kps = plan
    for key, v in (("COC_SLAB", 1), ("COC_SLAB_BOXES", b), ("COC_SLAB_SPLIT", sp), ("COC_SLAB_KPS", kps)):
        monkeypatch.setenv(key, str(v))
    s = wl.ColumnParallelSP(R=R, m_shard=ms, n_shard=ns, k=k, dtype=dt, x_dist="uniform[-1,1]",
                            w_dist="uniform[-1,1]", seed=760 + ms)
    xs, ws = s.make()
    m = R * ms
    slab = Slab([(m, ns)] * R + [(m, k)] * R, [dt] * (2 * R))
    outs, gathered = slab.views[:R], slab.views[R:]
    g = [t if r % 3 != 1 else None for r, t in enumerate(gathered)]   # some copies skipped
    coc.all_gather_matmul_v2(to_dev(xs), to_dev(ws), outs, g)
    coc.sync_status()
    slab.check_guards("AllGather-V2 column slab")
    bx, bw = bits(xs), bits(ws)
    xg = orc.all_gather(bx)
    for r in range(R):
        Slab.assert_written(outs[r], f"AG-V2 column slab product rank {r}")
        assert_close(outs[r], orc.all_gather_matmul(CODE[dt], bx, bw, r), k, f"AG-V2 column slab rank {r}")
        raw = gathered[r].view(torch.int16).cpu().numpy().view(np.uint16)
        if g[r] is None:
            assert np.all(raw == CANARY), f"skipped gather buffer {r} was written"
        else:
            assert np.array_equal(raw, xg), f"gather copy rank {r}"


def test_all_gather_v2_skipped_copies_leave_buffers_alone():
    """NULL gather entries: the library must not write those buffers."""
    R, ms, ns, k, dt = 4, 40, 136, 72, BF16
    s = wl.ColumnParallelSP(R=R, m_shard=ms, n_shard=ns, k=k, dtype=dt, x_dist="uniform[-1,1]",
                            w_dist="uniform[-1,1]", seed=731)
    xs, ws = s.make()
    m = R * ms
    slab = Slab([(m, ns)] * R + [(m, k)] * R, [dt] * (2 * R))
    outs, gathered = slab.views[:R], slab.views[R:]
    coc.all_gather_matmul_v2(to_dev(xs), to_dev(ws), outs, [gathered[0], None, gathered[2], None])
    coc.sync_status()
    slab.check_guards("AllGather-V2 with skipped copies")
    xg = orc.all_gather(bits(xs))
    for r in (0, 2):
        assert np.array_equal(wl.bits16(gathered[r].cpu()), xg)
    for r in (1, 3):
        raw = gathered[r].view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.all(raw == CANARY), f"skipped gather buffer {r} was written"


@pytest.mark.parametrize("gran,path", [("channel", "fused"), ("group", "fused"), ("tensor", "prepass"),
                                       ("channel", "ts"), ("group", "ts")])
def test_w8a16_guards(gran, path, monkeypatch):
    monkeypatch.setenv("COC_W8_PATH", path)
    R, m, n, ks, group = 4, 200, 272, 128, 64
    s = wl.W8A16(R=R, m=m, n=n, k_shard=ks, group=group, seed=801)
    xs, wqs, scales = s.make(gran)
    slab = Slab([(m, n)] * R, [F16] * R)
    coc.matmul_all_reduce_w8a16(to_dev(xs), to_dev(wqs), to_dev(scales), gran, group, slab.views)
    coc.sync_status()
    slab.check_guards(f"w8A16 {gran} {path}")
    code = {"tensor": 0, "channel": 1, "group": 2}[gran]
    ref = orc.matmul_all_reduce_w8a16(bits(xs), [w.numpy() for w in wqs], bits(scales), code, group)
    for r, o in enumerate(slab.views):
        Slab.assert_written(o, f"w8A16 rank {r}")
        assert_close(o, ref, s.K, f"w8A16 rank {r}")


def test_moe_dispatch_and_combine_guards():
    """Token permute (xd), dispatched expert outputs (y) and the fused top-1
    combine scatter into the source ranks' token rows (y_tok)."""
    s = wl.MoEDispatch(R=4, T=150, h=128, f=200, e_loc=2, seed=901, dtype=BF16)
    xs, idxs, ws = s.make()
    R, E = s.R, s.E
    cap = coc.moe_capacity(R, s.T, s.e_loc)
    w = torch.stack(ws).to(DEV)
    dx, di = to_dev(xs), to_dev(idxs)
    slab = Slab([(cap, s.h)] * R + [(s.T, s.f)] * R, [BF16] * (2 * R))
    xd, y_tok = slab.views[:R], slab.views[R:]
    coc.moe_dispatch_grouped_matmul(dx, di, w, s.e_loc, xd=xd, y=y_tok, combine=True)
    coc.sync_status()
    slab.check_guards("MoE dispatch + combine")
    ref = orc.moe_token_outputs(orc.BF16, bits(xs), [i.numpy() for i in idxs], bits(ws))
    for r in range(R):
        Slab.assert_written(y_tok[r], f"MoE combine rank {r}")
        assert_close(y_tok[r], ref[r], s.h, f"MoE combine rank {r}")
    # the dispatched layout with y in the slab as well
    slab2 = Slab([(cap, s.h)] * R + [(cap, s.f)] * R, [BF16] * (2 * R))
    y, xd2, counts, offsets = coc.moe_dispatch_grouped_matmul(dx, di, w, s.e_loc, xd=slab2.views[:R],
                                                              y=slab2.views[R:])
    coc.sync_status()
    slab2.check_guards("MoE dispatch")
    res = orc.moe_dispatch_grouped_matmul(orc.BF16, bits(xs), [i.numpy() for i in idxs], bits(ws))
    cnt, off = counts.cpu().tolist(), offsets.cpu().tolist()
    for e, (pairs, Xd, Y) in enumerate(res):
        q, n_e = e // s.e_loc, pairs.shape[0]
        assert cnt[e] == n_e
        if n_e:
            assert np.array_equal(wl.bits16(xd2[q][off[e]:off[e] + n_e].cpu()), Xd)
            assert_close(y[q][off[e]:off[e] + n_e], Y, s.h, f"MoE expert {e}")


def test_moe_topk_combine_guards():
    s = wl.MoEDispatch(R=2, T=130, h=64, f=136, e_loc=3, seed=902, dtype=F16)
    xs, _, ws = s.make()
    ti, tg = s.routing_topk(2)
    R = s.R
    cap = coc.moe_capacity(R, s.T * 2, s.e_loc)
    slab = Slab([(cap, s.h)] * R + [(cap, s.f)] * R + [(s.T, s.f)] * R, [F16] * (3 * R))
    xd, y, y_tok = slab.views[:R], slab.views[R:2 * R], slab.views[2 * R:]
    coc.moe_topk_grouped_matmul_combine(to_dev(xs), to_dev(ti), to_dev(tg), torch.stack(ws).to(DEV), s.e_loc,
                                        xd=xd, y=y, y_tok=y_tok)
    coc.sync_status()
    slab.check_guards("MoE top-k combine")
    ref = orc.moe_topk_combine(orc.F16, bits(xs), [i.numpy() for i in ti], [g.numpy() for g in tg], bits(ws))
    for r in range(R):
        Slab.assert_written(y_tok[r], f"top-k combine rank {r}")
        assert_close(y_tok[r], ref[r], s.h, f"top-k combine rank {r}")


def test_weight_grad_and_nk_guards():
    """The Megatron n x k weight path (K-major B) and the weight-gradient pass
    (MN-major A), both TMA-stored, at ragged shapes."""
    R, m, n, ks, dt = 4, 136, 200, 72, BF16
    xs, ws = _rp(R, m, n, ks, dt, seed=950)
    wnk = [w.t().contiguous() for w in ws]
    slab = Slab([(m, n)] * R, [dt] * R)
    coc.fused_matmul("all_reduce", to_dev(xs), to_dev(wnk), w_layout="nk", outs=slab.views)
    coc.sync_status()
    slab.check_guards("AllReduce, n x k weights")
    ref = orc.matmul_all_reduce(CODE[dt], bits(xs), bits(ws))
    for r, o in enumerate(slab.views):
        Slab.assert_written(o, f"nk rank {r}")
        assert_close(o, ref, R * ks, f"nk rank {r}")
    # weight gradient: dW_r = dY_r^T X_r with dY_r tokens x rows, X_r tokens x cols
    T, rows, cols = 72, 136, 200
    dys = [wl.to16(wl.uniform((T, rows), -1.0, 1.0, 952, r), dt) for r in range(R)]
    xin = [wl.to16(wl.uniform((T, cols), -1.0, 1.0, 953, r), dt) for r in range(R)]
    slab2 = Slab([(rows, cols)] * R, [dt] * R)
    coc.weight_grad(to_dev(dys), to_dev(xin), slab2.views)
    coc.sync_status()
    slab2.check_guards("weight gradient")
    for r in range(R):
        Slab.assert_written(slab2.views[r], f"wgrad rank {r}")
        ref = orc.matmul_all_reduce(CODE[dt], [np.ascontiguousarray(wl.bits16(dys[r]).T)], [wl.bits16(xin[r])])
        assert_close(slab2.views[r], ref, T, f"wgrad rank {r}")
