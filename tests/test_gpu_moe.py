"""MoE expert-parallel dispatch + GroupedMatMul on the GPU against the oracle.

Checked: the expert group sizes and offsets exactly, the dispatched token
rows bit for bit, the expert outputs within the tolerance, repeat calls
bit-identical, and the edge cases (no tokens, every token on one expert,
experts without tokens, an out-of-range expert id reported)."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from tensor_matmul_collective_gb300 import coc
from tensor_matmul_collective_gb300 import workloads as wl

from gpu_util import assert_close, bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
CODE = {torch.float16: orc.F16, torch.bfloat16: orc.BF16}


def _run(s, xs, idxs, ws):
    w = torch.stack(ws).to(DEV)
    return coc.moe_dispatch_grouped_matmul([x.to(DEV) for x in xs], [i.to(DEV) for i in idxs], w, s.e_loc)


def _check(s, xs, idxs, ws, y, xd, counts, offsets, rows_per_group=None):
    coc.sync_status()
    res = orc.moe_dispatch_grouped_matmul(CODE[s.dtype], bits(xs), [i.numpy() for i in idxs], bits(ws))
    cnt, off = counts.cpu().numpy(), offsets.cpu().numpy()
    expect_off = np.zeros(s.E, np.int64)
    for e in range(s.E):
        expect_off[e] = 0 if e % s.e_loc == 0 else \
            expect_off[e - 1] + -(-res[e - 1][0].shape[0] // 256) * 256
    assert [g[0].shape[0] for g in res] == cnt.tolist()
    assert np.array_equal(off, expect_off)
    for e, (pairs, Xd, Y) in enumerate(res):
        q, n = e // s.e_loc, pairs.shape[0]
        if n == 0:
            continue
        got_xd = wl.bits16(xd[q][off[e]:off[e] + n].cpu())
        assert np.array_equal(got_xd, Xd), f"expert {e}: dispatched rows differ"
        sel = slice(None) if rows_per_group is None else np.linspace(0, n - 1, min(n, rows_per_group)).astype(int)
        assert_close(y[q][off[e]:off[e] + n][sel], Y[sel], s.h, f"expert {e} output")


CASES = [
    # R, T, h, f, e_loc, dtype
    (2, 100, 128, 136, 1, torch.bfloat16),
    (4, 300, 192, 264, 2, torch.float16),
    (8, 257, 64, 520, 3, torch.bfloat16),
    (1, 50, 128, 64, 4, torch.bfloat16),
]


@pytest.mark.parametrize("R,T,h,f,e_loc,dt", CASES)
def test_moe_parity(R, T, h, f, e_loc, dt):
    s = wl.MoEDispatch(R=R, T=T, h=h, f=f, e_loc=e_loc, seed=R + T, dtype=dt)
    xs, idxs, ws = s.make()
    y, xd, counts, offsets = _run(s, xs, idxs, ws)
    _check(s, xs, idxs, ws, y, xd, counts, offsets)


def test_moe_repeat_is_bitwise_identical():
    s = wl.MoEDispatch(R=4, T=500, h=128, f=256, e_loc=2, seed=7)
    xs, idxs, ws = s.make()
    a = _run(s, xs, idxs, ws)
    b = _run(s, xs, idxs, ws)
    coc.sync_status()
    for q in range(s.R):
        for e in range(s.E):
            if e // s.e_loc != q:
                continue
            o, n = int(a[3][e]), int(a[2][e])
            assert torch.equal(a[0][q][o:o + n], b[0][q][o:o + n])
    assert torch.equal(a[2], b[2]) and torch.equal(a[3], b[3])


def test_moe_one_expert_takes_everything_and_empty_experts():
    s = wl.MoEDispatch(R=4, T=333, h=128, f=128, e_loc=2, seed=8)
    xs, _, ws = s.make()
    idxs = [torch.full((s.T,), 5, dtype=torch.int32) for _ in range(s.R)]   # expert 5 (rank 2) only
    y, xd, counts, offsets = _run(s, xs, idxs, ws)
    _check(s, xs, idxs, ws, y, xd, counts, offsets)
    assert counts.cpu().tolist() == [0, 0, 0, 0, 0, s.R * s.T, 0, 0]


def test_moe_no_tokens():
    s = wl.MoEDispatch(R=2, T=0, h=64, f=64, e_loc=1, seed=1)
    xs = [torch.empty(0, 64, dtype=torch.bfloat16) for _ in range(2)]
    idxs = [torch.empty(0, dtype=torch.int32) for _ in range(2)]
    ws = [torch.zeros(64, 64, dtype=torch.bfloat16) for _ in range(2)]
    _, _, counts, offsets = _run(s, xs, idxs, ws)
    coc.sync_status()
    assert counts.cpu().tolist() == [0, 0] and offsets.cpu().tolist() == [0, 0]


def test_moe_out_of_range_expert_id_is_reported():
    """The routing kernel's own bounds check: ids outside [0, E) are not
    dispatched and the call reports COC_ERR_INVALID_ARG; the device stays
    usable and the next call is correct."""
    s = wl.MoEDispatch(R=2, T=64, h=64, f=64, e_loc=1, seed=2)
    xs, idxs, ws = s.make()
    bad = [i.clone() for i in idxs]
    bad[1][3] = 7
    _run(s, xs, bad, ws)
    with pytest.raises(coc.CocError) as ei:
        coc.sync_status()
    assert ei.value.status == coc.ERR_INVALID_ARG
    y, xd, counts, offsets = _run(s, xs, idxs, ws)
    _check(s, xs, idxs, ws, y, xd, counts, offsets)


def test_moe_layer_shape_sampled():
    """Mixtral-style layer on 8 EP ranks (one expert each), 4096 tokens per
    rank, h 4096, f 14336: counts, offsets and dispatched rows exactly;
    outputs on 24 rows of every expert against the oracle."""
    s = wl.MoEDispatch(R=8, T=4096, h=4096, f=14336, e_loc=1, seed=21)
    xs, idxs, ws = s.make()
    y, xd, counts, offsets = _run(s, xs, idxs, ws)
    coc.sync_status()
    groups = orc.moe_dispatch_order([i.numpy() for i in idxs], s.E)
    cnt, off = counts.cpu().numpy(), offsets.cpu().numpy()
    assert [g.shape[0] for g in groups] == cnt.tolist() and not off.any()
    xb = bits(xs)
    for e, pairs in enumerate(groups):
        n = pairs.shape[0]
        pick = np.linspace(0, n - 1, 24).astype(int)
        Xd = np.stack([xb[r][t] for r, t in pairs[pick]])
        assert np.array_equal(wl.bits16(xd[e][pick].cpu()), Xd)
        ref = orc.matmul_all_reduce(orc.BF16, [Xd], [wl.bits16(ws[e])])
        assert_close(y[e][pick], ref, s.h, f"expert {e}")


@pytest.mark.parametrize("R,T,h,f,e_loc,dt", CASES)
def test_moe_combine_parity(R, T, h, f, e_loc, dt):
    """The all-to-all back: y_tok[r][t] = x[r][t] @ W_{idx[r][t]} for every token."""
    s = wl.MoEDispatch(R=R, T=T, h=h, f=f, e_loc=e_loc, seed=R + 3 * T, dtype=dt)
    xs, idxs, ws = s.make()
    y, xd, counts, offsets = coc.moe_dispatch_grouped_matmul([x.to(DEV) for x in xs], [i.to(DEV) for i in idxs],
                                                             torch.stack(ws).to(DEV), s.e_loc, combine=True)
    coc.sync_status()
    ref = orc.moe_token_outputs(CODE[s.dtype], bits(xs), [i.numpy() for i in idxs], bits(ws))
    for r in range(R):
        assert y[r].shape == (T, f)
        assert_close(y[r], ref[r], s.h, f"combine rank {r}")


def test_moe_combine_matches_dispatched_layout_bits():
    """Combine and the dispatched layout hold the same bits, row for row."""
    s = wl.MoEDispatch(R=4, T=200, h=128, f=136, e_loc=2, seed=17)
    xs, idxs, ws = s.make()
    args = ([x.to(DEV) for x in xs], [i.to(DEV) for i in idxs], torch.stack(ws).to(DEV), s.e_loc)
    y, _, counts, offsets = coc.moe_dispatch_grouped_matmul(*args)
    yt, _, _, _ = coc.moe_dispatch_grouped_matmul(*args, combine=True)
    coc.sync_status()
    groups = orc.moe_dispatch_order([i.numpy() for i in idxs], s.E)
    off = offsets.cpu().tolist()
    for e, pairs in enumerate(groups):
        q = e // s.e_loc
        for i, (r, t) in enumerate(pairs):
            assert torch.equal(y[q][off[e] + i], yt[r][t])


def test_moe_combine_layer_shape_sampled():
    s = wl.MoEDispatch(R=8, T=4096, h=4096, f=14336, e_loc=1, seed=22)
    xs, idxs, ws = s.make()
    y, _, _, _ = coc.moe_dispatch_grouped_matmul([x.to(DEV) for x in xs], [i.to(DEV) for i in idxs],
                                                 torch.stack(ws).to(DEV), s.e_loc, combine=True)
    coc.sync_status()
    xb, wb = bits(xs), bits(ws)
    for r in range(s.R):
        pick = np.linspace(0, s.T - 1, 16).astype(int)
        ib = idxs[r].numpy()
        ref = np.concatenate([orc.matmul_all_reduce(orc.BF16, [xb[r][t:t + 1]], [wb[ib[t]]]) for t in pick])
        assert_close(y[r][pick], ref, s.h, f"combine rank {r}")


@pytest.mark.parametrize("R,T,h,f,e_loc,k,dt", [
    (2, 100, 128, 136, 2, 2, torch.bfloat16),
    (4, 257, 192, 264, 2, 2, torch.float16),
    (8, 64, 64, 128, 1, 4, torch.bfloat16),
    (1, 40, 128, 64, 4, 3, torch.bfloat16),
])
def test_moe_topk_parity(R, T, h, f, e_loc, k, dt):
    """Top-k: every (token, slot) entry dispatched (counts, offsets and rows
    exact), the gated combine against the oracle."""
    s = wl.MoEDispatch(R=R, T=T, h=h, f=f, e_loc=e_loc, seed=5 * R + T, dtype=dt)
    xs, _, ws = s.make()
    idxs, gates = s.routing_topk(k)
    y_tok, y, xd, counts, offsets = coc.moe_topk_grouped_matmul_combine(
        [x.to(DEV) for x in xs], [i.to(DEV) for i in idxs], [g.to(DEV) for g in gates], torch.stack(ws).to(DEV), e_loc)
    coc.sync_status()
    flat = [i.numpy().reshape(-1) for i in idxs]
    groups = orc.moe_dispatch_order(flat, s.E)
    cnt, off = counts.cpu().numpy(), offsets.cpu().numpy()
    assert [g_.shape[0] for g_ in groups] == cnt.tolist()
    xb = bits(xs)
    for e, pairs in enumerate(groups):
        q, n = e // e_loc, pairs.shape[0]
        if n:
            want = np.stack([xb[r][ent // k] for r, ent in pairs])
            assert np.array_equal(wl.bits16(xd[q][off[e]:off[e] + n].cpu()), want)
    ref = orc.moe_topk_combine(CODE[dt], xb, [i.numpy() for i in idxs], [g.numpy() for g in gates], bits(ws))
    for r in range(R):
        assert_close(y_tok[r], ref[r], s.h, f"top-{k} combine rank {r}")


@pytest.mark.parametrize("R,T,e_loc,f", [(8, 300, 8, 72), (8, 50, 32, 200)])
def test_moe_many_experts(R, T, e_loc, f):
    """64 and 256 experts (the maximum): most groups small or empty, f not a
    multiple of the tile width; dispatch exact, dispatched outputs and the
    combine against the oracle."""
    s = wl.MoEDispatch(R=R, T=T, h=64, f=f, e_loc=e_loc, seed=T + e_loc)
    xs, idxs, ws = s.make()
    y, xd, counts, offsets = _run(s, xs, idxs, ws)
    _check(s, xs, idxs, ws, y, xd, counts, offsets)
    yt, _, _, _ = coc.moe_dispatch_grouped_matmul([x.to(DEV) for x in xs], [i.to(DEV) for i in idxs],
                                                  torch.stack(ws).to(DEV), s.e_loc, combine=True)
    coc.sync_status()
    ref = orc.moe_token_outputs(CODE[s.dtype], bits(xs), [i.numpy() for i in idxs], bits(ws))
    for r in range(R):
        assert_close(yt[r], ref[r], s.h, f"combine rank {r}")
