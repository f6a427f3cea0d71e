"""Pins for the fp64 CPU oracle, independent of the oracle itself.

Each check compares the oracle with something it does not share code with:
exhaustive format tables from numpy / torch, exact rational arithmetic on tiny
inputs, numpy.matmul in float64 on the unsharded problem, closed forms, and
explicit index bookkeeping for the gather.  The "mutant" tests plant a
plausible mistake in a copy of an oracle result (a dropped rank, a shifted row
block, a transposed operand, a wrong scale index) and show the same check
rejects it, so the pins have teeth.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from tensor_matmul_collective_gb300 import workloads as wl

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand16(shape, dtype, seed, lo=-1.0, hi=1.0):
    a = wl.uniform(shape, lo, hi, seed, 99)
    return wl.bits16(wl.to16(a, dtype))


def _dec(bits, dt):
    if dt == torch.float16:
        return bits.view(np.float16).astype(np.float64)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


# ------------------------------------------------------------- formats ---

def test_f16_decode_exhaustive(oracle_mod):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.decode16(allbits, oracle_mod.F16)
    ref = allbits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_bf16_decode_exhaustive(oracle_mod):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.decode16(allbits, oracle_mod.BF16)
    ref = torch.from_numpy(allbits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_f16_encode_roundtrip_all_finite(oracle_mod):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = allbits.view(np.float16).astype(np.float64)
    fin = np.isfinite(vals)
    assert np.array_equal(oracle_mod.encode_f16(vals[fin]), allbits[fin])


def test_f16_encode_ties_and_random_vs_numpy(oracle_mod):
    # numpy's double -> binary16 cast rounds to nearest, ties to even.
    rng = np.random.default_rng(5)
    allbits = np.arange(0, 0x7c00, dtype=np.uint32).astype(np.uint16)  # non-negative finite
    v = allbits.view(np.float16).astype(np.float64)
    mids = (v[:-1] + v[1:]) / 2            # exact ties between neighbours
    near = np.concatenate([np.nextafter(mids, 0), np.nextafter(mids, np.inf)])
    rand = np.ldexp(rng.random(200000) + 0.5, rng.integers(-30, 18, 200000))
    edge = np.array([65504.0, 65519.999, 65520.0, 65536.0, 1e6, 2.0 ** -25, 2.0 ** -24 * 1.5,
                     2.0 ** -25 * 1.0000001, 2.0 ** -14 - 2.0 ** -25, 0.0])
    x = np.concatenate([mids, near, rand, edge])
    x = np.concatenate([x, -x])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle_mod.encode_f16(x), ref)


# ----------------------------------------------------- exact brute force ---

def _exact_ar(xs_bits, ws_bits, dt):
    """sum_r X_r W_r with every product and sum in exact rationals."""
    xs = [[[Fraction(float(v)) for v in row] for row in _dec(x, dt)] for x in xs_bits]
    ws = [[[Fraction(float(v)) for v in row] for row in _dec(w, dt)] for w in ws_bits]
    m, n = len(xs[0]), len(ws[0][0])
    Y = [[Fraction(0)] * n for _ in range(m)]
    absum = [[Fraction(0)] * n for _ in range(m)]
    for x, w in zip(xs, ws):
        for i in range(m):
            for t in range(len(w)):
                for j in range(n):
                    p = x[i][t] * w[t][j]
                    Y[i][j] += p
                    absum[i][j] += abs(p)
    return Y, absum


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
def test_ar_matches_exact_rational(oracle_mod, dt):
    R, m, ks, n = 3, 5, 16, 7
    xs = [_rand16((m, ks), dt, 10 + r) for r in range(R)]
    ws = [_rand16((ks, n), dt, 20 + r) for r in range(R)]
    code = oracle_mod.F16 if dt == torch.float16 else oracle_mod.BF16
    got = oracle_mod.matmul_all_reduce(code, xs, ws)
    Y, absum = _exact_ar(xs, ws, dt)
    K = R * ks
    for i in range(m):
        for j in range(n):
            bound = Fraction(K + 1, 2 ** 53) * absum[i][j]
            assert abs(Fraction(float(got[i, j])) - Y[i][j]) <= bound

    # a dropped rank (plausible indexing slip) is far outside that bound
    mutant = oracle_mod.matmul_all_reduce(code, xs[:-1], ws[:-1])
    assert max(abs(Fraction(float(mutant[i, j])) - Y[i][j]) - Fraction(K + 1, 2 ** 53) * absum[i][j]
               for i in range(m) for j in range(n)) > 0


def test_small_integers_are_exact(oracle_mod):
    # |x|, |w| <= 4 and K <= 1024: every partial sum is an integer below 2^24.
    rng = np.random.default_rng(3)
    R, m, ks, n = 4, 9, 64, 11
    xi = [rng.integers(-4, 5, (m, ks)) for _ in range(R)]
    wi = [rng.integers(-4, 5, (ks, n)) for _ in range(R)]
    xs = [wl.bits16(torch.tensor(a, dtype=torch.bfloat16)) for a in xi]
    ws = [wl.bits16(torch.tensor(a, dtype=torch.bfloat16)) for a in wi]
    got = oracle_mod.matmul_all_reduce(oracle_mod.BF16, xs, ws)
    exact = sum(np.asarray(a, dtype=object).dot(np.asarray(b, dtype=object)) for a, b in zip(xi, wi))
    assert np.array_equal(got, exact.astype(np.float64))


# ------------------------------------------------------------ closed forms ---

def test_closed_form_constant_shards(oracle_mod):
    # X_r all ones, W_r all c_r  =>  Y = k_shard * sum_r c_r everywhere.
    R, m, ks, n = 4, 6, 40, 5
    cs = [0.5, -1.25, 2.0, 0.125]
    xs = [wl.bits16(torch.ones(m, ks, dtype=torch.bfloat16)) for _ in range(R)]
    ws = [wl.bits16(torch.full((ks, n), c, dtype=torch.bfloat16)) for c in cs]
    got = oracle_mod.matmul_all_reduce(oracle_mod.BF16, xs, ws)
    assert np.array_equal(got, np.full((m, n), ks * sum(cs)))


def test_closed_form_identity(oracle_mod):
    # R = 1, X = I  =>  Y = W exactly.
    k = n = 24
    W = _rand16((k, n), torch.float16, 7)
    X = wl.bits16(torch.eye(k, dtype=torch.float16))
    got = oracle_mod.matmul_all_reduce(oracle_mod.F16, [X], [W])
    assert np.array_equal(got, _dec(W, torch.float16))


# ------------------------------------------- library-routine special cases ---

def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def test_r1_is_plain_gemm(oracle_mod):
    X = _rand16((37, 45), torch.bfloat16, 1)
    W = _rand16((45, 29), torch.bfloat16, 2)
    got = oracle_mod.matmul_all_reduce(oracle_mod.BF16, [X], [W])
    ref = _dec(X, torch.bfloat16) @ _dec(W, torch.bfloat16)
    assert _rel(got, ref) < 1e-13
    # transposed-operand mutant: X @ W with W read as column-major
    Wt = np.ascontiguousarray(W.reshape(29, 45).T)
    assert _rel(oracle_mod.matmul_all_reduce(oracle_mod.BF16, [X], [Wt]), ref) > 1e-2


def _unsharded(xs, ws, dt):
    X = np.concatenate([_dec(x, dt) for x in xs], axis=1)
    W = np.concatenate([_dec(w, dt) for w in ws], axis=0)
    return X @ W


@pytest.mark.parametrize("R", [1, 2, 4, 8])
def test_sharded_ar_equals_unsharded_gemm(oracle_mod, R):
    m, ks, n = 33, 24, 40
    xs = [_rand16((m, ks), torch.bfloat16, 30 + r) for r in range(R)]
    ws = [_rand16((ks, n), torch.bfloat16, 40 + r) for r in range(R)]
    got = oracle_mod.matmul_all_reduce(oracle_mod.BF16, xs, ws)
    assert _rel(got, _unsharded(xs, ws, torch.bfloat16)) < 1e-13
    rows = np.array([0, 5, 32], dtype=np.int64)
    assert np.array_equal(oracle_mod.matmul_all_reduce(oracle_mod.BF16, xs, ws, rows), got[rows])


@pytest.mark.parametrize("R", [2, 4, 8])
def test_reduce_scatter_blocks_concat_to_allreduce(oracle_mod, R):
    m, ks, n = 8 * R, 16, 24
    xs = [_rand16((m, ks), torch.float16, 50 + r) for r in range(R)]
    ws = [_rand16((ks, n), torch.float16, 60 + r) for r in range(R)]
    ref = _unsharded(xs, ws, torch.float16)
    outs = [oracle_mod.matmul_reduce_scatter(oracle_mod.F16, xs, ws, r) for r in range(R)]
    assert all(o.shape == (m // R, n) for o in outs)
    assert _rel(np.concatenate(outs, axis=0), ref) < 1e-13
    # row-block mix-up mutant: hand rank r the block of rank r+1
    shifted = np.concatenate(outs[1:] + outs[:1], axis=0)
    assert _rel(shifted, ref) > 1e-2
    with pytest.raises(ValueError):   # m not divisible by R
        oracle_mod.matmul_reduce_scatter(oracle_mod.F16, [x[:m - 1] for x in xs], ws, 0)


@pytest.mark.parametrize("R", [1, 2, 8])
def test_all_gather_matmul_equals_gemm_of_concat(oracle_mod, R):
    ms, k, ns = 9, 32, 12
    xs = [_rand16((ms, k), torch.bfloat16, 70 + r) for r in range(R)]
    ws = [_rand16((k, ns), torch.bfloat16, 80 + r) for r in range(R)]
    Xg = np.concatenate([_dec(x, torch.bfloat16) for x in xs], axis=0)
    outs = []
    for r in range(R):
        out, gathered = oracle_mod.all_gather_matmul_v2(oracle_mod.BF16, xs, ws, r)
        assert _rel(out, Xg @ _dec(ws[r], torch.bfloat16)) < 1e-13
        # the intermediate is a bit copy: check it element by element
        for q in range(R):
            for i in range(ms):
                assert np.array_equal(gathered[q * ms + i], xs[q][i])
        outs.append(out)
    Wcat = np.concatenate([_dec(w, torch.bfloat16) for w in ws], axis=1)
    assert _rel(np.concatenate(outs, axis=1), Xg @ Wcat) < 1e-13
    if R > 1:   # gathering in reverse rank order must be caught
        Xrev = np.concatenate([_dec(x, torch.bfloat16) for x in xs[::-1]], axis=0)
        assert _rel(outs[0], Xrev @ _dec(ws[0], torch.bfloat16)) > 1e-2


# --------------------------------------------------------------- w8A16 ---

def _numpy_dequant(wq, S, gran, group):
    q = wq.astype(np.float64)
    s = S.view(np.float16).astype(np.float64)
    if gran == "tensor":
        full = np.broadcast_to(s.reshape(1, 1), q.shape)
    elif gran == "channel":
        full = np.broadcast_to(s.reshape(1, -1), q.shape)
    else:
        full = np.repeat(s, group, axis=0)[: q.shape[0]]
    with np.errstate(over="ignore"):
        return (q * full).astype(np.float16).view(np.uint16)


GRAN_CODE = {"tensor": 0, "channel": 1, "group": 2}


@pytest.mark.parametrize("gran", ["tensor", "channel", "group"])
def test_w8a16_dequant_and_ar(oracle_mod, gran):
    shape = wl.W8A16(R=4, m=12, n=48, k_shard=64, group=32, seed=11)
    xs, wqs, scales = shape.make(gran)
    xs = [wl.bits16(x) for x in xs]
    wqs = [w.numpy() for w in wqs]
    scales = [wl.bits16(s) for s in scales]
    code = GRAN_CODE[gran]
    wds = []
    for wq, s in zip(wqs, scales):
        wd = oracle_mod.dequant_w8a16(wq, s, code, shape.group)
        assert np.array_equal(wd, _numpy_dequant(wq, s, gran, shape.group))
        wds.append(wd)
    got = oracle_mod.matmul_all_reduce_w8a16(xs, wqs, scales, code, shape.group)
    assert _rel(got, _unsharded(xs, wds, torch.float16)) < 1e-13
    if gran == "group":
        # scale rows indexed per rank slab (not by global k) must differ
        bad = _numpy_dequant(wqs[1], scales[0], gran, shape.group)
        assert not np.array_equal(bad, wds[1])


def test_w8a16_unit_scale_is_plain_fp16_ar(oracle_mod):
    rng = np.random.default_rng(4)
    R, m, ks, n = 2, 8, 32, 16
    wqs = [rng.integers(-127, 128, (ks, n)).astype(np.int8) for _ in range(R)]
    xs = [_rand16((m, ks), torch.float16, 90 + r) for r in range(R)]
    one = np.array([0x3C00], dtype=np.uint16)       # binary16 1.0
    got = oracle_mod.matmul_all_reduce_w8a16(xs, wqs, [one] * R, 0)
    wf = [wl.bits16(torch.from_numpy(w.astype(np.float32)).half()) for w in wqs]
    assert np.array_equal(got, oracle_mod.matmul_all_reduce(oracle_mod.F16, xs, wf))


# ------------------------------------------- w8A16 extensions (zero point, bf16) ---

def _bf16_bits_of_f32(x):
    """torch's fp32 -> bfloat16 cast (round to nearest, ties to even)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_encode_ties_and_random_vs_torch(oracle_mod):
    # Values exact in fp32 (so torch's fp32 -> bf16 cast sees the exact value):
    # every tie between neighbouring bf16 values of a few binades, the floats
    # on either side of each tie, random fp32 values and the edges.
    rng = np.random.default_rng(8)
    bits = np.arange(0x3700, 0x4400, dtype=np.uint32)             # [2^-17, 2^9)
    v = (bits << 16).view(np.float32).astype(np.float64)
    mids = (v[:-1] + v[1:]) / 2
    near = np.concatenate([np.nextafter(mids.astype(np.float32), np.float32(0)),
                           np.nextafter(mids.astype(np.float32), np.float32(np.inf))]).astype(np.float64)
    rand = rng.standard_normal(200000).astype(np.float32).astype(np.float64) * 10.0 ** rng.integers(-30, 30, 200000)
    rand = rand.astype(np.float32).astype(np.float64)
    edge = np.array([3.3895313892515355e38, 3.4e38, 1e-40, 9.18355e-41, 1.1754943508222875e-38, 0.0, 1.0, 255.0, 257.0])
    x = np.concatenate([mids, near, rand, edge])
    x = x[np.isfinite(x.astype(np.float32))]
    x = np.concatenate([x, -x])
    assert np.array_equal(oracle_mod.encode_bf16(x), _bf16_bits_of_f32(x))
    assert oracle_mod.encode_bf16(np.array([1e39]))[0] == 0x7f80          # overflow -> inf


def _scale_full(S, gran, group, shape, dt):
    s = _dec(S, dt)
    if gran == "tensor":
        return np.broadcast_to(s.reshape(1, 1), shape)
    if gran == "channel":
        return np.broadcast_to(s.reshape(1, -1), shape)
    return np.repeat(s, group, axis=0)[: shape[0]]


def _zero_full(Z, gran, group, shape):
    z = np.asarray(Z, dtype=np.float64)
    if gran == "tensor":
        return np.broadcast_to(z.reshape(1, 1), shape)
    if gran == "channel":
        return np.broadcast_to(z.reshape(1, -1), shape)
    return np.repeat(z, group, axis=0)[: shape[0]]


@pytest.mark.parametrize("gran", ["tensor", "channel", "group"])
@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
def test_w8a16_zero_point_dequant_vs_brute_force(oracle_mod, gran, dt):
    shape = wl.W8A16(R=4, m=12, n=48, k_shard=64, group=32, seed=13, dtype=dt)
    xs, wqs, scales = shape.make(gran)
    zeros = shape.zeros(gran)
    code = oracle_mod.BF16 if dt == torch.bfloat16 else oracle_mod.F16
    wds = []
    for wq, S, Z in zip(wqs, scales, zeros):
        q, Sb, Zn = wq.numpy(), wl.bits16(S), Z.numpy()
        got = oracle_mod.dequant_w8a16_ex(q, Sb, GRAN_CODE[gran], shape.group, 0, Zn, code)
        exact = (q.astype(np.float64) - _zero_full(Zn, gran, shape.group, q.shape)) * \
            _scale_full(Sb, gran, shape.group, q.shape, dt)
        # the product is exact in fp32 (<= 9 x 11 significant bits), so a single
        # rounding by numpy (binary16) or torch (bfloat16) is the reference
        with np.errstate(over="ignore"):
            ref = exact.astype(np.float16).view(np.uint16) if dt == torch.float16 else _bf16_bits_of_f32(exact)
        assert np.array_equal(got, ref)
        wds.append(got)
    xb = [wl.bits16(x) for x in xs]
    sb = [wl.bits16(S) for S in scales]
    y = oracle_mod.matmul_all_reduce_w8a16(xb, [w.numpy() for w in wqs], sb, GRAN_CODE[gran], shape.group,
                                           zeros=[Z.numpy() for Z in zeros], dtype=code)
    assert _rel(y, _unsharded(xb, wds, dt)) < 1e-13
    # a mutant that ignores the zero point is rejected
    wrong = oracle_mod.dequant_w8a16_ex(wqs[0].numpy(), sb[0], GRAN_CODE[gran], shape.group, 0, None, code)
    assert not np.array_equal(wrong, wds[0])


def test_w8a16_zero_point_special_cases(oracle_mod):
    rng = np.random.default_rng(21)
    k, n = 64, 32
    q = rng.integers(-127, 128, (k, n)).astype(np.int8)
    S = wl.bits16(wl.to16(wl.uniform((n,), 0.001, 0.01, 3, 1), torch.float16))
    # z = 0 is the symmetric form, bit for bit
    sym = oracle_mod.dequant_w8a16(q, S, 1, 0)
    assert np.array_equal(oracle_mod.dequant_w8a16_ex(q, S, 1, 0, 0, np.zeros(n, np.int8), oracle_mod.F16), sym)
    assert np.array_equal(oracle_mod.dequant_w8a16_ex(q, S, 1, 0, 0, None, oracle_mod.F16), sym)
    # q == z everywhere: the weight is exactly zero, so is the AllReduce
    zq = q[0].copy()
    qz = np.broadcast_to(zq, (k, n)).copy()
    assert not np.any(oracle_mod.dequant_w8a16_ex(qz, S, 1, 0, 0, zq, oracle_mod.F16) & 0x7FFF)
    # extreme zero points: q - z = +-255 is exact in both formats
    one16, one_bf = np.array([0x3C00], np.uint16), np.array([0x3F80], np.uint16)
    qe = np.array([[127, -128]], dtype=np.int8).reshape(1, 2)
    ze = np.array([-128], dtype=np.int8)
    d16 = oracle_mod.dequant_w8a16_ex(qe, one16, 0, 0, 0, ze, oracle_mod.F16).view(np.float16).astype(np.float64)
    dbf = _dec(oracle_mod.dequant_w8a16_ex(qe, one_bf, 0, 0, 0, ze, oracle_mod.BF16), torch.bfloat16)
    assert d16.tolist() == [[255.0, 0.0]] and dbf.tolist() == [[255.0, 0.0]]


# ------------------------------------------- MoE dispatch + GroupedMatMul ---

def _dispatch_properties(groups, idxs, T):
    """Checks that do not re-run the construction: every token is dispatched
    exactly once, to the expert it was routed to, and each expert's group is
    ordered by (source rank, token index)."""
    seen = np.zeros((len(idxs), T), dtype=np.int64)
    for e, pairs in enumerate(groups):
        for r, t in pairs:
            seen[r, t] += 1
            if int(idxs[r][t]) != e:
                return False
        keys = pairs[:, 0] * T + pairs[:, 1]
        if np.any(np.diff(keys) <= 0):
            return False
    return bool(np.all(seen == 1))


@pytest.mark.parametrize("R,e_loc", [(1, 1), (2, 2), (4, 3)])
def test_moe_dispatch_properties_and_grouped_gemm(oracle_mod, R, e_loc):
    s = wl.MoEDispatch(R=R, T=37, h=24, f=20, e_loc=e_loc, seed=3 + R, dtype=torch.bfloat16)
    xs, idxs, ws = s.make()
    xb, ib, wb = [wl.bits16(x) for x in xs], [i.numpy() for i in idxs], [wl.bits16(w) for w in ws]
    res = oracle_mod.moe_dispatch_grouped_matmul(oracle_mod.BF16, xb, ib, wb)
    assert len(res) == s.E
    assert _dispatch_properties([g[0] for g in res], ib, s.T)
    assert sum(g[0].shape[0] for g in res) == R * s.T
    for e, (pairs, Xd, Y) in enumerate(res):
        # the dispatched rows are the source rows, bit for bit
        for i, (r, t) in enumerate(pairs):
            assert np.array_equal(Xd[i], xb[r][t])
        if pairs.shape[0]:
            ref = _dec(Xd, torch.bfloat16) @ _dec(wb[e], torch.bfloat16)   # numpy float64
            assert _rel(Y, ref) < 1e-13


def test_moe_single_expert_is_plain_gemm(oracle_mod):
    s = wl.MoEDispatch(R=1, T=16, h=32, f=8, e_loc=1, seed=5, dtype=torch.float16)
    xs, idxs, ws = s.make()
    (pairs, Xd, Y), = oracle_mod.moe_dispatch_grouped_matmul(oracle_mod.F16, [wl.bits16(xs[0])], [idxs[0].numpy()],
                                                             [wl.bits16(ws[0])])
    assert np.array_equal(pairs[:, 1], np.arange(16)) and np.array_equal(Xd, wl.bits16(xs[0]))
    ref = _dec(wl.bits16(xs[0]), torch.float16) @ _dec(wl.bits16(ws[0]), torch.float16)
    assert _rel(Y, ref) < 1e-13


@pytest.mark.parametrize("R,e_loc", [(2, 1), (3, 2)])
def test_moe_combine_per_token_matches_dispatch_and_numpy(oracle_mod, R, e_loc):
    """Two formulations of the combined output: per token (no dispatch order)
    and the dispatched groups mapped back; plus numpy per token."""
    s = wl.MoEDispatch(R=R, T=29, h=16, f=12, e_loc=e_loc, seed=40 + R)
    xs, idxs, ws = s.make()
    xb, ib, wb = [wl.bits16(x) for x in xs], [i.numpy() for i in idxs], [wl.bits16(w) for w in ws]
    per_tok = oracle_mod.moe_token_outputs(oracle_mod.BF16, xb, ib, wb)
    back = [np.full((s.T, s.f), np.nan) for _ in range(R)]
    for pairs, _, Y in oracle_mod.moe_dispatch_grouped_matmul(oracle_mod.BF16, xb, ib, wb):
        for i, (r, t) in enumerate(pairs):
            back[r][t] = Y[i]
    for r in range(R):
        assert np.array_equal(per_tok[r], back[r])
        ref = np.stack([_dec(xb[r][t:t + 1], torch.bfloat16)[0] @ _dec(wb[ib[r][t]], torch.bfloat16)
                        for t in range(s.T)])
        assert _rel(per_tok[r], ref) < 1e-13


def test_moe_topk_combine_pins(oracle_mod):
    """Top-k combine: k = 1 with unit gates is the rounded per-token output
    exactly; for k = 2 the result is within the rounding bound of the exact
    gated sum computed by numpy; swapping the gates of the two slots is
    detected."""
    s = wl.MoEDispatch(R=2, T=31, h=16, f=24, e_loc=2, seed=50)
    xs, _, ws = s.make()
    xb, wb = [wl.bits16(x) for x in xs], [wl.bits16(w) for w in ws]
    idx1, _ = s.routing_topk(1)
    ones = [np.ones((s.T, 1), np.float32) for _ in range(s.R)]
    got1 = oracle_mod.moe_topk_combine(oracle_mod.BF16, xb, [i.numpy() for i in idx1], ones, wb)
    tok = oracle_mod.moe_token_outputs(oracle_mod.BF16, xb, [i.numpy()[:, 0] for i in idx1], wb)
    for r in range(s.R):
        assert np.array_equal(got1[r], oracle_mod.decode16(oracle_mod.encode_bf16(tok[r]), oracle_mod.BF16))
    idx2, g2 = s.routing_topk(2)
    i2, gg = [i.numpy() for i in idx2], [g.numpy() for g in g2]
    for r in range(s.R):
        assert np.all(i2[r][:, 0] != i2[r][:, 1]) and np.allclose(gg[r].sum(axis=1), 1.0, atol=1e-6)
    got2 = oracle_mod.moe_topk_combine(oracle_mod.BF16, xb, i2, gg, wb)
    for r in range(s.R):
        X = _dec(xb[r], torch.bfloat16)
        exact = np.zeros((s.T, s.f))
        bound = np.zeros((s.T, s.f))
        for t in range(s.T):
            for j in range(2):
                y = X[t] @ _dec(wb[i2[r][t, j]], torch.bfloat16)
                exact[t] += np.float64(gg[r][t, j]) * y
                bound[t] += np.float64(gg[r][t, j]) * np.abs(y) * 2.0 ** -8 + 1e-30   # half-ulp of bf16
        assert np.all(np.abs(got2[r] - exact) <= bound)
    swapped = [g[:, ::-1].copy() for g in gg]
    bad = oracle_mod.moe_topk_combine(oracle_mod.BF16, xb, i2, swapped, wb)
    assert not np.allclose(bad[0], got2[0])


def test_moe_dispatch_mutants_rejected(oracle_mod):
    s = wl.MoEDispatch(R=3, T=20, h=8, f=8, e_loc=2, seed=9)
    _, idxs, _ = s.make()
    ib = [i.numpy() for i in idxs]
    groups = oracle_mod.moe_dispatch_order(ib, s.E)
    assert _dispatch_properties(groups, ib, s.T)
    big = max(range(s.E), key=lambda e: groups[e].shape[0])
    swapped = [g.copy() for g in groups]
    swapped[big] = swapped[big][::-1].copy()               # rank/token order reversed
    assert not _dispatch_properties(swapped, ib, s.T)
    dropped = [g.copy() for g in groups]
    dropped[big] = dropped[big][1:]                         # one token lost
    assert not _dispatch_properties(dropped, ib, s.T)
    moved = [g.copy() for g in groups]
    moved[(big + 1) % s.E] = np.concatenate([moved[(big + 1) % s.E], moved[big][:1]])
    moved[big] = moved[big][1:]                             # a token sent to the wrong expert
    assert not _dispatch_properties(moved, ib, s.T)


def test_thread_count_does_not_change_results(oracle_mod):
    xs = [_rand16((20, 64), torch.bfloat16, 100 + r) for r in range(2)]
    ws = [_rand16((64, 37), torch.bfloat16, 110 + r) for r in range(2)]
    a = oracle_mod.matmul_all_reduce(oracle_mod.BF16, xs, ws, nthreads=1)
    b = oracle_mod.matmul_all_reduce(oracle_mod.BF16, xs, ws, nthreads=5)
    assert np.array_equal(a, b)
