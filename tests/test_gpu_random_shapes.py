"""Seeded random shapes for every operator against the fp64 oracle (AllReduce,
ReduceScatter, AllGather-V2, w8A16, MoE dispatch + GroupedMatMul + combine,
and the column-slab kernel under random schedules).

Each case draws the rank count, sizes (ragged against the 128 / 256-row,
256-column and 64-deep tiles, from decode-sized m to several tiles), dtype
and chunk count from a fixed seed, within the operators' documented
constraints, so that unit decoding, the 2-SM / single-CTA choice, the rank
split, row groups and chunk orders meet combinations the hand-picked cases
do not."""
import random

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from tensor_matmul_collective_gb300 import coc
from tensor_matmul_collective_gb300 import workloads as wl

from gpu_util import assert_close, bits, to_dev

pytestmark = pytest.mark.gpu
BF16, F16 = torch.bfloat16, torch.float16
CODE = {F16: orc.F16, BF16: orc.BF16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_matmul_collective_gb300 import build
    build.build()
    coc.lib()
    yield
    coc.sync_status()


def _chunks(rng, m):
    return rng.choice([c for c in (1, 2, 4, 8) if m % c == 0])


@pytest.mark.parametrize("seed", range(40))
def test_random_row_parallel(seed):
    rng = random.Random(1000 + seed)
    R = rng.choice([1, 2, 4, 8])
    dt = rng.choice([BF16, F16])
    n = 8 * rng.randint(1, 80)                       # up to 640 columns
    ks = 8 * rng.randint(1, 40)                      # up to 320 per shard
    m = rng.choice([1, 8, 16, 64, 100, 128, 136, 200, 256, 264, 384, 520])
    xs, ws = wl.RowParallel(R=R, m=m, n=n, k_shard=ks, dtype=dt, x_dist="normal(0,1)", w_dist="normal(0,0.02)",
                            seed=seed).make()
    dx, dw = to_dev(xs), to_dev(ws)
    c = _chunks(rng, m)
    det = rng.random() < 0.5
    outs = coc.matmul_all_reduce(dx, dw, chunks=c, deterministic=det)
    coc.sync_status()
    ref = orc.matmul_all_reduce(CODE[dt], bits(xs), bits(ws))
    what = f"AR R={R} m={m} n={n} ks={ks} {dt} chunks={c}"
    for r in range(R):
        assert_close(outs[r], ref, R * ks, what)
        assert torch.equal(outs[r], outs[0])
    if m % (8 * R) == 0:                             # ReduceScatter: m / R in 8-row blocks
        rs = coc.matmul_reduce_scatter(dx, dw, chunks=c, deterministic=det)
        coc.sync_status()
        assert torch.equal(torch.cat(rs, 0), outs[0]), what + " RS concat"


@pytest.mark.parametrize("seed", range(24))
def test_random_all_gather_v2(seed):
    rng = random.Random(2000 + seed)
    R = rng.choice([1, 2, 4, 8])
    dt = rng.choice([BF16, F16])
    ms = rng.choice([8, 16, 24, 64, 72, 128, 136])
    ns = 8 * rng.randint(1, 48)
    k = 8 * rng.randint(1, 40)
    s = wl.ColumnParallelSP(R=R, m_shard=ms, n_shard=ns, k=k, dtype=dt, x_dist="normal(0,1)",
                            w_dist="normal(0,0.02)", seed=seed)
    xs, ws = s.make()
    c = _chunks(rng, R * ms)
    outs, gathered = coc.all_gather_matmul_v2(to_dev(xs), to_dev(ws), chunks=c)
    coc.sync_status()
    xg = orc.all_gather(bits(xs))
    what = f"AG-V2 R={R} ms={ms} ns={ns} k={k} {dt} chunks={c}"
    for r in range(R):
        assert_close(outs[r], orc.all_gather_matmul(CODE[dt], bits(xs), bits(ws), r), k, what)
        assert np.array_equal(wl.bits16(gathered[r].cpu()), xg), what + " gathered"


@pytest.mark.parametrize("seed", range(20))
def test_random_w8a16(seed):
    rng = random.Random(3000 + seed)
    R = rng.choice([1, 2, 4, 8])
    group = rng.choice([64, 128])
    ks = group * rng.randint(1, 3)
    n = 16 * rng.randint(1, 24)
    m = rng.choice([1, 16, 100, 128, 200, 264])
    gran = rng.choice(["tensor", "channel", "group"])
    dt = rng.choice([F16, BF16])
    zero = rng.random() < 0.5
    s = wl.W8A16(R=R, m=m, n=n, k_shard=ks, group=group, seed=seed, dtype=dt)
    xs, wqs, scales = s.make(gran)
    zs = s.zeros(gran) if zero else None
    outs = coc.matmul_all_reduce_w8a16(to_dev(xs), to_dev(wqs), to_dev(scales), gran, group,
                                       zeros=to_dev(zs) if zs is not None else None, chunks=_chunks(rng, m))
    coc.sync_status()
    code = {"tensor": 0, "channel": 1, "group": 2}[gran]
    ref = orc.matmul_all_reduce_w8a16(bits(xs), [w.numpy() for w in wqs], bits(scales), code, group,
                                      zeros=[z.numpy() for z in zs] if zs is not None else None, dtype=CODE[dt])
    for r in range(R):
        assert_close(outs[r], ref, s.K, f"w8A16 R={R} m={m} n={n} ks={ks} {gran} {dt} zero={zero}")


@pytest.mark.parametrize("seed", range(30))
def test_random_column_slab(seed, monkeypatch):
    """The column-slab kernel (decode-sized m), taken whatever the SM count,
    with a random schedule (slab width, cluster split, k-blocks per stage;
    the library reduces what does not fit) on AllReduce, ReduceScatter and
    w8A16 shapes: ragged slabs, k_shard ending inside a k-block, one to
    several slabs per CTA."""
    rng = random.Random(5000 + seed)
    R = rng.choice([1, 2, 4, 8])
    m = rng.choice([1, 3, 8, 16, 31, 32, 33, 64, 96, 100, 127, 128])
    kind = rng.choice(["ar", "rs", "w8"])
    if kind == "rs" and m % (8 * R) != 0:
        kind = "ar"
    n = 16 * rng.randint(1, 400)                     # up to 6400 columns
    plan = (rng.choice([1, 2, 4] if kind == "w8" else [1, 2]), rng.choice([1, 2, 4]), rng.choice([1, 2, 4]))
    for k, v in zip(("COC_SLAB", "COC_SLAB_BOXES", "COC_SLAB_SPLIT", "COC_SLAB_KPS", "COC_W8_PATH"),
                    (1,) + plan + ("slab",)):
        monkeypatch.setenv(k, str(v))
    dt = rng.choice([F16, BF16])
    c = _chunks(rng, m)
    what = f"{kind} R={R} m={m} n={n} {dt} plan={plan} chunks={c}"
    if kind == "w8":
        gran = rng.choice(["tensor", "channel", "group"])
        group = rng.choice([64, 128, 256])
        ks = group * rng.randint(1, 3) if gran == "group" else 8 * rng.randint(1, 64)
        zero = rng.random() < 0.5
        sh = wl.W8A16(R=R, m=m, n=n, k_shard=ks, group=group, seed=seed, dtype=dt)
        xs, wqs, scales = sh.make(gran)
        zs = sh.zeros(gran) if zero else None
        outs = coc.matmul_all_reduce_w8a16(to_dev(xs), to_dev(wqs), to_dev(scales), gran, group,
                                           zeros=to_dev(zs) if zs is not None else None, chunks=c)
        coc.sync_status()
        code = {"tensor": 0, "channel": 1, "group": 2}[gran]
        ref = orc.matmul_all_reduce_w8a16(bits(xs), [w.numpy() for w in wqs], bits(scales), code, group,
                                          zeros=[z.numpy() for z in zs] if zs is not None else None,
                                          dtype=CODE[dt])
        for r in range(R):
            assert_close(outs[r], ref, sh.K, f"{what} ks={ks} {gran} zero={zero}")
            assert torch.equal(outs[r], outs[0])
        return
    ks = 8 * rng.randint(1, 64)                      # up to 512 per shard
    xs, ws = wl.RowParallel(R=R, m=m, n=n, k_shard=ks, dtype=dt, x_dist="normal(0,1)", w_dist="normal(0,0.02)",
                            seed=seed).make()
    dx, dw = to_dev(xs), to_dev(ws)
    ar = coc.matmul_all_reduce(dx, dw, chunks=c)
    rs = coc.matmul_reduce_scatter(dx, dw, chunks=c) if kind == "rs" else None
    coc.sync_status()
    ref = orc.matmul_all_reduce(CODE[dt], bits(xs), bits(ws))
    for r in range(R):
        assert_close(ar[r], ref, R * ks, f"{what} ks={ks} AR rank {r}")
        assert torch.equal(ar[r], ar[0])
    if rs is not None:
        assert torch.equal(torch.cat(rs, 0), ar[0]), what + " concat(RS) != AR"


@pytest.mark.parametrize("seed", range(24))
def test_random_ag_column_slab(seed, monkeypatch):
    """AllGather and AllGather-V2 at decode-sized gathered m through the
    column-slab kernel with a random schedule: m_shard a multiple of 8 with
    R m_shard <= 128, ragged n_shard and k, k x n or n x k weights, V2 with
    random skipped copies (A then read from the first kept copy, or from
    scratch when none is kept)."""
    rng = random.Random(6000 + seed)
    R = rng.choice([1, 2, 4, 8])
    ms = 8 * rng.randint(1, 16 // R)
    ns = 8 * rng.randint(1, 800)                     # up to 6400 columns
    k = 8 * rng.randint(1, 256)                      # up to 2048
    plan = (rng.choice([1, 2]), rng.choice([1, 2, 4]), rng.choice([1, 2, 4]))
    for key, v in zip(("COC_SLAB", "COC_SLAB_BOXES", "COC_SLAB_SPLIT", "COC_SLAB_KPS"), (1,) + plan):
        monkeypatch.setenv(key, str(v))
    dt = rng.choice([F16, BF16])
    nk = rng.random() < 0.3
    v2 = rng.random() < 0.6
    what = f"AG R={R} ms={ms} ns={ns} k={k} {dt} plan={plan} nk={nk} v2={v2}"
    xs, ws = wl.ColumnParallelSP(R=R, m_shard=ms, n_shard=ns, k=k, dtype=dt, x_dist="normal(0,1)",
                                 w_dist="normal(0,0.02)", seed=seed).make()
    dx, dw = to_dev(xs), to_dev(ws)
    m = R * ms
    keep = [rng.random() < 0.6 for _ in range(R)]
    gath = [torch.full((m, k), 5.0, dtype=dt, device=dx[0].device) if kk else None for kk in keep]
    op = "all_gather_v2" if v2 else "all_gather"
    wl_ = [w.t().contiguous() for w in dw] if nk else dw
    res = coc.fused_matmul(op, dx, wl_, w_layout="nk" if nk else "kn", gathered=gath if v2 else None)
    outs = res[0] if v2 else res
    coc.sync_status()
    bx, bw = bits(xs), bits(ws)
    xg = orc.all_gather(bx)
    for r in range(R):
        assert_close(outs[r], orc.all_gather_matmul(CODE[dt], bx, bw, r), k, f"{what} rank {r}")
        if v2 and keep[r]:
            assert np.array_equal(wl.bits16(gath[r].cpu()), xg), f"{what} gathered copy {r}"


@pytest.mark.parametrize("seed", range(16))
def test_random_moe(seed):
    """MoE dispatch + GroupedMatMul + combine: top-1 through the fused combine,
    top-2 / top-3 through the gated combine."""
    rng = random.Random(4000 + seed)
    R = rng.choice([1, 2, 4, 8])
    e_loc = rng.choice([1, 2, 3, 4])
    T = rng.randint(1, 300)
    h = 64 * rng.randint(1, 4)                       # the operator takes h in 64-column steps
    f = 8 * rng.randint(1, 40)
    dt = rng.choice([BF16, F16])
    k = min(rng.choice([1, 1, 2, 3]), R * e_loc)   # k distinct experts
    s = wl.MoEDispatch(R=R, T=T, h=h, f=f, e_loc=e_loc, seed=seed, dtype=dt)
    xs, idxs, ws = s.make()
    dx, w = to_dev(xs), torch.stack(ws).cuda()
    what = f"MoE R={R} T={T} h={h} f={f} e_loc={e_loc} top-{k} {dt}"
    if k == 1:
        y, _, _, _ = coc.moe_dispatch_grouped_matmul(dx, to_dev(idxs), w, e_loc, combine=True)
        coc.sync_status()
        ref = orc.moe_token_outputs(CODE[dt], bits(xs), [i.numpy() for i in idxs], bits(ws))
    else:
        ti, tg = s.routing_topk(k)
        y, _, _, _, _ = coc.moe_topk_grouped_matmul_combine(dx, to_dev(ti), to_dev(tg), w, e_loc)
        coc.sync_status()
        ref = orc.moe_topk_combine(CODE[dt], bits(xs), [i.numpy() for i in ti], [g.numpy() for g in tg], bits(ws))
    for r in range(R):
        assert_close(y[r], ref[r], h, what)
