"""Parity of every fused operator at shapes where the 2-SM (CTA pair) and the
single-CTA kernels differ: row counts that end inside a pair tile or inside
one CTA's half, ReduceScatter rank blocks that straddle the two CTAs of a
pair, AllGather shards smaller than a CTA's rows, ragged n and k.

Run as a script (python tests/variant_check.py) in a process whose COC_PAIR
environment variable selects the variant; exits non-zero on a mismatch.
"""
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

from oracle import oracle as orc  # noqa: E402
from tensor_matmul_collective_gb300 import coc  # noqa: E402
from tensor_matmul_collective_gb300 import workloads as wl  # noqa: E402

from gpu_util import assert_close, bits, to_dev  # noqa: E402

BF16, F16 = torch.bfloat16, torch.float16
CODE = {F16: orc.F16, BF16: orc.BF16}


def check_ar(R, m, n, ks, dt, chunks):
    xs, ws = wl.RowParallel(R=R, m=m, n=n, k_shard=ks, dtype=dt, x_dist="uniform[-1,1]",
                            w_dist="uniform[-1,1]", seed=m + n).make()
    outs = coc.matmul_all_reduce(to_dev(xs), to_dev(ws), chunks=chunks, deterministic=True)
    coc.sync_status()
    ref = orc.matmul_all_reduce(CODE[dt], bits(xs), bits(ws))
    for r, o in enumerate(outs):
        assert_close(o, ref, R * ks, f"AR m={m} rank {r}")
        assert torch.equal(o, outs[0])


def check_rs(R, m, n, ks, dt, chunks):
    xs, ws = wl.RowParallel(R=R, m=m, n=n, k_shard=ks, dtype=dt, x_dist="uniform[-1,1]",
                            w_dist="uniform[-1,1]", seed=m + 7).make()
    outs = coc.matmul_reduce_scatter(to_dev(xs), to_dev(ws), chunks=chunks)
    coc.sync_status()
    for r, o in enumerate(outs):
        assert_close(o, orc.matmul_reduce_scatter(CODE[dt], bits(xs), bits(ws), r), R * ks, f"RS m={m} rank {r}")


def check_ag(R, ms, ns, k, dt, chunks):
    s = wl.ColumnParallelSP(R=R, m_shard=ms, n_shard=ns, k=k, dtype=dt, x_dist="uniform[-1,1]",
                            w_dist="uniform[-1,1]", seed=ms + ns)
    xs, ws = s.make()
    outs, gathered = coc.all_gather_matmul_v2(to_dev(xs), to_dev(ws), chunks=chunks)
    coc.sync_status()
    xg = orc.all_gather(bits(xs))
    for r in range(R):
        assert_close(outs[r], orc.all_gather_matmul(CODE[dt], bits(xs), bits(ws), r), k, f"AG ms={ms} rank {r}")
        assert np.array_equal(wl.bits16(gathered[r].cpu()), xg)


def check_w8(R, m, n, ks, group, gran, dt=F16, zero=False):
    s = wl.W8A16(R=R, m=m, n=n, k_shard=ks, group=group, seed=m, dtype=dt)
    xs, wqs, scales = s.make(gran)
    zs = s.zeros(gran) if zero else None
    outs = coc.matmul_all_reduce_w8a16(to_dev(xs), to_dev(wqs), to_dev(scales), gran, group,
                                       zeros=to_dev(zs) if zs is not None else None)
    coc.sync_status()
    code = {"tensor": 0, "channel": 1, "group": 2}[gran]
    ref = orc.matmul_all_reduce_w8a16(bits(xs), [w.numpy() for w in wqs], bits(scales), code, group,
                                      zeros=[z.numpy() for z in zs] if zs is not None else None, dtype=CODE[dt])
    for r, o in enumerate(outs):
        assert_close(o, ref, s.K, f"w8A16 {dt} zero={zero} {gran} m={m} rank {r}")


def main():
    check_ar(4, 384, 520, 200, BF16, 2)     # second pair tile: its upper CTA has no rows
    check_ar(2, 200, 136, 72, F16, 1)       # rows end inside the upper CTA of the first tile
    check_ar(8, 640, 264, 64, BF16, 8)      # 2.5 pair tiles, chunks of 80 rows
    check_rs(4, 160, 264, 136, BF16, 1)     # rank 3's 40-row block straddles the pair's CTAs
    check_rs(8, 512, 256, 64, F16, 4)
    check_ag(4, 40, 136, 72, BF16, 1)       # 8-row A boxes; shards span both CTAs of a pair
    check_ag(2, 200, 264, 136, F16, 1)      # 400 gathered rows
    check_ag(8, 512, 264, 64, BF16, 1)      # whole-tile A boxes from 512-row shards
    for gran in ("tensor", "channel", "group"):
        check_w8(2, 200, 272, 256, 128, gran)
        check_w8(2, 200, 272, 256, 128, gran, dt=BF16, zero=True)
    print("variant ok:", os.environ.get("COC_PAIR", "auto"))


if __name__ == "__main__":
    main()
