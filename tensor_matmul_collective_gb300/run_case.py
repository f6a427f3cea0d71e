"""Run one fused operator on seeded synthetic data of a chosen size.

Used to profile a single kernel (e.g. under Nsight Compute) and for quick
timing of one shape:

  python -m tensor_matmul_collective_gb300.run_case --op ag_v2 --R 8 --m 512 --n 1792 --k 8192 --iters 3

--op   ar | rs | ag | ag_v2 | w8a16 | plain | moe
--m    rows (ar/rs/w8a16/plain: m; ag/ag_v2: m_shard; moe: tokens per rank)
--n    columns (ag/ag_v2: n_shard; moe: f)
--k    contraction per shard (ag/ag_v2: full k; moe: h)
--eloc experts per rank (moe); --topk routing slots (moe, gated combine if > 1)
--deterministic  fixed rank-order reduction (ar/rs)
"""
from __future__ import annotations

import argparse
import json

import torch

from tensor_matmul_collective_gb300 import coc
from tensor_matmul_collective_gb300 import workloads as wl


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", required=True, choices=["ar", "rs", "ag", "ag_v2", "w8a16", "plain", "moe"])
    ap.add_argument("--R", type=int, default=8)
    ap.add_argument("--m", type=int, required=True)
    ap.add_argument("--n", type=int, required=True)
    ap.add_argument("--k", type=int, required=True)
    ap.add_argument("--dtype", choices=["bf16", "fp16"], default="bf16")
    ap.add_argument("--chunks", type=int, default=1)
    ap.add_argument("--gran", choices=list(wl.SCALE_GRANS), default="group")
    ap.add_argument("--group", type=int, default=128)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--zero", action="store_true", help="w8a16: int8 zero points (asymmetric weights)")
    ap.add_argument("--eloc", type=int, default=1)
    ap.add_argument("--topk", type=int, default=1)
    ap.add_argument("--deterministic", action="store_true", help="ar/rs: fixed rank-order reduction")
    a = ap.parse_args()

    dev = torch.device("cuda:0")
    dt = torch.bfloat16 if a.dtype == "bf16" else torch.float16
    if a.op in ("ag", "ag_v2"):
        s = wl.ColumnParallelSP(R=a.R, m_shard=a.m, n_shard=a.n, k=a.k, dtype=dt, x_dist="normal(0,1)",
                                w_dist="normal(0,0.02)", seed=2)
        xs, ws = s.make()
        dx, dw = [x.to(dev) for x in xs], [w.to(dev) for w in ws]
        outs = [torch.empty(s.m, s.n_shard, dtype=dt, device=dev) for _ in range(a.R)]
        if a.op == "ag_v2":
            g = [torch.empty(s.m, s.k, dtype=dt, device=dev) for _ in range(a.R)]
            run = lambda: coc.all_gather_matmul_v2(dx, dw, outs, g, chunks=a.chunks)  # noqa: E731
        else:
            run = lambda: coc.all_gather_matmul(dx, dw, outs, chunks=a.chunks)  # noqa: E731
        flops = s.flops()
    elif a.op == "moe":
        s = wl.MoEDispatch(R=a.R, T=a.m, h=a.k, f=a.n, e_loc=a.eloc, seed=21, dtype=dt)
        xs, idxs, ws = s.make()
        dx, w = [x.to(dev) for x in xs], torch.stack(ws).to(dev)
        if a.topk > 1:
            ti, tg = s.routing_topk(a.topk)
            ti, tg = [i.to(dev) for i in ti], [g.to(dev) for g in tg]
            run = lambda: coc.moe_topk_grouped_matmul_combine(dx, ti, tg, w, a.eloc)  # noqa: E731
        else:
            di = [i.to(dev) for i in idxs]
            run = lambda: coc.moe_dispatch_grouped_matmul(dx, di, w, a.eloc)  # noqa: E731
        flops = s.flops() * a.topk
    elif a.op == "w8a16":
        s = wl.W8A16(R=a.R, m=a.m, n=a.n, k_shard=a.k, group=a.group, seed=3, dtype=dt)
        xs, wqs, scales = s.make(a.gran)
        dx, dw, dsc = [x.to(dev) for x in xs], [w.to(dev) for w in wqs], [t.to(dev) for t in scales]
        dz = [z.to(dev) for z in s.zeros(a.gran)] if a.zero else None
        outs = [torch.empty(s.m, s.n, dtype=dt, device=dev) for _ in range(a.R)]
        run = lambda: coc.matmul_all_reduce_w8a16(dx, dw, dsc, a.gran, a.group, outs, chunks=a.chunks,  # noqa: E731
                                                  zeros=dz)
        flops = s.flops()
    else:
        s = wl.RowParallel(R=a.R, m=a.m, n=a.n, k_shard=a.k, dtype=dt, x_dist="normal(0,1)",
                           w_dist="normal(0,0.02)", seed=1)
        xs, ws = s.make()
        dx, dw = [x.to(dev) for x in xs], [w.to(dev) for w in ws]
        if a.op == "ar":
            outs = [torch.empty(s.m, s.n, dtype=dt, device=dev) for _ in range(a.R)]
            run = lambda: coc.matmul_all_reduce(dx, dw, outs, chunks=a.chunks,  # noqa: E731
                                                deterministic=a.deterministic)
        elif a.op == "rs":
            outs = [torch.empty(s.m // a.R, s.n, dtype=dt, device=dev) for _ in range(a.R)]
            run = lambda: coc.matmul_reduce_scatter(dx, dw, outs, chunks=a.chunks,  # noqa: E731
                                                    deterministic=a.deterministic)
        else:
            out = torch.empty(s.m, s.n, dtype=dt, device=dev)
            run = lambda: coc.matmul(dx, dw, out)  # noqa: E731
        flops = s.flops()

    run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.iters):
        run()
    e1.record()
    torch.cuda.synchronize()
    coc.sync_status()
    ms = e0.elapsed_time(e1) / a.iters
    print(json.dumps({"op": a.op, "R": a.R, "m": a.m, "n": a.n, "k": a.k, "ms": ms,
                      "tflops": flops / (ms / 1e3) / 1e12}))


if __name__ == "__main__":
    main()
