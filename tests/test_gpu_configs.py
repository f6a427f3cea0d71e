"""The full-size configurations (BLOOM-7B, LLaMA2-70B, BLOOM-176B TP8 layer
shapes and the w8A16 layer), in the launch configuration bench.py times,
checked against the fp64 oracle on 256 seeded output rows (seed 1234), plus
the bitwise properties that hold at any size: AllReduce copies identical,
ReduceScatter blocks equal to AllReduce rows, the V2 gather a bit copy, and
deterministic results identical across 10 runs and chunk counts 1/2/4/8."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from tensor_matmul_collective_gb300 import coc
from tensor_matmul_collective_gb300 import workloads as wl

from gpu_util import assert_close, bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_matmul_collective_gb300 import build
    build.build()
    coc.lib()
    yield
    torch.cuda.empty_cache()


def test_bloom7b_allreduce():
    s = wl.BLOOM7B_AR
    xs, ws = s.make()
    outs = coc.matmul_all_reduce(to_dev(xs), to_dev(ws), chunks=4)
    coc.sync_status()
    rows = wl.sample_rows(s.m)
    ref = orc.matmul_all_reduce(orc.BF16, bits(xs), bits(ws), rows)
    idx = torch.from_numpy(rows).to(outs[0].device)
    for r, o in enumerate(outs):
        assert torch.equal(o, outs[0])
    assert_close(outs[0].index_select(0, idx), ref, s.K, "bloom7b AR")


def test_llama70b_all_gather_v2():
    s = wl.LLAMA70B_AG
    xs, ws = s.make()
    outs, gathered = coc.all_gather_matmul_v2(to_dev(xs), to_dev(ws), chunks=4)
    coc.sync_status()
    xg = orc.all_gather(bits(xs))
    for g in gathered:
        assert np.array_equal(wl.bits16(g.cpu()), xg)
    rows = wl.sample_rows(s.m)
    bx, bw = bits(xs), bits(ws)
    for r in range(s.R):
        rr = rows if r == 0 else rows[r::8]      # 256 rows on rank 0, 32 on the others
        ref = orc.all_gather_matmul(orc.BF16, bx, bw, r, rr)
        idx = torch.from_numpy(rr).to(outs[r].device)
        assert_close(outs[r].index_select(0, idx), ref, s.k, f"llama70b AG rank {r}")


def test_llama70b_reduce_scatter():
    s = wl.LLAMA70B_RS
    xs, ws = s.make()
    dx, dw = to_dev(xs), to_dev(ws)
    outs = coc.matmul_reduce_scatter(dx, dw, chunks=4)
    coc.sync_status()
    rows = wl.sample_rows(s.m)
    ms = s.m // s.R
    bx, bw = bits(xs), bits(ws)
    for r in range(s.R):
        local = rows[(rows >= r * ms) & (rows < (r + 1) * ms)] - r * ms
        ref = orc.matmul_reduce_scatter(orc.BF16, bx, bw, r, local)
        idx = torch.from_numpy(local).to(outs[r].device)
        assert_close(outs[r].index_select(0, idx), ref, s.K, f"llama70b RS rank {r}")


@pytest.mark.parametrize("gran", ["tensor", "channel", "group"])
def test_w8a16_allreduce(gran):
    s = wl.W8A16_AR
    xs, wqs, scales = s.make(gran)
    outs = coc.matmul_all_reduce_w8a16(to_dev(xs), to_dev(wqs), to_dev(scales), gran, s.group, chunks=4)
    coc.sync_status()
    for o in outs:
        assert torch.equal(o, outs[0])
    rows = wl.sample_rows(s.m)
    code = {"tensor": 0, "channel": 1, "group": 2}[gran]
    ref = orc.matmul_all_reduce_w8a16(bits(xs), [w.numpy() for w in wqs], bits(scales), code, s.group, rows)
    idx = torch.from_numpy(rows).to(outs[0].device)
    assert_close(outs[0].index_select(0, idx), ref, s.K, f"w8A16 {gran}")


def test_bloom176b_deterministic_allreduce_and_reduce_scatter():
    s = wl.BLOOM176B
    xs, ws = s.make()
    dx, dw = to_dev(xs), to_dev(ws)
    ar0 = [t.clone() for t in coc.matmul_all_reduce(dx, dw, chunks=1, deterministic=True)]
    rs0 = [t.clone() for t in coc.matmul_reduce_scatter(dx, dw, chunks=1, deterministic=True)]
    coc.sync_status()
    for o in ar0:
        assert torch.equal(o, ar0[0])
    assert torch.equal(torch.cat(rs0, 0), ar0[0])
    ar_out = [torch.empty_like(t) for t in ar0]
    rs_out = [torch.empty_like(t) for t in rs0]
    for chunks in (1, 2, 4, 8):
        for _ in range(10):
            coc.matmul_all_reduce(dx, dw, ar_out, chunks=chunks, deterministic=True)
            coc.matmul_reduce_scatter(dx, dw, rs_out, chunks=chunks, deterministic=True)
            assert all(torch.equal(a, b) for a, b in zip(ar_out, ar0)), f"AR chunks={chunks}"
            assert all(torch.equal(a, b) for a, b in zip(rs_out, rs0)), f"RS chunks={chunks}"
    coc.sync_status()
    rows = wl.sample_rows(s.m)
    ref = orc.matmul_all_reduce(orc.BF16, bits(xs), bits(ws), rows)
    idx = torch.from_numpy(rows).to(ar0[0].device)
    assert_close(ar0[0].index_select(0, idx), ref, s.K, "bloom176b AR")
