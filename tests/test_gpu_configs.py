"""The full-size configurations (BLOOM-7B, LLaMA2-70B, BLOOM-176B TP8 layer
shapes and the w8A16 layer) checked against the fp64 oracle on seeded output
rows (seed 1234), plus the bitwise properties that hold at any size:
AllReduce copies identical, ReduceScatter blocks equal to AllReduce rows, the
V2 gather a bit copy, and deterministic results identical across 10 runs and
chunk counts 1/2/4/8.

Every operator runs at the chunk count bench.py times it with (the TP8 suite
in workloads.TP8_SUITE) and at chunks = 4 as a second schedule; the chunk
count changes the work-unit order and the L2 row grouping, so both launch
configurations are checked.  test_bench_suite_outputs goes one step further:
it builds the suite with bench.py's own code and checks the outputs of the
very calls the benchmark times."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from tensor_matmul_collective_gb300 import coc
from tensor_matmul_collective_gb300 import workloads as wl

from gpu_util import DEV, assert_close, bits, to_dev

pytestmark = pytest.mark.gpu

SUITE_CHUNKS = {w.name: w.chunks for w in wl.TP8_SUITE}


def _chunk_cases(name):
    """The benchmark's chunk count for this layer, then chunks = 4."""
    c = SUITE_CHUNKS[name]
    return [c] + ([4] if c != 4 else [1])


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_matmul_collective_gb300 import build
    build.build()
    coc.lib()
    yield
    torch.cuda.empty_cache()


@pytest.mark.parametrize("chunks", _chunk_cases("bloom7b_ar"))
def test_bloom7b_allreduce(chunks):
    s = wl.BLOOM7B_AR
    xs, ws = s.make()
    outs = coc.matmul_all_reduce(to_dev(xs), to_dev(ws), chunks=chunks)
    coc.sync_status()
    rows = wl.sample_rows(s.m)
    ref = orc.matmul_all_reduce(orc.BF16, bits(xs), bits(ws), rows)
    idx = torch.from_numpy(rows).to(outs[0].device)
    for r, o in enumerate(outs):
        assert torch.equal(o, outs[0])
    assert_close(outs[0].index_select(0, idx), ref, s.K, "bloom7b AR")


@pytest.mark.parametrize("chunks", _chunk_cases("llama70b_ag_v2"))
def test_llama70b_all_gather_v2(chunks):
    s = wl.LLAMA70B_AG
    xs, ws = s.make()
    outs, gathered = coc.all_gather_matmul_v2(to_dev(xs), to_dev(ws), chunks=chunks)
    coc.sync_status()
    xg = orc.all_gather(bits(xs))
    for g in gathered:
        assert np.array_equal(wl.bits16(g.cpu()), xg)
    bx, bw = bits(xs), bits(ws)
    for r in range(s.R):
        # 256 rows on rank 0, 64 on every other rank (a different seeded sample each)
        rr = wl.sample_rows(s.m) if r == 0 else wl.sample_rows(s.m, 64, seed=1234 + r)
        ref = orc.all_gather_matmul(orc.BF16, bx, bw, r, rr)
        idx = torch.from_numpy(rr).to(outs[r].device)
        assert_close(outs[r].index_select(0, idx), ref, s.k, f"llama70b AG rank {r}")


@pytest.mark.parametrize("chunks", _chunk_cases("llama70b_rs"))
def test_llama70b_reduce_scatter(chunks):
    s = wl.LLAMA70B_RS
    xs, ws = s.make()
    dx, dw = to_dev(xs), to_dev(ws)
    outs = coc.matmul_reduce_scatter(dx, dw, chunks=chunks)
    coc.sync_status()
    rows = wl.sample_rows(s.m)
    ms = s.m // s.R
    bx, bw = bits(xs), bits(ws)
    for r in range(s.R):
        local = rows[(rows >= r * ms) & (rows < (r + 1) * ms)] - r * ms
        ref = orc.matmul_reduce_scatter(orc.BF16, bx, bw, r, local)
        idx = torch.from_numpy(local).to(outs[r].device)
        assert_close(outs[r].index_select(0, idx), ref, s.K, f"llama70b RS rank {r}")


@pytest.mark.parametrize("chunks", _chunk_cases("w8a16_ar"))
@pytest.mark.parametrize("gran", ["tensor", "channel", "group"])
def test_w8a16_allreduce(gran, chunks):
    s = wl.W8A16_AR
    xs, wqs, scales = s.make(gran)
    outs = coc.matmul_all_reduce_w8a16(to_dev(xs), to_dev(wqs), to_dev(scales), gran, s.group, chunks=chunks)
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


def test_bench_suite_outputs():
    """The benchmark's own calls: bench.build_suite sets up every operator of
    the timed step (same shapes, seeds, chunk counts, output buffers and
    call sites); each is run once here and its outputs are checked against
    the oracle on 64 seeded rows, plus the bitwise copy properties."""
    import bench

    ops, host = bench.build_suite(DEV)
    for op in ops:
        op.run()
    coc.sync_status()
    by = {op.name: op for op in ops}
    rows = lambda m: wl.sample_rows(m, 64, seed=4321)  # noqa: E731

    def sel(t, rr):
        return t.index_select(0, torch.from_numpy(rr).to(t.device))

    # BLOOM-7B AllReduce
    s, op = wl.BLOOM7B_AR, by["bloom7b_ar"]
    xs, ws = host["bloom7b"]
    rr = rows(s.m)
    assert all(torch.equal(o, op.outputs[0]) for o in op.outputs)
    assert_close(sel(op.outputs[0], rr), orc.matmul_all_reduce(orc.BF16, bits(xs), bits(ws), rr), s.K, "bench 7B AR")
    # LLaMA2-70B AllGather-V2: every rank's product, every gather copy
    s, op = wl.LLAMA70B_AG, by["llama70b_ag_v2"]
    xs, ws = host["llama_ag"]
    bx, bw = bits(xs), bits(ws)
    xg = orc.all_gather(bx)
    for r in range(s.R):
        assert np.array_equal(wl.bits16(op.outputs[s.R + r].cpu()), xg), f"bench AG-V2 gather {r}"
        rr = wl.sample_rows(s.m, 16, seed=4321 + r)
        assert_close(sel(op.outputs[r], rr), orc.all_gather_matmul(orc.BF16, bx, bw, r, rr), s.k,
                     f"bench AG-V2 rank {r}")
    # LLaMA2-70B ReduceScatter
    s, op = wl.LLAMA70B_RS, by["llama70b_rs"]
    xs, ws = host["llama_rs"]
    bx, bw = bits(xs), bits(ws)
    ms = s.m // s.R
    for r in range(s.R):
        rr = wl.sample_rows(ms, 8, seed=4321 + r)
        assert_close(sel(op.outputs[r], rr), orc.matmul_reduce_scatter(orc.BF16, bx, bw, r, rr), s.K,
                     f"bench RS rank {r}")
    # w8A16 at the three granularities
    s = wl.W8A16_AR
    for code, gran in enumerate(wl.SCALE_GRANS):
        op = by[f"w8a16_ar_{gran}"]
        xs, wqs, scales = host[f"w8_{gran}"]
        rr = rows(s.m)
        assert all(torch.equal(o, op.outputs[0]) for o in op.outputs)
        ref = orc.matmul_all_reduce_w8a16(bits(xs), [w.numpy() for w in wqs], bits(scales), code, s.group, rr)
        assert_close(sel(op.outputs[0], rr), ref, s.K, f"bench w8A16 {gran}")
    # BLOOM-176B deterministic AllReduce and ReduceScatter (same inputs)
    s = wl.BLOOM176B
    xs, ws = host["bloom176b"]
    bx, bw = bits(xs), bits(ws)
    ar, rs = by["bloom176b_det_ar"], by["bloom176b_det_rs"]
    assert all(torch.equal(o, ar.outputs[0]) for o in ar.outputs)
    assert torch.equal(torch.cat(rs.outputs, 0), ar.outputs[0])
    rr = wl.sample_rows(s.m, 32, seed=4321)
    assert_close(sel(ar.outputs[0], rr), orc.matmul_all_reduce(orc.BF16, bx, bw, rr), s.K, "bench 176B AR")
    del ops, host
    torch.cuda.empty_cache()
