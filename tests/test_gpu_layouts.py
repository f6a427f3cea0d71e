"""Weight layouts and the Megatron forward / backward pairings (coc_fused_matmul).

A Megatron linear layer keeps W as [out_features, in_features] (n x k), so
its forward pass is X @ W^T (COC_W_NK) and its data-gradient pass multiplies
by W itself (COC_W_KN with inner = out_features).  These tests check the n x k
layout against the oracle and bitwise against the k x n call on the
transposed weights, for every kernel variant (single-CTA and CTA-pair
tiles, the column-slab kernel at decode-sized AllGather rows), and run the
four TP pairings of the CoC page's layers."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from tensor_matmul_collective_gb300 import coc
from tensor_matmul_collective_gb300 import workloads as wl

from gpu_util import DEV, assert_close, bits, to_dev

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


def _nk(ws):
    """k x n shards -> their n x k (Megatron) storage."""
    return [w.t().contiguous() for w in ws]


ROW_CASES = [
    # op, R, m, n, k_shard, dtype, chunks
    ("all_reduce", 4, 96, 136, 72, BF16, 1),        # single-CTA kernel
    ("all_reduce", 2, 384, 264, 200, F16, 2),       # CTA pairs, ragged n and k
    ("reduce_scatter", 4, 160, 264, 136, BF16, 1),  # rank blocks straddle a pair
    ("reduce_scatter", 2, 64, 72, 64, F16, 2),
]


@pytest.mark.parametrize("op,R,m,n,ks,dt,chunks", ROW_CASES)
def test_row_parallel_nk_layout(op, R, m, n, ks, dt, chunks):
    xs, ws = wl.RowParallel(R=R, m=m, n=n, k_shard=ks, dtype=dt, x_dist="uniform[-1,1]",
                            w_dist="uniform[-1,1]", seed=m + ks).make()
    dx, dw = to_dev(xs), to_dev(ws)
    got = coc.fused_matmul(op, dx, to_dev(_nk(ws)), w_layout="nk", chunks=chunks, deterministic=True)
    ref_kn = coc.fused_matmul(op, dx, dw, w_layout="kn", chunks=chunks, deterministic=True)
    coc.sync_status()
    for r in range(R):
        assert torch.equal(got[r], ref_kn[r]), f"{op} rank {r}: n x k and k x n layouts differ"
        if op == "all_reduce":
            ref = orc.matmul_all_reduce(CODE[dt], bits(xs), bits(ws))
        else:
            ref = orc.matmul_reduce_scatter(CODE[dt], bits(xs), bits(ws), r)
        assert_close(got[r], ref, R * ks, f"{op} nk rank {r}")


AG_CASES = [
    # R, m_shard, n_shard, k, dtype
    (2, 40, 136, 72, BF16),      # 80 gathered rows: the column-slab kernel
    (4, 64, 264, 136, F16),      # 256 rows: CTA pairs on the stacked X (64-row shards)
    (2, 128, 264, 72, BF16),     # 256 rows of whole 128-row shards: CTA pairs, A straight from the shards
    (8, 48, 1400, 136, F16),     # 384 rows x 48 (rank, n-tile) columns: single-CTA tiles on the stacked X
]


@pytest.mark.parametrize("R,ms,ns,k,dt", AG_CASES)
def test_all_gather_nk_layout(R, ms, ns, k, dt):
    s = wl.ColumnParallelSP(R=R, m_shard=ms, n_shard=ns, k=k, dtype=dt, x_dist="uniform[-1,1]",
                            w_dist="uniform[-1,1]", seed=ms + k)
    xs, ws = s.make()
    dx = to_dev(xs)
    outs, gathered = coc.fused_matmul("all_gather_v2", dx, to_dev(_nk(ws)), w_layout="nk")
    plain = coc.fused_matmul("all_gather", dx, to_dev(ws), w_layout="kn")
    coc.sync_status()
    xg = orc.all_gather(bits(xs))
    for r in range(R):
        assert torch.equal(outs[r], plain[r])
        assert_close(outs[r], orc.all_gather_matmul(CODE[dt], bits(xs), bits(ws), r), k, f"AG nk rank {r}")
        assert np.array_equal(wl.bits16(gathered[r].cpu()), xg)


def test_megatron_row_parallel_sp_forward_backward():
    """RowParallelLinear with sequence parallelism, W_r = [n, k_r]:
    forward Y_r = ReduceScatter(X_r @ W_r^T); backward dX_r = AllGather(dY) @ W_r."""
    R, m, n, ks = 4, 256, 264, 128
    xs, ws = wl.RowParallel(R=R, m=m, n=n, k_shard=ks, dtype=BF16, x_dist="normal(0,1)",
                            w_dist="normal(0,0.02)", seed=91).make()
    w_nk = _nk(ws)                                        # Megatron storage of each shard
    y = coc.fused_matmul("reduce_scatter", to_dev(xs), to_dev(w_nk), w_layout="nk")
    dys = [wl.to16(wl.normal((m // R, n), 1.0, 92, r), BF16) for r in range(R)]
    dx = coc.fused_matmul("all_gather", to_dev(dys), to_dev(w_nk), w_layout="kn")
    coc.sync_status()
    for r in range(R):
        assert_close(y[r], orc.matmul_reduce_scatter(orc.BF16, bits(xs), bits(ws), r), R * ks, f"fwd rank {r}")
        ref = orc.all_gather_matmul(orc.BF16, bits(dys), bits(w_nk), r)      # dY_gathered @ W_r
        assert_close(dx[r], ref, n, f"dgrad rank {r}")


def test_megatron_column_parallel_sp_forward_backward():
    """ColumnParallelLinear with sequence parallelism, W_r = [n_r, k]:
    forward Y_r = AllGather(X) @ W_r^T; backward dX = ReduceScatter(dY_r @ W_r)."""
    R, ms, ns, k = 4, 64, 136, 128
    s = wl.ColumnParallelSP(R=R, m_shard=ms, n_shard=ns, k=k, dtype=BF16, x_dist="normal(0,1)",
                            w_dist="normal(0,0.02)", seed=93)
    xs, ws = s.make()
    w_nk = _nk(ws)
    y = coc.fused_matmul("all_gather", to_dev(xs), to_dev(w_nk), w_layout="nk")
    dys = [wl.to16(wl.normal((R * ms, ns), 1.0, 94, r), BF16) for r in range(R)]
    dx = coc.fused_matmul("reduce_scatter", to_dev(dys), to_dev(w_nk), w_layout="kn")
    coc.sync_status()
    for r in range(R):
        assert_close(y[r], orc.all_gather_matmul(orc.BF16, bits(xs), bits(ws), r), k, f"fwd rank {r}")
        ref = orc.matmul_reduce_scatter(orc.BF16, bits(dys), bits(w_nk), r)   # rows of sum_r dY_r @ W_r
        assert_close(dx[r], ref, R * ns, f"dgrad rank {r}")


# ------------------------------------------------------- weight gradient ---

WG_CASES = [
    # R, tokens (inner), out_features (rows), in_features (cols), dtype
    (2, 200, 96, 136, BF16),      # <= 128 rows: single-CTA kernel, ragged tokens
    (4, 256, 264, 72, F16),       # CTA pairs, ragged rows and cols
    (2, 136, 776, 200, BF16),     # 4 pair row tiles, ragged rows, cols and tokens
]


@pytest.mark.parametrize("R,t,rows,cols,dt", WG_CASES)
def test_weight_grad_parity(R, t, rows, cols, dt):
    dys = [wl.to16(wl.uniform((t, rows), -1, 1, 95, r), dt) for r in range(R)]
    xs = [wl.to16(wl.uniform((t, cols), -1, 1, 96, r), dt) for r in range(R)]
    outs = coc.weight_grad(to_dev(dys), to_dev(xs))
    coc.sync_status()
    for r in range(R):
        dyt = np.ascontiguousarray(wl.bits16(dys[r]).T)                      # rows x tokens
        ref = orc.partial_sum(CODE[dt], [dyt], [wl.bits16(xs[r])], np.arange(rows))   # dY_r^T @ X_r
        assert_close(outs[r], ref, t, f"wgrad rank {r}")


def test_megatron_column_parallel_sp_weight_grad_uses_v2_gather():
    """ColumnParallelLinear with SP: the forward pass's V2 gather output is the
    X the weight gradient needs: dW_r = dY_r^T @ AllGather(X)."""
    R, ms, ns, k = 4, 64, 136, 128
    s = wl.ColumnParallelSP(R=R, m_shard=ms, n_shard=ns, k=k, dtype=BF16, x_dist="normal(0,1)",
                            w_dist="normal(0,0.02)", seed=97)
    xs, ws = s.make()
    _, gathered = coc.fused_matmul("all_gather_v2", to_dev(xs), to_dev(_nk(ws)), w_layout="nk")
    dys = [wl.to16(wl.normal((R * ms, ns), 1.0, 98, r), BF16) for r in range(R)]
    dw = coc.weight_grad(to_dev(dys), gathered)
    coc.sync_status()
    xg = orc.all_gather(bits(xs))
    for r in range(R):
        ref = orc.partial_sum(orc.BF16, [np.ascontiguousarray(wl.bits16(dys[r]).T)], [xg], np.arange(ns))
        assert_close(dw[r], ref, R * ms, f"wgrad rank {r}")
        assert dw[r].shape == ws[r].t().shape          # Megatron's [out, in] layout
