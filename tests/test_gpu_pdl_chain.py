"""Dependent launches in a chain.

Both kernels are launched as programmatic dependent launches: a kernel may
start its set-up while the previous one in the stream finishes and waits for
it before its first global-memory access.  Here the second call of a chain
reads what the first one wrote: Y = AllReduce(X, W) (R rank copies), then
Z = AllReduce(Y_r as the rank shards, V), so Z = sum_r Y_r V_r.  The
outputs start filled with a NaN canary, so a read of Y before the first call
finished shows as non-finite or wrong values.  Chains of 2 and 6 calls, at
decode size (column-slab kernel) and at row counts that take the persistent
kernel, eagerly and replayed from a CUDA graph; every link is checked
against the fp64 oracle applied to the previous link's GPU result."""
import pytest
import torch

from oracle import oracle as orc
from tensor_matmul_collective_gb300 import coc
from tensor_matmul_collective_gb300 import workloads as wl

from gpu_util import DEV, assert_close, bits

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16
NAN16 = 0x7FC1   # a quiet NaN as bf16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_matmul_collective_gb300 import build
    build.build()
    coc.lib()
    yield
    coc.sync_status()


def _canary(shape, R):
    return [torch.full(shape, NAN16, dtype=torch.int16, device=DEV).view(BF16) for _ in range(R)]


def _weights(R, k, n, seed):
    gen = torch.Generator().manual_seed(seed)
    return [(0.02 * torch.randn(k, n, generator=gen)).to(BF16).to(DEV) for _ in range(R)]


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
@pytest.mark.parametrize("R,m,n,ks,links", [
    (8, 16, 4096, 512, 2),      # decode size: column-slab kernels back to back
    (4, 16, 1024, 256, 6),      # a longer chain of small calls
    (8, 200, 2048, 256, 2),     # single-CTA persistent tiles
    (2, 384, 1024, 128, 3),     # 2-SM pair tiles
])
def test_chained_allreduce_reads_the_previous_result(R, m, n, ks, links, graph):
    xs, ws = wl.RowParallel(R=R, m=m, n=n, k_shard=ks, dtype=BF16, x_dist="normal(0,1)", w_dist="normal(0,0.02)",
                            seed=m + links).make()
    x0 = [x.to(DEV) for x in xs]
    w0 = [w.to(DEV) for w in ws]
    # link i > 0: the rank shards are the previous link's R output copies (m x n)
    vs = [_weights(R, n, n, 100 + i) for i in range(1, links)]
    outs = [_canary((m, n), R) for _ in range(links)]

    def chain():
        coc.matmul_all_reduce(x0, w0, outs[0])
        for i in range(1, links):
            coc.matmul_all_reduce(outs[i - 1], vs[i - 1], outs[i])

    if graph:
        chain()                       # first call on the device outside capture
        torch.cuda.synchronize()
        for o in outs:
            for t in o:
                t.view(torch.int16).fill_(NAN16)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            chain()
        for o in outs:
            for t in o:
                t.view(torch.int16).fill_(NAN16)
        g.replay()
    else:
        chain()
    coc.sync_status()
    torch.cuda.synchronize()
    ref0 = orc.matmul_all_reduce(orc.BF16, bits(xs), bits(ws))
    assert_close(outs[0][0], ref0, R * ks, "link 0")
    for i in range(1, links):
        prev = [t.cpu() for t in outs[i - 1]]
        ref = orc.matmul_all_reduce(orc.BF16, bits(prev), bits([v.cpu() for v in vs[i - 1]]))
        for r in range(R):
            assert_close(outs[i][r], ref, R * n, f"link {i} rank {r}")
            assert torch.equal(outs[i][r], outs[i][0])
