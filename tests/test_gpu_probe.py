"""The in-kernel clock probe (coc_debug_clock_probe / _read) the benchmark
uses to report the SM clock its kernels ran at: a recorded launch gives a
plausible clock (cycles / ns between 0.3 and 3 GHz), an unselected slot
stays empty, and reading clears the slot."""
import pytest
import torch

from tensor_matmul_collective_gb300 import coc
from tensor_matmul_collective_gb300 import workloads as wl

from gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_matmul_collective_gb300 import build
    build.build()
    coc.lib()


def test_clock_probe_records_a_plausible_clock():
    xs, ws = wl.RowParallel(R=8, m=1024, n=2048, k_shard=1024, dtype=torch.bfloat16, x_dist="normal(0,1)",
                            w_dist="normal(0,0.02)", seed=3).make()
    dx, dw = to_dev(xs), to_dev(ws)
    outs = coc.matmul_all_reduce(dx, dw)
    for s in range(8):
        coc.clock_read(s)
    coc.clock_probe(3)
    try:
        for _ in range(5):
            coc.matmul_all_reduce(dx, dw, outs)
    finally:
        coc.clock_probe(-1)
    coc.sync_status()
    cyc, ns = coc.clock_read(3)
    assert ns > 0 and cyc > 0
    assert 300.0 < 1e3 * cyc / ns < 3000.0, (cyc, ns)
    assert coc.clock_read(3) == (0, 0)          # read clears the slot
    assert coc.clock_read(2) == (0, 0)          # nothing recorded elsewhere
    coc.matmul_all_reduce(dx, dw, outs)         # probe off: nothing recorded
    coc.sync_status()
    assert coc.clock_read(3) == (0, 0)
    with pytest.raises(coc.CocError):
        coc.clock_probe(8)
