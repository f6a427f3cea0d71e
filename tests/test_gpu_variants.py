"""Both variants of the persistent kernel — the 2-SM CTA-pair kernel and the
single-CTA kernel — against the oracle at edge shapes.  The variant is
chosen per process (COC_PAIR), so each runs in a subprocess; COC_SLAB=0
keeps the decode-sized rows on the persistent kernel too (by default the
column-slab kernel takes them)."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("pair", ["0", "1"])
def test_kernel_variant_parity(pair):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_matmul_collective_gb300 import build
    build.build()
    env = dict(os.environ, COC_PAIR=pair, COC_SLAB="0")
    r = subprocess.run([sys.executable, os.path.join(HERE, "variant_check.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "variant ok" in r.stdout
