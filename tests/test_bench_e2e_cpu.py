"""The bench's end-to-end leg on CPU: which tensors cross the host link per
operator kind (no GPU needed; tensors stand in for the device buffers)."""
import os
import sys
from types import SimpleNamespace

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _op(kind, R=4, shares=False, n_out=None):
    xs = [torch.zeros(2, 3) for _ in range(R)]
    ws = [torch.ones(3, 5) for _ in range(R)]
    outs = [torch.full((2, 5), float(r)) for r in range(n_out or R)]
    op = bench.Op("x", kind, 1.0, lambda: None, xs + ws, outs, SimpleNamespace(R=R))
    op.shares_prev_inputs = shares
    return op, xs, ws, outs


def test_step_inputs_are_the_activations_only():
    op, xs, ws, _ = _op("ar")
    got = op.step_inputs()
    assert len(got) == len(xs) and all(a is b for a, b in zip(got, xs))
    op, *_ = _op("rs", shares=True)
    assert op.step_inputs() == []


def test_readback_is_every_distinct_result():
    op, _, _, outs = _op("ar")
    assert op.readback() == outs[:1]                      # R bitwise-equal copies: one
    op, _, _, outs = _op("w8a16_ar")
    assert op.readback() == outs[:1]
    op, _, _, outs = _op("rs")
    assert op.readback() == outs                          # distinct row blocks: all
    R = 4
    op, _, _, outs = _op("ag_v2", R=R, n_out=2 * R)       # R products + R equal gathers
    got = op.readback()
    assert len(got) == R + 1 and all(a is b for a, b in zip(got, outs[:R] + outs[R:R + 1]))
