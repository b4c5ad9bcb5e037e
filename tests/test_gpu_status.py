"""Bounded device waits: a wait that nothing completes gives up by itself,
reports TPMLP_ERR_DEVICE_TIMEOUT through the status word, and leaves the
context usable (no trap, no hang)."""

import pytest
import torch

from tensor_transformer_mlp_forward_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    assert binding.device_status() == binding.TPMLP_OK
    status = binding.selftest_bounded_wait(20000)  # 20 ms limit
    assert status == binding.TPMLP_ERR_DEVICE_TIMEOUT
    assert binding.device_status() == binding.TPMLP_OK  # reading cleared it
    w = inputs.TINY
    g = {k: v.cuda() for k, v in inputs.make_inputs(w).items()}
    Y, _, _ = binding.tp_mlp_forward(g["X"], g["A"], g["b1"], g["B"], g["b2"], g["residual"], w.t)
    torch.cuda.synchronize()
    assert torch.isfinite(Y.float()).all()
    assert binding.device_status() == binding.TPMLP_OK


def test_launch_counts():
    w = inputs.TINY
    g = {k: v.cuda() for k, v in inputs.make_inputs(w).items()}
    split = 1 if binding.split_workspace_bytes(w.T, w.h, w.F, w.t) > 0 else 0
    Y, Z, H = binding.tp_mlp_forward(g["X"], g["A"], g["b1"], g["B"], g["b2"], g["residual"], w.t)
    # column GEMM, row-parallel GEMM (+ the partial-sum reduction when split)
    assert binding.last_launch_count() == 2 + split
    binding.tp_mlp_backward(g["dY"], g["X"], g["A"], g["B"], Z, H, w.t)
    # db2 column sums (one or two kernels), dZ GEMM, db1 reduction, dX (+ its
    # reduction when split), dA, dB
    assert binding.last_launch_count() in (6 + split, 7 + split)
