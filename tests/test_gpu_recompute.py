"""Activation recompute: the forward pass saves only X, the backward pass
rebuilds Z and H with the column GEMM.  Same kernels and the same sums as the
plain block, so the outputs must agree with it bit for bit, and with the fp64
oracle within the block's tolerances (1e-2 forward, 2e-2 gradients)."""

import numpy as np
import pytest
import torch

import oracle
from tensor_transformer_mlp_forward_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

TOL_FWD = 1e-2
TOL_BWD = 2e-2


def rel(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    den = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(got - ref)))
    return err / den if den > 0 else err


def np64(x: torch.Tensor) -> np.ndarray:
    return x.detach().to("cpu", torch.float64).numpy()


def both_paths(g, t):
    Y, Z, H = binding.tp_mlp_forward(g["X"], g["A"], g["b1"], g["B"], g["b2"], g["residual"], t)
    plain = (Y,) + binding.tp_mlp_backward(g["dY"], g["X"], g["A"], g["B"], Z, H, t)
    Yr = binding.tp_mlp_forward_recompute(g["X"], g["A"], g["b1"], g["B"], g["b2"],
                                          g["residual"], t)
    rec = (Yr,) + binding.tp_mlp_backward_recompute(g["dY"], g["X"], g["A"], g["b1"], g["B"], t)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    return plain, rec


NAMES = ("Y", "dX", "dA", "dB", "db1", "db2")

SMALL = [
    inputs.TINY,
    inputs.custom(T=300, h=200, F=1536, t=4, seed=31),
    inputs.custom(T=257, h=520, F=1600, t=8, seed=32),
    inputs.custom(T=1, h=8, F=8, t=1, seed=33),
    inputs.SWEEP.with_shape(T=512, t=4),  # a3 and a7 split their reduction
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: f"T{w.T}_h{w.h}_F{w.F}_t{w.t}")
def test_recompute_matches_plain_and_oracle(w):
    cpu = inputs.make_inputs(w)
    g = {k: v.cuda() for k, v in cpu.items()}
    plain, rec = both_paths(g, w.t)
    for name, a, b in zip(NAMES, plain, rec):
        assert torch.equal(a, b), name
    if w.T * w.h * w.F > 2**31:
        return  # the plain path's oracle comparison covers this shape
    Yr, _, _ = oracle.forward(cpu["X"], cpu["A"], cpu["b1"], cpu["B"], cpu["b2"],
                              cpu["residual"], w.t)
    refs = (Yr,) + tuple(oracle.backward(cpu["dY"], cpu["X"], cpu["A"], cpu["b1"], cpu["B"], w.t))
    errs = {n: rel(np64(v), r) for n, v, r in zip(NAMES, rec, refs)}
    bad = {n: e for n, e in errs.items() if e > (TOL_FWD if n == "Y" else TOL_BWD)}
    assert not bad, errs


def test_h_only_column_gemm():
    w = inputs.custom(T=300, h=200, F=1536, t=4, seed=34)
    g = {k: v.cuda() for k, v in inputs.make_inputs(w, keys=("X", "A", "b1")).items()}
    Z, H = binding.tp_mlp_column_gelu(g["X"], g["A"], g["b1"], w.t)
    sentinel = torch.full_like(H, 7.0)
    Z2, H2 = binding.tp_mlp_column_gelu(g["X"], g["A"], g["b1"], w.t, H=sentinel, want_z=False)
    torch.cuda.synchronize()
    assert Z2 is None and torch.equal(H, H2)


def test_recompute_empty_batch():
    w = inputs.custom(T=0, h=64, F=256, t=2, seed=35)
    g = {k: v.cuda() for k, v in inputs.make_inputs(w).items()}
    Y = binding.tp_mlp_forward_recompute(g["X"], g["A"], g["b1"], g["B"], g["b2"],
                                         g["residual"], w.t)
    dX, dA, dB, db1, db2 = binding.tp_mlp_backward_recompute(g["dY"], g["X"], g["A"], g["b1"],
                                                             g["B"], w.t)
    torch.cuda.synchronize()
    assert Y.numel() == 0 and dX.numel() == 0
    for v in (dA, dB, db1, db2):
        assert float(v.abs().max()) == 0.0


def test_recompute_full_size_sampled():
    """MT-NLG 530B (T=2048, h=20480, F=81920, t=8): bitwise equal to the plain
    path, and sampled rows/columns against the oracle."""
    w = inputs.MTNLG_530B
    cpu = inputs.make_inputs(w)
    g = {k: v.cuda() for k, v in cpu.items()}
    plain, rec = both_paths(g, w.t)
    for name, a, b in zip(NAMES, plain, rec):
        assert torch.equal(a, b), name
    del plain
    rows = inputs.sample_indices(w.T, 4, w.seed + 11).numpy()
    cols = inputs.sample_indices(w.F, 8, w.seed + 12).numpy()
    Yr, _, _ = oracle.forward_rows(cpu, w.t, rows)
    dXr = oracle.backward_rows(cpu, w.t, rows)
    dAc, dBr, db1c = oracle.backward_cols(cpu, w.t, cols)
    ri, ci = torch.as_tensor(rows), torch.as_tensor(cols)
    Y, dX, dA, dB, db1, _ = (v.cpu() for v in rec)
    errs = {"Y": (rel(np64(Y[ri]), Yr), TOL_FWD), "dX": (rel(np64(dX[ri]), dXr), TOL_BWD),
            "dA": (rel(np64(dA[:, ci]), dAc), TOL_BWD), "dB": (rel(np64(dB[ci]), dBr), TOL_BWD),
            "db1": (rel(np64(db1[ci]), db1c), TOL_BWD)}
    bad = {k: v for k, v in errs.items() if not v[0] <= v[1]}
    assert not bad, errs
