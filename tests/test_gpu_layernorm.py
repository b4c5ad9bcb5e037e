"""Residual add + LayerNorm (the step that produces the MLP block's input X)
against the fp64 oracle, through the C ABI.  Tolerances as for the block:
max|err| / max|ref| <= 1e-2 forward, <= 2e-2 for gradients."""

import numpy as np
import pytest
import torch

import oracle
from tensor_transformer_mlp_forward_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

TOL_FWD = 1e-2
TOL_BWD = 2e-2
EPS = 1e-5


def rel(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    return err / den if den > 0 else err


def np64(x):
    return x.detach().to("cpu", torch.float64).numpy()


def ln_inputs(T, h, seed):
    g = torch.Generator().manual_seed(seed)
    bf = lambda *s, std=1.0, mean=0.0: (torch.randn(*s, generator=g) * std + mean).to(torch.bfloat16)
    return dict(a=bf(T, h), r=bf(T, h), gamma=bf(h, std=0.1, mean=1.0), beta=bf(h, std=0.1),
                dX=bf(T, h), dres=bf(T, h))


# Long rows (4096 .. 32768 columns), ragged row counts and fewer rows than
# SMs as well as the short shapes.
@pytest.mark.parametrize("T,h", [(1, 8), (5, 24), (37, 200), (300, 1024), (64, 20480), (3, 49152),
                                 (130, 4096), (257, 8192), (100, 12288), (33, 16384), (5, 32768),
                                 (3, 20480), (1, 4096)])
@pytest.mark.parametrize("with_dres", [True, False])
def test_layernorm_against_oracle(T, h, with_dres):
    c = ln_inputs(T, h, 100 + T + h)
    g = {k: v.cuda() for k, v in c.items()}
    X, s, mean, rstd = binding.tp_ln_residual_forward(g["a"], g["r"], g["gamma"], g["beta"], EPS)
    ds, dgam, dbet = binding.tp_ln_residual_backward(g["dX"], g["dres"] if with_dres else None,
                                                     g["a"], g["r"], g["gamma"], mean, rstd)
    torch.cuda.synchronize()
    Xr, sr, mr, rr = oracle.ln_forward(c["a"], c["r"], c["gamma"], c["beta"], EPS)
    dsr, dgr, dbr = oracle.ln_backward(c["dX"], c["dres"] if with_dres else None, c["a"], c["r"],
                                       c["gamma"], EPS)
    errs = {"X": (rel(np64(X), Xr), TOL_FWD), "s": (rel(np64(s), sr), TOL_FWD),
            "mean": (rel(np64(mean), mr), TOL_FWD), "rstd": (rel(np64(rstd), rr), TOL_FWD),
            "ds": (rel(np64(ds), dsr), TOL_BWD), "dgamma": (rel(np64(dgam), dgr), TOL_BWD),
            "dbeta": (rel(np64(dbet), dbr), TOL_BWD)}
    bad = {k: v for k, v in errs.items() if not v[0] <= v[1]}
    assert not bad, errs


def test_layernorm_full_size_and_no_s_output():
    T, h = 2048, 20480  # the MT-NLG 530B activations
    c = ln_inputs(T, h, 7)
    g = {k: v.cuda() for k, v in c.items()}
    X, s, mean, rstd = binding.tp_ln_residual_forward(g["a"], g["r"], g["gamma"], g["beta"], EPS,
                                                      want_s=False)
    assert s is None
    ds, dgam, dbet = binding.tp_ln_residual_backward(g["dX"], g["dres"], g["a"], g["r"],
                                                     g["gamma"], mean, rstd)
    torch.cuda.synchronize()
    Xr, _, _, _ = oracle.ln_forward(c["a"], c["r"], c["gamma"], c["beta"], EPS)
    dsr, dgr, dbr = oracle.ln_backward(c["dX"], c["dres"], c["a"], c["r"], c["gamma"], EPS)
    assert rel(np64(X), Xr) <= TOL_FWD
    assert rel(np64(ds), dsr) <= TOL_BWD
    assert rel(np64(dgam), dgr) <= TOL_BWD
    assert rel(np64(dbet), dbr) <= TOL_BWD


@pytest.mark.parametrize("T,h", [(2048, 20480), (700, 8192)])
def test_layernorm_backward_deterministic(T, h):
    """Every sum of the backward (the row sums in the CTA, the column partials
    over row chunks and their total) runs in a fixed order: repeated calls
    agree bit for bit."""
    c = ln_inputs(T, h, 11)
    g = {k: v.cuda() for k, v in c.items()}
    _, _, mean, rstd = binding.tp_ln_residual_forward(g["a"], g["r"], g["gamma"], g["beta"], EPS)
    first = binding.tp_ln_residual_backward(g["dX"], g["dres"], g["a"], g["r"], g["gamma"], mean, rstd)
    for _ in range(3):
        again = binding.tp_ln_residual_backward(g["dX"], g["dres"], g["a"], g["r"], g["gamma"], mean,
                                                rstd)
        for x, y in zip(first, again):
            assert torch.equal(x, y)
    assert binding.device_status() == 0


def test_empty_batch_layernorm():
    h = 64
    gam = torch.ones(h, dtype=torch.bfloat16, device="cuda")
    e = torch.empty((0, h), dtype=torch.bfloat16, device="cuda")
    X, s, mean, rstd = binding.tp_ln_residual_forward(e, e, gam, gam, EPS)
    ds, dg, db = binding.tp_ln_residual_backward(e, None, e, e, gam, mean, rstd,
                                                 dgamma=torch.ones(h, device="cuda"),
                                                 dbeta=torch.ones(h, device="cuda"))
    torch.cuda.synchronize()
    assert X.numel() == 0 and float(dg.abs().max()) == 0.0 and float(db.abs().max()) == 0.0


def test_layer_chain_against_oracle():
    """LayerNorm -> MLP block -> MLP backward -> LayerNorm backward, the GPU
    chain (bf16 between steps) against the fp64 oracle chain."""
    w = inputs.TINY  # T=128, h=256, F=1024, t=2
    mlp = inputs.make_inputs(w)
    c = ln_inputs(w.T, w.h, 5)
    g = {k: v.cuda() for k, v in {**mlp, **c}.items()}
    X, s, mean, rstd = binding.tp_ln_residual_forward(g["a"], g["r"], g["gamma"], g["beta"], EPS)
    Y, Z, H = binding.tp_mlp_forward(X, g["A"], g["b1"], g["B"], g["b2"], s, w.t)
    dX, dA, dB, db1, db2 = binding.tp_mlp_backward(g["dY"], X, g["A"], g["B"], Z, H, w.t)
    ds, dgam, dbet = binding.tp_ln_residual_backward(dX, g["dY"], g["a"], g["r"], g["gamma"],
                                                     mean, rstd)
    torch.cuda.synchronize()
    Xr, sr, _, _ = oracle.ln_forward(c["a"], c["r"], c["gamma"], c["beta"], EPS)
    Yr, _, _ = oracle.forward(Xr, mlp["A"], mlp["b1"], mlp["B"], mlp["b2"], sr, w.t)
    dXr, dAr, dBr, db1r, db2r = oracle.backward(mlp["dY"], Xr, mlp["A"], mlp["b1"], mlp["B"], w.t)
    dsr, dgr, dbr = oracle.ln_backward(dXr, mlp["dY"], c["a"], c["r"], c["gamma"], EPS)
    errs = {"Y": (rel(np64(Y), Yr), TOL_FWD), "dA": (rel(np64(dA), dAr), TOL_BWD),
            "ds": (rel(np64(ds), dsr), TOL_BWD), "dgamma": (rel(np64(dgam), dgr), TOL_BWD),
            "dbeta": (rel(np64(dbet), dbr), TOL_BWD)}
    bad = {k: v for k, v in errs.items() if not v[0] <= v[1]}
    assert not bad, errs
