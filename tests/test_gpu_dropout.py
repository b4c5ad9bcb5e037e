"""Dropout before the residual add, CUDA path against the fp64 oracle through
the C ABI.  The keep decision is integer work (a Philox word against
floor(p * 2^32)), so the GPU's mask must equal the oracle's bit for bit; the
values keep the block's tolerances (1e-2 forward, 2e-2 gradients)."""

import numpy as np
import pytest
import torch

import oracle
from tensor_transformer_mlp_forward_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

TOL_FWD = 1e-2
TOL_BWD = 2e-2
P_DROP = 0.1  # the training recipe's rate


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


@pytest.fixture(params=[0, 2], ids=["single_cta", "cta_pairs"])
def pair_mode(request):
    prev = binding.set_cta_pair_mode(request.param)
    yield request.param
    binding.set_cta_pair_mode(prev)


# (T, h, p, seed, offset): ragged sizes, seeds and offsets past 2^32 (both
# halves of the Philox key and counter in use), p at 0 and far from 0.1.
MASKS = [
    (300, 200, 0.1, 1234, 0),
    (37, 64, 0.5, (7 << 32) | 99, 1 << 34),
    (1, 8, 0.1, 5, 4),
    (513, 4096, 0.9, 2**64 - 1, 2**40 + 8),
    (64, 128, 0.0, 42, 0),
]


@pytest.mark.parametrize("T,h,p,seed,offset", MASKS)
def test_mask_bit_exact(T, h, p, seed, offset):
    dY = torch.ones(T, h, dtype=torch.bfloat16, device="cuda")
    dP = binding.tp_mlp_dropout_grad(dY, p, seed, offset)
    torch.cuda.synchronize()
    keep_gpu = (dP != 0).cpu().numpy().reshape(-1).astype(np.uint8)
    keep_ref = oracle.dropout_mask(seed, offset, T * h, p)
    assert np.array_equal(keep_gpu, keep_ref)
    scale = float(torch.tensor(1.0 / (1.0 - p), dtype=torch.bfloat16))
    kept = dP[dP != 0]
    assert bool((kept.float() == scale).all())


def test_dropout_grad_values():
    T, h, p, seed = 300, 200, P_DROP, 77
    g = torch.Generator().manual_seed(3)
    dY = torch.randn(T, h, generator=g).to(torch.bfloat16)
    dP = binding.tp_mlp_dropout_grad(dY.cuda(), p, seed, 16)
    torch.cuda.synchronize()
    keep = oracle.dropout_mask(seed, 16, T * h, p).reshape(T, h)
    ref = keep * dY.double().numpy() / (1.0 - p)
    assert rel(np64(dP), ref) <= 2.0**-8


SMALL = [
    inputs.TINY,
    inputs.custom(T=300, h=200, F=1536, t=4, seed=21),
    inputs.custom(T=257, h=520, F=1600, t=8, seed=22),   # ragged shard tail
    inputs.custom(T=1, h=8, F=8, t=1, seed=23),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: f"T{w.T}_h{w.h}_F{w.F}_t{w.t}")
def test_forward_backward_against_oracle(w, pair_mode):
    seed, offset = 2024 + w.T, 4 * w.h
    cpu = inputs.make_inputs(w)
    g = {k: v.cuda() for k, v in cpu.items()}
    Y, Z, H = binding.tp_mlp_forward_dropout(g["X"], g["A"], g["b1"], g["B"], g["b2"],
                                             g["residual"], w.t, P_DROP, seed, offset)
    dX, dA, dB, db1, db2 = binding.tp_mlp_backward_dropout(g["dY"], g["X"], g["A"], g["B"], Z, H,
                                                           w.t, P_DROP, seed, offset)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    Yr, Zr, Hr = oracle.forward_dropout(cpu["X"], cpu["A"], cpu["b1"], cpu["B"], cpu["b2"],
                                        cpu["residual"], w.t, P_DROP, seed, offset)
    dXr, dAr, dBr, db1r, db2r = oracle.backward_dropout(cpu["dY"], cpu["X"], cpu["A"], cpu["b1"],
                                                        cpu["B"], w.t, P_DROP, seed, offset)
    errs = {"Y": (rel(np64(Y), Yr), TOL_FWD), "Z": (rel(np64(Z), Zr), TOL_FWD),
            "H": (rel(np64(H), Hr), TOL_FWD), "dX": (rel(np64(dX), dXr), TOL_BWD),
            "dA": (rel(np64(dA), dAr), TOL_BWD), "dB": (rel(np64(dB), dBr), TOL_BWD),
            "db1": (rel(np64(db1), db1r), TOL_BWD), "db2": (rel(np64(db2), db2r), TOL_BWD)}
    bad = {k: v for k, v in errs.items() if not v[0] <= v[1]}
    assert not bad, errs
    # a dropped element is the residual itself, exactly
    keep = oracle.dropout_mask(seed, offset, w.T * w.h, P_DROP).reshape(w.T, w.h).astype(bool)
    dropped = torch.as_tensor(~keep)
    assert torch.equal(Y.cpu()[dropped], cpu["residual"][dropped])


def test_zero_rate_equals_plain_block():
    w = inputs.custom(T=300, h=200, F=1536, t=4, seed=24)
    g = {k: v.cuda() for k, v in inputs.make_inputs(w).items()}
    Y0, _, _ = binding.tp_mlp_forward(g["X"], g["A"], g["b1"], g["B"], g["b2"], g["residual"], w.t)
    Y1, Z, H = binding.tp_mlp_forward_dropout(g["X"], g["A"], g["b1"], g["B"], g["b2"],
                                              g["residual"], w.t, 0.0, 9)
    d0 = binding.tp_mlp_backward(g["dY"], g["X"], g["A"], g["B"], Z, H, w.t)
    d1 = binding.tp_mlp_backward_dropout(g["dY"], g["X"], g["A"], g["B"], Z, H, w.t, 0.0, 9)
    torch.cuda.synchronize()
    assert torch.equal(Y0, Y1)
    for a, b in zip(d0, d1):
        assert torch.equal(a, b)


def test_split_reduction_same_mask():
    """Few output tiles (T=512, h=4096): a3 splits its reduction and the
    dropout moves to the reduction kernel; it must draw the same pattern."""
    w = inputs.SWEEP.with_shape(T=512, t=4)
    cpu = inputs.make_inputs(w, keys=("B", "b2", "residual"))
    g = {k: v.cuda() for k, v in cpu.items()}
    assert binding.split_workspace_bytes(w.T, w.h, w.F, w.t) > 0
    H = torch.randn(w.T, w.F, device="cuda").mul_(0.5).to(torch.bfloat16)
    seed, offset = 31337, 1 << 33
    y_split = binding.tp_mlp_row_sum_dropout(H, g["B"], g["b2"], g["residual"], w.t, P_DROP, seed,
                                             offset)
    empty = torch.empty(0, dtype=torch.uint8, device="cuda")
    y_one = binding.tp_mlp_row_sum_dropout(H, g["B"], g["b2"], g["residual"], w.t, P_DROP, seed,
                                           offset, workspace=empty)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert rel(np64(y_split), np64(y_one)) < TOL_FWD
    keep = oracle.dropout_mask(seed, offset, w.T * w.h, P_DROP).reshape(w.T, w.h).astype(bool)
    dropped = torch.as_tensor(~keep)
    res = cpu["residual"]
    assert torch.equal(y_split.cpu()[dropped], res[dropped])
    assert torch.equal(y_one.cpu()[dropped], res[dropped])


def test_same_seed_same_pattern_across_shard_counts():
    """The pattern lives outside the model-parallel region: t must not change it."""
    outs = []
    for t in (1, 2, 8):
        w = inputs.custom(T=300, h=200, F=2048, t=t, seed=25)
        g = {k: v.cuda() for k, v in inputs.make_inputs(w).items()}
        Y, _, _ = binding.tp_mlp_forward_dropout(g["X"], g["A"], g["b1"], g["B"], g["b2"],
                                                 g["residual"], t, P_DROP, 5, 0)
        outs.append(Y)
    torch.cuda.synchronize()
    for Y in outs[1:]:
        assert torch.equal(outs[0], Y)


def test_full_size_sampled():
    """MT-NLG 530B activations (T=2048, h=20480, F=81920, t=8): sampled rows of
    Y against the oracle's rows with the oracle's mask, and the whole dP."""
    w = inputs.MTNLG_530B
    seed, offset = 0x5EED, 1 << 36
    cpu = inputs.make_inputs(w)
    g = {k: v.cuda() for k, v in cpu.items()}
    Y, Z, H = binding.tp_mlp_forward_dropout(g["X"], g["A"], g["b1"], g["B"], g["b2"],
                                             g["residual"], w.t, P_DROP, seed, offset)
    dP = binding.tp_mlp_dropout_grad(g["dY"], P_DROP, seed, offset)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    rows = inputs.sample_indices(w.T, 8, w.seed + 1).numpy()
    no_res = dict(cpu, residual=torch.zeros_like(cpu["residual"]))
    Pr, _, _ = oracle.forward_rows(no_res, w.t, rows)
    Ycpu = Y.cpu()
    for i, r in enumerate(rows):
        keep = oracle.dropout_mask(seed, offset + int(r) * w.h, w.h, P_DROP).astype(bool)
        res = cpu["residual"][int(r)].double().numpy()
        ref = res + np.where(keep, Pr[i] / (1.0 - P_DROP), 0.0)
        assert rel(np64(Ycpu[int(r)]), ref) <= TOL_FWD, int(r)
        assert torch.equal(Ycpu[int(r)][torch.as_tensor(~keep)],
                           cpu["residual"][int(r)][torch.as_tensor(~keep)])
    keep_all = oracle.dropout_mask(seed, offset, w.T * w.h, P_DROP)
    assert np.array_equal((dP != 0).cpu().numpy().reshape(-1).astype(np.uint8),
                          keep_all & (cpu["dY"] != 0).numpy().reshape(-1).astype(np.uint8))
