"""The transposed-operand form of the weight gradients: tp_transpose against
torch's transpose (bit for bit), and tp_mlp_dA_kmajor / tp_mlp_dB_kmajor
against the row-major tp_mlp_dA / tp_mlp_dB and the fp64 oracle.

Both GEMM forms accumulate the same 64-deep k blocks of the token dimension
in the same order in fp32, so their bf16 outputs are compared for equality;
the oracle comparison uses the block's gradient tolerance (2e-2 of max|ref|).
tp_mlp_backward itself runs the transposed form: every backward test of the
block covers it end to end.
"""

import numpy as np
import pytest
import torch

import oracle
from tensor_transformer_mlp_forward_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

TOL_BWD = 2e-2
SENTINEL = -12345.0


@pytest.mark.parametrize("rows,cols,extra", [
    (130, 72, 0), (130, 72, 16), (1, 8, 0), (64, 64, 0), (257, 520, 8), (2048, 1536, 0),
    (77, 4104, 0), (7, 16, 24),
])
def test_transpose_bit_exact(rows, cols, extra):
    g = torch.Generator().manual_seed(rows * 7919 + cols)
    x = torch.randn(rows, cols, generator=g).to(torch.bfloat16).cuda()
    ld = binding.pitch(rows) + extra
    out = torch.full((cols, ld), SENTINEL, dtype=torch.bfloat16, device="cuda")
    binding.tp_transpose(x, ld=ld, out=out)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert torch.equal(out[:, :rows], x.t())
    p = binding.pitch(rows)
    assert bool((out[:, rows:p] == 0).all())             # padding to 8 is zeroed
    assert bool((out[:, p:] == SENTINEL).all())          # nothing further is touched


CASES = [
    inputs.custom(T=300, h=200, F=1536, t=4, seed=41),    # T ragged against 8: ldT = 304
    inputs.custom(T=257, h=520, F=1600, t=8, seed=42),    # f = 200: ragged shard tail
    inputs.custom(T=77, h=64, F=512, t=64, seed=43),      # f = 8
    inputs.custom(T=1, h=8, F=8, t=1, seed=44),
    inputs.custom(T=640, h=384, F=2048, t=2, seed=45),    # several k blocks and tiles
]


@pytest.fixture(params=[0, 2], ids=["single_cta", "cta_pairs"])
def pair_mode(request):
    prev = binding.set_cta_pair_mode(request.param)
    yield request.param
    binding.set_cta_pair_mode(prev)


@pytest.mark.parametrize("w", CASES, ids=lambda w: f"T{w.T}_h{w.h}_F{w.F}_t{w.t}")
def test_kmajor_weight_grads(w, pair_mode):
    cpu = inputs.make_inputs(w)
    g = {k: v.cuda() for k, v in cpu.items()}
    # dZ and H stand-ins with the block's value ranges: the oracle's own
    # forward and backward give them below
    _, _, Hr = oracle.forward(cpu["X"], cpu["A"], cpu["b1"], cpu["B"], cpu["b2"],
                                cpu["residual"], w.t)
    H = torch.as_tensor(Hr).to(torch.bfloat16).cuda()
    dZ = torch.randn(w.T, w.F, generator=torch.Generator().manual_seed(w.seed)).to(torch.bfloat16).cuda()
    X, dY = g["X"], g["dY"]
    dA_mn = binding.tp_mlp_dA(X, dZ, w.t)
    dB_mn = binding.tp_mlp_dB(H, dY, w.t)
    Xt, dZt = binding.tp_transpose(X), binding.tp_transpose(dZ)
    Ht, dYt = binding.tp_transpose(H), binding.tp_transpose(dY)
    dA_k = binding.tp_mlp_dA_kmajor(Xt, dZt, w.T, w.t)
    dB_k = binding.tp_mlp_dB_kmajor(Ht, dYt, w.T, w.t)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert torch.equal(dA_k, dA_mn)
    assert torch.equal(dB_k, dB_mn)
    # against the definition: dA = X^T dZ, dB = H^T dY (fp64, from the bf16 operands)
    x64 = X.double().cpu().numpy()
    refA = x64.T @ dZ.double().cpu().numpy()
    refB = H.double().cpu().numpy().T @ dY.double().cpu().numpy()
    for got, ref in ((dA_k, refA), (dB_k, refB)):
        err = np.max(np.abs(got.double().cpu().numpy() - ref)) / max(np.max(np.abs(ref)), 1e-30)
        assert err <= TOL_BWD


def test_kmajor_empty_batch_zeroes_the_gradient():
    w = inputs.custom(T=0, h=64, F=256, t=2, seed=46)
    Xt = torch.empty((w.h, 0), dtype=torch.bfloat16, device="cuda")
    dZt = torch.empty((w.F, 0), dtype=torch.bfloat16, device="cuda")
    dA = torch.full((w.h, w.F), 3.0, dtype=torch.bfloat16, device="cuda")
    binding.tp_mlp_dA_kmajor(Xt, dZt, 0, w.t, dA=dA)
    torch.cuda.synchronize()
    assert float(dA.abs().max()) == 0.0
