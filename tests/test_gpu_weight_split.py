"""Weight gradients with the token reduction split over idle SM pairs.

tp_mlp_dA_ws / tp_mlp_dB_ws cut the reduction of an M x N gradient with
few output tiles into k ranges (fp32 partial outputs added in range order);
the attention block's dWo and dWqkv at h = 1024 take this path.  The oracle
checks those through the attention block (test_gpu_attention's full-size
GPT-2 355M case); here the split result is held to the unsplit one
computed by the same kernels: the two differ only in where the fp32 sum is
cut, so after rounding to bf16 they agree to one bf16 step (at most 2^-7
of the larger magnitude) plus the fp32 difference itself, which matters
only for sums that cancel to near zero (a floor of 1e-3 of the largest
entry), and a split call gives the same bits every time.
"""

import pytest
import torch

from tensor_transformer_mlp_forward_gb300 import binding, inputs

CASES = [
    ("dWo", 8192, 1024, 1024),     # 16 tiles -> 4 k ranges
    ("dWqkv", 8192, 1024, 3072),   # 48 tiles -> 3 k ranges
]


@pytest.mark.gpu
@pytest.mark.parametrize("name,T,M,N", CASES)
def test_split_weight_grad_matches_whole(name, T, M, N):
    assert binding.weight_grad_workspace_bytes(T, M, N) > 0
    w = inputs.custom(T=T, h=M, F=N, t=1, seed=41)
    cpu = inputs.make_inputs(w, keys=("X",))
    X = cpu["X"].cuda()
    # a [T, N] gradient drawn as the dY of an N-wide block
    dZ = inputs.make_inputs(inputs.custom(T=T, h=N, F=8, t=1, seed=42), keys=("dY",))["dY"].cuda()
    whole = binding.tp_mlp_dA(X, dZ, 1)
    split = binding.tp_mlp_dA_ws(X, dZ, 1)
    again = binding.tp_mlp_dA_ws(X, dZ, 1)
    # dB = H^T dY with H = dZ, dY = X: the N x M gradient, MN-major both
    whole_b = binding.tp_mlp_dB(dZ, X, 1)
    split_b = binding.tp_mlp_dB_ws(dZ, X, 1)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.TPMLP_OK
    for a, b in ((split, whole), (split_b, whole_b)):
        diff = (a.float() - b.float()).abs()
        step = (torch.maximum(a.float().abs(), b.float().abs()) * 2.0 ** -7
                + 1e-3 * float(b.float().abs().max()))
        assert bool((diff <= step).all()), float((diff / step).max())
    assert torch.equal(split, again)
