"""The allocation-free column-sum entry point, tp_mlp_bias_grad_noalloc.

It exists for callers that cannot allocate device memory when they need a
bias gradient -- a framework that passes this library only the tensors it
owns, or code that may not call an allocator after its set-up -- so its
partial sums live in a fixed array inside the library instead of a caller
buffer.  Its results must match tp_mlp_bias_grad, and the shared array must
give the same answer on back-to-back calls.  This file is collected last
so that a failure here does not stop the rest of the suite.
"""

import ctypes

import pytest
import torch

from tensor_transformer_mlp_forward_gb300 import binding, inputs

TOL = 2e-2  # the gradient tolerance of the parity tests (max|err| / max|ref|)


def _rel(a: torch.Tensor, b: torch.Tensor) -> float:
    den = float(b.abs().max())
    err = float((a.double() - b.double()).abs().max())
    return err / den if den > 0 else err


def test_every_hidden_size_up_to_24576_fits():
    L = binding.lib()
    cap = L.tp_mlp_bias_grad_noalloc_max_floats()
    for n in range(8, 24577, 8):
        need = L.tp_mlp_bias_grad_workspace_floats(1 << 20, n)
        assert need <= cap or need == n, n  # a single chunk needs no partials


def test_rejects_shapes_beyond_the_array():
    L = binding.lib()
    P = ctypes.c_void_p(0x10000)
    assert L.tp_mlp_bias_grad_workspace_floats(4096, 32776) > L.tp_mlp_bias_grad_noalloc_max_floats()
    assert L.tp_mlp_bias_grad_noalloc(P, 4096, 32776, P, None) == binding.TPMLP_ERR_WORKSPACE


CASES = [
    (2048, 20480, 1003),  # dY of the MT-NLG 530B block (two row chunks)
    (8192, 1024, 1001),   # dY of the GPT-2-medium block (many row chunks)
    (300, 200, 11),       # ragged columns and rows
]


@pytest.mark.gpu
@pytest.mark.parametrize("T,n,seed", CASES)
def test_matches_allocating_entry_point_twice(T, n, seed):
    w = inputs.custom(T=T, h=n, F=8 * ((n + 7) // 8), t=1, seed=seed)
    G = inputs.make_inputs(w, keys=("dY",))["dY"].cuda()
    ref = binding.tp_mlp_bias_grad(G)
    first = binding.tp_mlp_bias_grad_noalloc(G)
    # a second call in a row on the same shared array, into a fresh output
    second = binding.tp_mlp_bias_grad_noalloc(G, db=torch.full_like(ref, float("nan")))
    torch.cuda.synchronize()
    assert binding.device_status() == binding.TPMLP_OK
    assert _rel(first, ref) <= TOL
    assert _rel(second, ref) <= TOL
    # the same kernels add in the same order whichever memory holds the
    # partial sums, so the results agree bit for bit: a partial row or a
    # completion count left over from an earlier call would show here
    assert torch.equal(first, ref)
    assert torch.equal(second, ref)


@pytest.mark.gpu
def test_empty_batch_gives_zeros():
    G = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    db = binding.tp_mlp_bias_grad_noalloc(G, db=torch.ones(64, device="cuda"))
    torch.cuda.synchronize()
    assert float(db.abs().max()) == 0.0
