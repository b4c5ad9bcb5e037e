"""Column sums (the bias gradients db2, dbo, dbqkv) against the oracle.

db[j] = sum_r G[r, j] is computed in fp32 from bf16 G: per thread over its
rows in order, then across lanes, warps and row chunks.  Every partial sum
is bounded by sum_r |G[r, j]|, so after at most `depth` additions the
error is at most depth * 2^-24 * sum_r |G[r, j]| -- the bound each column
is held to here.  depth counts the thread's rows (T / 32), the shuffle,
warp and chunk levels (at most 700 with the 640-CTA target).

The shapes cross the kernel's boundaries: fewer rows than one 32-row step,
one 256-row batch and a ragged one, a single row chunk (db written
directly) and many, column counts that leave a 64-column block partly
empty.
"""

import numpy as np
import pytest
import torch

import oracle
from tensor_transformer_mlp_forward_gb300 import binding, inputs

CASES = [
    (1, 8, 1),
    (31, 64, 2),
    (33, 72, 3),
    (255, 136, 4),
    (257, 520, 5),
    (1000, 1000, 6),
    (4099, 2056, 7),
    (8192, 1024, 8),
]


def _g(T, n, seed):
    w = inputs.custom(T=T, h=n, F=8, t=1, seed=seed)
    return inputs.make_inputs(w, keys=("dY",))["dY"]


def test_oracle_column_sum_closed_form():
    """The oracle's fp64 sum of bf16 values is exact to 2^-52 relative:
    its sum of a column of equal values is that value times T."""
    T, n = 4099, 16
    G = torch.full((T, n), 0.375, dtype=torch.bfloat16)
    assert np.array_equal(oracle.db2(G), np.full(n, 0.375 * T))


@pytest.mark.gpu
@pytest.mark.parametrize("T,n,seed", CASES)
def test_column_sums_within_fp32_bound(T, n, seed):
    cpu = _g(T, n, seed)
    ref = oracle.db2(cpu)
    mag = oracle.db2(cpu.abs())
    db = binding.tp_mlp_bias_grad(cpu.cuda())
    again = binding.tp_mlp_bias_grad(cpu.cuda())
    torch.cuda.synchronize()
    assert binding.device_status() == binding.TPMLP_OK
    got = db.cpu().double().numpy()
    depth = T // 32 + 700
    bound = depth * 2.0 ** -24 * mag + 1e-30
    worst = float(np.max(np.abs(got - ref) / bound))
    assert worst <= 1.0, (T, n, worst)
    assert torch.equal(db, again)  # a fixed order of additions
