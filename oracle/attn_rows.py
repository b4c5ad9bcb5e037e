"""Sampled token rows of the head-parallel attention block: Y and dX.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may use it.
It shares no code with the CUDA path.

The full-size blocks are too large for the plain-loop oracle to evaluate
whole, and a row of Y or dX depends on much more than that row: Y[r] needs
the keys and values of every earlier token of r's sequence, and dX[r] needs
the gradient reaching r's key and value from every later query of the
sequence.  So this evaluates, for each sequence that holds a sampled row,
the whole block on that sequence, and keeps the sampled rows.  The
projections are float64 numpy matmuls (a library primitive standing for one
step of the definition); everything else follows the definition as written,
in float64, from the exactly widened bf16 inputs.

Definition ("Megatron-LM: Tensor Model Parallel", section "Attention: split
Q/K/V by head", Figure 3b, with the f and g operators of section "f / g
Operators", Figure 4), for shard i of t owning heads i nh/t .. (i+1) nh/t - 1:

    QKV_i = X Wqkv_i + bqkv_i             (Wqkv_i: shard i's columns of Q, K, V)
    per sequence and head j of shard i:
        S = Q_j K_j^T / sqrt(d), causal (key k visible to query q iff k <= q)
        P = softmax of each row of S ; O_j = P V_j
    Y   = sum_i O_i Wo_i + bo + residual   (g: the shards' partials summed)

    dO_i = dY Wo_i^T
    per head: dP = dO_j V_j^T ; dS = P * (dP - rowsum(P * dP))
              dQ_j = dS K_j / sqrt(d) ; dK_j = dS^T Q_j / sqrt(d) ; dV_j = P^T dO_j
    dX  = sum_i dQKV_i Wqkv_i^T           (f: the shards' partials summed)

Parity status: pinned by ``tests/oracle_pins.py`` (pin_attn_rows_match_full:
equal to the full C oracle, itself pinned by library restatement, closed
forms, invariants and finite differences) and by planted mistakes in
``tests/test_oracle_pins.py``.
"""

from __future__ import annotations

import math

import numpy as np
import torch


def _f64(x: torch.Tensor) -> np.ndarray:
    """Exact widening of a bf16 (or wider) CPU tensor to float64."""
    return x.detach().to("cpu", torch.float64).numpy()


def attn_rows(inp: dict, nb: int, nh: int, t: int, rows):
    """Y[rows] and dX[rows] ([len(rows), h] float64 each) of the attention
    block over nb sequences with t shards, from bf16 CPU tensors X, Wqkv,
    bqkv, Wo, bo, residual, dY."""
    X, Wqkv, bqkv, Wo = inp["X"], inp["Wqkv"], inp["bqkv"], inp["Wo"]
    T, h = X.shape
    rows = np.asarray(rows, dtype=np.int64)
    if nb < 1 or T % nb or h % nh or nh % t:
        raise ValueError("attention shape")
    if rows.size and (rows.min() < 0 or rows.max() >= T):
        raise ValueError("row out of range")
    s, d, w, hs = T // nb, h // nh, h // t, nh // t
    scale = 1.0 / math.sqrt(d)
    Y = np.zeros((rows.size, h))
    dX = np.zeros((rows.size, h))
    causal = np.tril(np.ones((s, s), dtype=bool))
    for i in range(t):
        # shard i's columns of Q, K and V, in that order
        cols = np.concatenate([np.arange(p * h + i * w, p * h + (i + 1) * w) for p in range(3)])
        Wi = _f64(Wqkv[:, cols])
        bi = _f64(bqkv[cols])
        Woi = _f64(Wo[i * w:(i + 1) * w])
        for n in np.unique(rows // s):
            sel = np.nonzero(rows // s == n)[0]   # sampled rows in sequence n
            pos = rows[sel] - n * s                # their positions in it
            seq = slice(n * s, (n + 1) * s)
            qkv = _f64(X[seq]) @ Wi + bi           # [s, 3w]
            dO = _f64(inp["dY"][seq]) @ Woi.T      # [s, w]
            O = np.zeros((s, w))
            dqkv = np.zeros((sel.size, 3 * w))
            for jj in range(hs):
                c = slice(jj * d, (jj + 1) * d)
                ck = slice(w + jj * d, w + (jj + 1) * d)
                cv = slice(2 * w + jj * d, 2 * w + (jj + 1) * d)
                Q, K, V = qkv[:, c], qkv[:, ck], qkv[:, cv]
                S = np.where(causal, Q @ K.T * scale, -np.inf)
                E = np.exp(S - S.max(axis=1, keepdims=True))
                P = E / E.sum(axis=1, keepdims=True)
                O[:, c] = P @ V
                dOj = dO[:, c]
                dP = dOj @ V.T
                dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
                dqkv[:, c] = dS[pos] @ K * scale
                dqkv[:, ck] = dS[:, pos].T @ Q * scale
                dqkv[:, cv] = P[:, pos].T @ dOj
            Y[sel] += O[pos] @ Woi    # g: shard i's partial of the output projection
            dX[sel] += dqkv @ Wi.T    # f: shard i's partial of the input gradient
    Y += _f64(inp["bo"]) + _f64(inp["residual"][torch.as_tensor(rows)])
    return Y, dX
