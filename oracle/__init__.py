"""fp64 CPU oracle of the tensor-parallel Transformer MLP block.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg import this package.  It shares no
code with the CUDA path: the arithmetic lives in ``tpmlp_oracle.c`` (plain
loops, double precision, inputs widened exactly from bfloat16) and this
module only converts tensors and calls it.

Definitions followed (see the C source for the formulas): "Megatron-LM:
Tensor Model Parallel" (charles2530.github.io), section "MLP: Column
Parallel first, then Row Parallel" (Figure 3a) and section "f / g Operators"
(Figure 4); GeLU is the tanh approximation (the pages name GeLU without
defining it).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force against float64 numpy matmul, GeLU closed forms and values,
finite differences, the shard-partition invariant, special cases); the pages
print no worked numeric example, so no value here is pinned to the pages'
own numbers.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import attn_rows as _attn_rows
from . import build as _build

class Oracle:
    """Calls into one build of the oracle library (the default one, or a
    mutated copy that the tests compile to check that the pins bite)."""

    def __init__(self, path: str | None = None, attn_rows_impl=None):
        self._attn_rows = attn_rows_impl or _attn_rows.attn_rows
        L = ctypes.CDLL(path or _build.build())
        dp = ctypes.POINTER(ctypes.c_double)
        up = ctypes.POINTER(ctypes.c_uint16)
        lp = ctypes.POINTER(ctypes.c_long)
        cl = ctypes.c_long
        L.orc_gelu.argtypes = [ctypes.c_double]
        L.orc_gelu.restype = ctypes.c_double
        L.orc_gelu_grad.argtypes = [ctypes.c_double]
        L.orc_gelu_grad.restype = ctypes.c_double
        L.orc_forward.argtypes = [dp] * 6 + [cl] * 4 + [dp] * 3
        L.orc_backward.argtypes = [dp] * 5 + [cl] * 4 + [dp] * 5
        L.orc_forward_rows_bf16.argtypes = [up] * 6 + [cl] * 4 + [lp, cl] + [dp] * 3
        L.orc_backward_rows_bf16.argtypes = [up] * 5 + [cl] * 4 + [lp, cl, dp]
        L.orc_backward_cols_bf16.argtypes = [up] * 5 + [cl] * 4 + [lp, cl] + [dp] * 3
        L.orc_db2_bf16.argtypes = [up, cl, cl, dp]
        L.orc_ln_forward.argtypes = [dp] * 4 + [cl, cl, ctypes.c_double] + [dp] * 4
        L.orc_ln_backward.argtypes = [dp] * 5 + [cl, cl, ctypes.c_double] + [dp] * 3
        u32p = ctypes.POINTER(ctypes.c_uint32)
        u64 = ctypes.c_uint64
        L.orc_philox4x32_10.argtypes = [u32p, u32p, u32p]
        L.orc_philox4x32_10.restype = None
        L.orc_dropout_mask.argtypes = [u64, u64, cl, ctypes.c_double, ctypes.POINTER(ctypes.c_uint8)]
        L.orc_forward_dropout.argtypes = [dp] * 6 + [cl] * 4 + [ctypes.c_double, u64, u64] + [dp] * 3
        L.orc_backward_dropout.argtypes = [dp] * 5 + [cl] * 4 + [ctypes.c_double, u64, u64] + [dp] * 5
        L.orc_attn_forward.argtypes = [dp] * 6 + [cl] * 5 + [dp] * 3
        L.orc_attn_backward.argtypes = [dp] * 5 + [cl] * 5 + [dp] * 5
        L.orc_attn_head_bf16.argtypes = [up] * 3 + [cl] * 5 + [dp]
        L.orc_attn_head_grads_bf16.argtypes = [up] * 5 + [cl] * 5 + [dp] * 3
        for name in ("orc_dropout_mask", "orc_forward_dropout", "orc_backward_dropout"):
            getattr(L, name).restype = ctypes.c_int
        for name in ("orc_ln_forward", "orc_ln_backward", "orc_forward", "orc_backward", "orc_forward_rows_bf16",
                     "orc_backward_rows_bf16", "orc_backward_cols_bf16", "orc_db2_bf16",
                     "orc_num_threads"):
            getattr(L, name).restype = ctypes.c_int
        self.L = L

    def num_threads(self) -> int:
        return int(self.L.orc_num_threads())

    def gelu(self, x: float) -> float:
        return float(self.L.orc_gelu(float(x)))

    def gelu_grad(self, x: float) -> float:
        return float(self.L.orc_gelu_grad(float(x)))

    def forward(self, X, A, b1, B, b2, R, t: int):
        """Y, Z, H (float64 numpy) of the block with t shards."""
        X, A, b1, B, b2, R = (_f64(v) for v in (X, A, b1, B, b2, R))
        T, h = X.shape
        F = A.shape[1]
        Y = np.zeros((T, h))
        Z = np.zeros((T, F))
        H = np.zeros((T, F))
        _check(self.L.orc_forward(_dp(X), _dp(A), _dp(b1), _dp(B), _dp(b2), _dp(R), T, h, F, t,
                                  _dp(Y), _dp(Z), _dp(H)), "forward")
        return Y, Z, H

    def backward(self, dY, X, A, b1, B, t: int):
        """dX, dA, dB, db1, db2 (float64 numpy) of the block with t shards."""
        dY, X, A, b1, B = (_f64(v) for v in (dY, X, A, b1, B))
        T, h = X.shape
        F = A.shape[1]
        dX = np.zeros((T, h))
        dA = np.zeros((h, F))
        dB = np.zeros((F, h))
        db1 = np.zeros(F)
        db2 = np.zeros(h)
        _check(self.L.orc_backward(_dp(dY), _dp(X), _dp(A), _dp(b1), _dp(B), T, h, F, t,
                                   _dp(dX), _dp(dA), _dp(dB), _dp(db1), _dp(db2)), "backward")
        return dX, dA, dB, db1, db2

    def forward_rows(self, inp: dict, t: int, rows):
        """Y, Z, H restricted to the given token rows, from bf16 CPU tensors."""
        X, A, b1, B, b2, R = (_u16(inp[k]) for k in ("X", "A", "b1", "B", "b2", "residual"))
        T, h = inp["X"].shape
        F = inp["A"].shape[1]
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = len(rows)
        Y = np.zeros((n, h))
        Z = np.zeros((n, F))
        H = np.zeros((n, F))
        _check(self.L.orc_forward_rows_bf16(_up(X), _up(A), _up(b1), _up(B), _up(b2), _up(R),
                                            T, h, F, t, _lp(rows), n, _dp(Y), _dp(Z), _dp(H)),
               "forward_rows")
        return Y, Z, H

    def backward_rows(self, inp: dict, t: int, rows):
        """dX restricted to the given token rows, from bf16 CPU tensors."""
        dY, X, A, b1, B = (_u16(inp[k]) for k in ("dY", "X", "A", "b1", "B"))
        T, h = inp["X"].shape
        F = inp["A"].shape[1]
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = len(rows)
        dX = np.zeros((n, h))
        _check(self.L.orc_backward_rows_bf16(_up(dY), _up(X), _up(A), _up(b1), _up(B),
                                             T, h, F, t, _lp(rows), n, _dp(dX)), "backward_rows")
        return dX

    def backward_cols(self, inp: dict, t: int, cols):
        """dA[:, cols] ([h, n]), dB[cols, :] ([n, h]) and db1[cols] from bf16 CPU tensors."""
        dY, X, A, b1, B = (_u16(inp[k]) for k in ("dY", "X", "A", "b1", "B"))
        T, h = inp["X"].shape
        F = inp["A"].shape[1]
        cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
        n = len(cols)
        dA = np.zeros((h, n))
        dB = np.zeros((n, h))
        db1 = np.zeros(n)
        _check(self.L.orc_backward_cols_bf16(_up(dY), _up(X), _up(A), _up(b1), _up(B),
                                             T, h, F, t, _lp(cols), n, _dp(dA), _dp(dB),
                                             _dp(db1)), "backward_cols")
        return dA, dB, db1

    def ln_forward(self, a, r, gamma, beta, eps: float = 1e-5):
        """X, s, mean, rstd of the residual add + LayerNorm (float64 numpy)."""
        a, r, gamma, beta = (_f64(v) for v in (a, r, gamma, beta))
        T, h = a.shape
        X = np.zeros((T, h))
        s = np.zeros((T, h))
        mean = np.zeros(T)
        rstd = np.zeros(T)
        _check(self.L.orc_ln_forward(_dp(a), _dp(r), _dp(gamma), _dp(beta), T, h, eps, _dp(X),
                                     _dp(s), _dp(mean), _dp(rstd)), "ln_forward")
        return X, s, mean, rstd

    def ln_backward(self, dX, dres, a, r, gamma, eps: float = 1e-5):
        """ds, dgamma, dbeta of the residual add + LayerNorm (dres may be None)."""
        dX, a, r, gamma = (_f64(v) for v in (dX, a, r, gamma))
        T, h = a.shape
        dr = None if dres is None else _f64(dres)
        ds = np.zeros((T, h))
        dg = np.zeros(h)
        db = np.zeros(h)
        _check(self.L.orc_ln_backward(_dp(dX), None if dr is None else _dp(dr), _dp(a), _dp(r),
                                      _dp(gamma), T, h, eps, _dp(ds), _dp(dg), _dp(db)),
               "ln_backward")
        return ds, dg, db

    def philox4x32_10(self, counter, key):
        c = (ctypes.c_uint32 * 4)(*counter)
        k = (ctypes.c_uint32 * 2)(*key)
        out = (ctypes.c_uint32 * 4)()
        self.L.orc_philox4x32_10(c, k, out)
        return list(out)

    def dropout_mask(self, seed: int, offset: int, n: int, p: float) -> np.ndarray:
        keep = np.zeros(max(n, 1), dtype=np.uint8)
        _check(self.L.orc_dropout_mask(seed, offset, n, p,
                                       keep.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))),
               "dropout_mask")
        return keep[:n]

    def forward_dropout(self, X, A, b1, B, b2, R, t: int, p: float, seed: int, offset: int = 0):
        X, A, b1, B, b2, R = (_f64(v) for v in (X, A, b1, B, b2, R))
        T, h = X.shape
        F = A.shape[1]
        Y, Z, H = np.zeros((T, h)), np.zeros((T, F)), np.zeros((T, F))
        _check(self.L.orc_forward_dropout(_dp(X), _dp(A), _dp(b1), _dp(B), _dp(b2), _dp(R), T, h,
                                          F, t, p, seed, offset, _dp(Y), _dp(Z), _dp(H)),
               "forward_dropout")
        return Y, Z, H

    def backward_dropout(self, dY, X, A, b1, B, t: int, p: float, seed: int, offset: int = 0):
        dY, X, A, b1, B = (_f64(v) for v in (dY, X, A, b1, B))
        T, h = X.shape
        F = A.shape[1]
        dX, dA, dB = np.zeros((T, h)), np.zeros((h, F)), np.zeros((F, h))
        db1, db2 = np.zeros(F), np.zeros(h)
        _check(self.L.orc_backward_dropout(_dp(dY), _dp(X), _dp(A), _dp(b1), _dp(B), T, h, F, t, p,
                                           seed, offset, _dp(dX), _dp(dA), _dp(dB), _dp(db1),
                                           _dp(db2)), "backward_dropout")
        return dX, dA, dB, db1, db2

    # ------------------------------------------------ attention block

    def attn_forward(self, X, Wqkv, bqkv, Wo, bo, R, nb: int, nh: int, t: int):
        """Y, QKV, O of the head-parallel attention block (nb sequences)."""
        X, Wqkv, bqkv, Wo, bo, R = (_f64(v) for v in (X, Wqkv, bqkv, Wo, bo, R))
        T, h = X.shape
        s = T // nb if nb else 0
        Y, QKV, O = np.zeros((T, h)), np.zeros((T, 3 * h)), np.zeros((T, h))
        _check(self.L.orc_attn_forward(_dp(X), _dp(Wqkv), _dp(bqkv), _dp(Wo), _dp(bo), _dp(R),
                                       nb, max(s, 1), h, nh, t, _dp(Y), _dp(QKV), _dp(O)),
               "attn_forward")
        return Y, QKV, O

    def attn_backward(self, dY, X, Wqkv, bqkv, Wo, nb: int, nh: int, t: int):
        """dX, dWqkv, dbqkv, dWo, dbo of the attention block."""
        dY, X, Wqkv, bqkv, Wo = (_f64(v) for v in (dY, X, Wqkv, bqkv, Wo))
        T, h = X.shape
        s = T // nb if nb else 0
        dX, dWqkv, dbqkv = np.zeros((T, h)), np.zeros((h, 3 * h)), np.zeros(3 * h)
        dWo, dbo = np.zeros((h, h)), np.zeros(h)
        _check(self.L.orc_attn_backward(_dp(dY), _dp(X), _dp(Wqkv), _dp(bqkv), _dp(Wo), nb,
                                        max(s, 1), h, nh, t, _dp(dX), _dp(dWqkv), _dp(dbqkv),
                                        _dp(dWo), _dp(dbo)), "attn_backward")
        return dX, dWqkv, dbqkv, dWo, dbo

    def attn_head(self, inp: dict, nb: int, nh: int, j: int) -> np.ndarray:
        """Head j's attention output O_j [T, d] from bf16 CPU tensors."""
        X, Wqkv, bqkv = (_u16(inp[k]) for k in ("X", "Wqkv", "bqkv"))
        T, h = inp["X"].shape
        d = h // nh
        Oj = np.zeros((T, d))
        _check(self.L.orc_attn_head_bf16(_up(X), _up(Wqkv), _up(bqkv), nb, T // nb, h, nh, j,
                                         _dp(Oj)), "attn_head")
        return Oj

    def attn_head_grads(self, inp: dict, nb: int, nh: int, j: int):
        """Head j's dWqkv columns [h, 3d] (Q, K, V), dbqkv [3d], dWo rows [d, h]."""
        dY, X, Wqkv, bqkv, Wo = (_u16(inp[k]) for k in ("dY", "X", "Wqkv", "bqkv", "Wo"))
        T, h = inp["X"].shape
        d = h // nh
        dW, db, dWo = np.zeros((h, 3 * d)), np.zeros(3 * d), np.zeros((d, h))
        _check(self.L.orc_attn_head_grads_bf16(_up(dY), _up(X), _up(Wqkv), _up(bqkv), _up(Wo), nb,
                                               T // nb, h, nh, j, _dp(dW), _dp(db), _dp(dWo)),
               "attn_head_grads")
        return dW, db, dWo

    def attn_rows(self, inp: dict, nb: int, nh: int, t: int, rows):
        """Y[rows] and dX[rows] of the attention block from bf16 CPU tensors
        (the sampled-row evaluation in attn_rows.py)."""
        return self._attn_rows(inp, nb, nh, t, rows)

    def db2(self, dY) -> np.ndarray:
        """Column sums of dY from a bf16 CPU tensor."""
        T, h = dY.shape
        d = _u16(dY)
        out = np.zeros(h)
        _check(self.L.orc_db2_bf16(_up(d), T, h, _dp(out)), "db2")
        return out


def _f64(x) -> np.ndarray:
    """Exact widening to a contiguous float64 numpy array."""
    if isinstance(x, torch.Tensor):
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _u16(x: torch.Tensor) -> np.ndarray:
    """Raw bfloat16 bit patterns of a CPU tensor."""
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _up(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def _lp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_long))


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with status {rc}")


_default = None


def default() -> Oracle:
    """The oracle built from the committed source."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def gelu(x):
    return default().gelu(x)


def gelu_grad(x):
    return default().gelu_grad(x)


def forward(*a, **k):
    return default().forward(*a, **k)


def backward(*a, **k):
    return default().backward(*a, **k)


def forward_rows(*a, **k):
    return default().forward_rows(*a, **k)


def backward_rows(*a, **k):
    return default().backward_rows(*a, **k)


def backward_cols(*a, **k):
    return default().backward_cols(*a, **k)


def db2(dY):
    return default().db2(dY)


def philox4x32_10(counter, key):
    return default().philox4x32_10(counter, key)


def dropout_mask(*a, **k):
    return default().dropout_mask(*a, **k)


def forward_dropout(*a, **k):
    return default().forward_dropout(*a, **k)


def backward_dropout(*a, **k):
    return default().backward_dropout(*a, **k)


def attn_forward(*a, **k):
    return default().attn_forward(*a, **k)


def attn_backward(*a, **k):
    return default().attn_backward(*a, **k)


def attn_head(*a, **k):
    return default().attn_head(*a, **k)


def attn_head_grads(*a, **k):
    return default().attn_head_grads(*a, **k)


def attn_rows(*a, **k):
    return default().attn_rows(*a, **k)


def ln_forward(*a, **k):
    return default().ln_forward(*a, **k)


def ln_backward(*a, **k):
    return default().ln_backward(*a, **k)


def num_threads() -> int:
    return default().num_threads()
