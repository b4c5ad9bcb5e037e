"""Checks that pin the fp64 oracle to facts outside itself.

The pages print no worked numeric example of the MLP block, so the oracle is
pinned by mathematics:

* GeLU: exact identities of the tanh form (g(x) - g(-x) = x, g(0) = 0,
  g'(0) = 1/2, g'(x) + g'(-x) = 1), its asymptotes, its distance to the
  exact erf GeLU x Phi(x) (a different function whose maximum distance from
  the tanh approximation is 4.73e-4, reached near |x| = 2.7), and the
  derivative against central finite differences of the oracle's own GeLU.
* Linear algebra: the oracle's loops against numpy float64 matmuls (a
  library primitive), composed with the separately pinned GeLU.
* Gradients: against central finite differences of L = <dY, Y>.
* Partition invariant: every shard count t gives the unsharded block
  ("Megatron-LM: Tensor Model Parallel", section "MLP: Column Parallel first,
  then Row Parallel", Figure 3a; "f / g Operators", Figure 4).
* Special cases: A = 0, B = 0, X = 0, linearity in residual and b2.
* The sampled (bf16-input) entry points against the full computation.
* Residual add + LayerNorm: row statistics against numpy's mean and biased
  variance (mean 0, mean square var/(var+eps)), affinity in gamma/beta,
  invariance to a per-row shift and (as eps -> 0) to scale, and every
  gradient against central differences.
* Dropout: the published Philox4x32-10 known-answer vectors, drop rates
  within binomial bounds, the counter/seed semantics, p = 0 equal to the
  plain block, and the gradients against central differences.

Each check returns True/False so that ``test_oracle_pins.py`` can run the same
list against deliberately mutated copies of the oracle and show that every
planted mistake fails at least one check.
"""

from __future__ import annotations

import math

import numpy as np
import torch

from tensor_transformer_mlp_forward_gb300 import inputs

ERF_GAP = 4.74e-4  # max |tanh-GeLU - erf-GeLU| over the reals (measured on a fine grid)


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.max(np.abs(b)) if b.size else 0.0
    if den == 0.0:
        return float(np.max(np.abs(a - b))) if a.size else 0.0
    return float(np.max(np.abs(a - b)) / den)


def _rand_block(T, h, F, seed, scale_w=0.3):
    rng = np.random.default_rng(seed)
    return dict(
        X=rng.standard_normal((T, h)),
        A=rng.standard_normal((h, F)) * scale_w,
        b1=rng.standard_normal(F) * 0.1,
        B=rng.standard_normal((F, h)) * scale_w,
        b2=rng.standard_normal(h) * 0.1,
        R=rng.standard_normal((T, h)),
        dY=rng.standard_normal((T, h)),
    )


# ----------------------------------------------------------------- GeLU pins

def pin_gelu_identities(o) -> bool:
    ok = o.gelu(0.0) == 0.0 and o.gelu_grad(0.0) == 0.5
    for x in np.linspace(-6, 6, 241):
        ok &= abs((o.gelu(x) - o.gelu(-x)) - x) <= 1e-14 * max(1.0, abs(x))
        ok &= abs(o.gelu_grad(x) + o.gelu_grad(-x) - 1.0) <= 1e-14
    return bool(ok)


def pin_gelu_asymptotes(o) -> bool:
    return (abs(o.gelu(12.0) - 12.0) < 1e-12 and abs(o.gelu(-12.0)) < 1e-12
            and abs(o.gelu_grad(12.0) - 1.0) < 1e-12 and abs(o.gelu_grad(-12.0)) < 1e-12)


def pin_gelu_vs_erf(o) -> bool:
    worst = 0.0
    for x in np.linspace(-8, 8, 3201):
        exact = 0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0)))
        worst = max(worst, abs(o.gelu(x) - exact))
    # the approximation is close to, but not equal to, the erf form
    return 4.0e-4 < worst <= ERF_GAP


def pin_gelu_known_values(o) -> bool:
    # tanh-approximation GeLU at +-1 and 3, seven significant digits
    return (abs(o.gelu(1.0) - 0.8411920) < 5e-8 and abs(o.gelu(-1.0) + 0.1588080) < 5e-8
            and abs(o.gelu(3.0) - 2.9963626) < 5e-8)


def pin_gelu_grad_fd(o) -> bool:
    eps = 1e-5
    for x in np.linspace(-5, 5, 101):
        fd = (o.gelu(x + eps) - o.gelu(x - eps)) / (2 * eps)
        if abs(fd - o.gelu_grad(x)) > 1e-8:
            return False
    return True


# ------------------------------------------------------- linear algebra pins

def _np_forward(o, p):
    g = np.vectorize(o.gelu, otypes=[np.float64])
    Z = p["X"] @ p["A"] + p["b1"]
    H = g(Z)
    return H @ p["B"] + p["b2"] + p["R"], Z, H


def _np_backward(o, p):
    g = np.vectorize(o.gelu, otypes=[np.float64])
    gd = np.vectorize(o.gelu_grad, otypes=[np.float64])
    Z = p["X"] @ p["A"] + p["b1"]
    H = g(Z)
    dZ = (p["dY"] @ p["B"].T) * gd(Z)
    return dZ @ p["A"].T, p["X"].T @ dZ, H.T @ p["dY"], dZ.sum(0), p["dY"].sum(0)


def pin_forward_vs_numpy(o) -> bool:
    for (T, h, F, t, seed) in ((5, 6, 8, 1, 1), (7, 4, 12, 3, 2), (1, 3, 8, 4, 3), (0, 3, 4, 2, 4)):
        p = _rand_block(T, h, F, seed)
        Y, Z, H = o.forward(p["X"], p["A"], p["b1"], p["B"], p["b2"], p["R"], t)
        Yn, Zn, Hn = _np_forward(o, p)
        if T and (_rel(Y, Yn) > 1e-12 or _rel(Z, Zn) > 1e-12 or _rel(H, Hn) > 1e-12):
            return False
        if Y.shape != (T, h):
            return False
    return True


def pin_backward_vs_numpy(o) -> bool:
    for (T, h, F, t, seed) in ((5, 6, 8, 1, 5), (7, 4, 12, 3, 6), (2, 5, 8, 8, 7)):
        p = _rand_block(T, h, F, seed)
        got = o.backward(p["dY"], p["X"], p["A"], p["b1"], p["B"], t)
        ref = _np_backward(o, p)
        for a, b in zip(got, ref):
            if _rel(a, b) > 1e-12:
                return False
    return True


# ---------------------------------------------------------- gradient pins

def pin_gradients_fd(o) -> bool:
    """Every gradient against central differences of L = <dY, Y>."""
    T, h, F, t = 3, 4, 8, 2
    p = _rand_block(T, h, F, 11, scale_w=0.5)

    def loss(q):
        Y, _, _ = o.forward(q["X"], q["A"], q["b1"], q["B"], q["b2"], q["R"], t)
        return float(np.sum(q["dY"] * Y))

    dX, dA, dB, db1, db2 = o.backward(p["dY"], p["X"], p["A"], p["b1"], p["B"], t)
    eps = 1e-6
    for key, an in (("X", dX), ("A", dA), ("B", dB), ("b1", db1), ("b2", db2), ("R", p["dY"])):
        fd = np.zeros_like(p[key])
        it = np.nditer(p[key], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            q = {k: v.copy() for k, v in p.items()}
            q[key][idx] += eps
            lp = loss(q)
            q[key][idx] -= 2 * eps
            lm = loss(q)
            fd[idx] = (lp - lm) / (2 * eps)
        if _rel(an, fd) > 1e-6:
            return False
    return True


# ------------------------------------------------------ partition invariant

def pin_partition_invariant(o) -> bool:
    T, h, F = 6, 8, 64
    p = _rand_block(T, h, F, 21)
    base_f = o.forward(p["X"], p["A"], p["b1"], p["B"], p["b2"], p["R"], 1)
    base_b = o.backward(p["dY"], p["X"], p["A"], p["b1"], p["B"], 1)
    for t in (2, 4, 8):
        f = o.forward(p["X"], p["A"], p["b1"], p["B"], p["b2"], p["R"], t)
        b = o.backward(p["dY"], p["X"], p["A"], p["b1"], p["B"], t)
        for a, c in zip(f + b, base_f + base_b):
            if _rel(a, c) > 1e-12:
                return False
    return True


# ------------------------------------------------------------ special cases

def pin_special_cases(o) -> bool:
    T, h, F, t = 4, 6, 16, 4
    p = _rand_block(T, h, F, 31)
    ok = True
    # A = 0: Y = GeLU(b1) B + b2 + R in every row, dX = 0
    q = dict(p, A=np.zeros_like(p["A"]))
    Y, _, _ = o.forward(q["X"], q["A"], q["b1"], q["B"], q["b2"], q["R"], t)
    row = np.array([o.gelu(v) for v in q["b1"]]) @ q["B"] + q["b2"]
    ok &= _rel(Y - q["R"], np.tile(row, (T, 1))) < 1e-12
    dX, *_ = o.backward(q["dY"], q["X"], q["A"], q["b1"], q["B"], t)
    ok &= float(np.max(np.abs(dX))) == 0.0
    # B = 0: Y = b2 + R, dA = 0, db1 = 0
    q = dict(p, B=np.zeros_like(p["B"]))
    Y, _, _ = o.forward(q["X"], q["A"], q["b1"], q["B"], q["b2"], q["R"], t)
    ok &= _rel(Y, q["b2"] + q["R"]) < 1e-15
    _, dA, _, db1, _ = o.backward(q["dY"], q["X"], q["A"], q["b1"], q["B"], t)
    ok &= float(np.max(np.abs(dA))) == 0.0 and float(np.max(np.abs(db1))) == 0.0
    # X = 0: dA = 0
    q = dict(p, X=np.zeros_like(p["X"]))
    _, dA, _, _, _ = o.backward(q["dY"], q["X"], q["A"], q["b1"], q["B"], t)
    ok &= float(np.max(np.abs(dA))) == 0.0
    # Y is affine in the residual and in b2 with unit slope
    Y0, _, _ = o.forward(p["X"], p["A"], p["b1"], p["B"], p["b2"], p["R"], t)
    Y1, _, _ = o.forward(p["X"], p["A"], p["b1"], p["B"], p["b2"] + 1.5, 2 * p["R"], t)
    ok &= _rel(Y1 - Y0, p["R"] + 1.5) < 1e-12
    # dY = 0: every gradient vanishes
    g = o.backward(np.zeros_like(p["dY"]), p["X"], p["A"], p["b1"], p["B"], t)
    ok &= all(float(np.max(np.abs(v))) == 0.0 for v in g)
    return bool(ok)


# --------------------------------------------------- sampled vs full (bf16)

def pin_sampled_matches_full(o) -> bool:
    w = inputs.custom(T=37, h=24, F=48, t=4, seed=77)
    inp = inputs.make_inputs(w)
    Y, Z, H = o.forward(inp["X"], inp["A"], inp["b1"], inp["B"], inp["b2"], inp["residual"], w.t)
    dX, dA, dB, db1, db2 = o.backward(inp["dY"], inp["X"], inp["A"], inp["b1"], inp["B"], w.t)
    rows = [0, 5, 36]
    cols = [0, 11, 12, 47]
    Yr, Zr, Hr = o.forward_rows(inp, w.t, rows)
    dXr = o.backward_rows(inp, w.t, rows)
    dAc, dBr, db1c = o.backward_cols(inp, w.t, cols)
    d2 = o.db2(inp["dY"])
    return (_rel(Yr, Y[rows]) < 1e-13 and _rel(Zr, Z[rows]) < 1e-13 and _rel(Hr, H[rows]) < 1e-13
            and _rel(dXr, dX[rows]) < 1e-13 and _rel(dAc, dA[:, cols]) < 1e-13
            and _rel(dBr, dB[cols]) < 1e-13 and _rel(db1c, db1[cols]) < 1e-13
            and _rel(d2, db2) < 1e-13)


# ------------------------------------------------- residual add + LayerNorm

def _ln_inputs(T, h, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((T, h)) * 1.5 + 0.3, rng.standard_normal((T, h)),
            1.0 + 0.2 * rng.standard_normal(h), 0.1 * rng.standard_normal(h))


def pin_ln_normalizes(o) -> bool:
    """gamma = 1, beta = 0: every row of X has mean 0 and mean square
    var / (var + eps) with the biased variance of s = input + residual."""
    a, r, _, _ = _ln_inputs(5, 24, 41)
    eps = 0.37  # large, so that its placement shows
    X, s, mean, rstd = o.ln_forward(a, r, np.ones(24), np.zeros(24), eps)
    su = a + r
    var = su.var(axis=1)  # numpy's biased variance: a library primitive
    return (_rel(s, su) == 0.0 and float(np.max(np.abs(X.mean(axis=1)))) < 1e-14
            and _rel((X * X).mean(axis=1), var / (var + eps)) < 1e-13
            and _rel(mean, su.mean(axis=1)) < 1e-14)


def pin_ln_affine_and_invariant(o) -> bool:
    a, r, g, b = _ln_inputs(4, 16, 42)
    X0, _, _, _ = o.ln_forward(a, r, np.ones(16), np.zeros(16))
    X1, _, _, _ = o.ln_forward(a, r, g, b)
    ok = _rel(X1, X0 * g + b) < 1e-14
    shift = np.arange(4.0)[:, None] * 3.0  # a per-row constant moves mu, not X
    X2, _, _, _ = o.ln_forward(a + shift, r, g, b)
    ok &= _rel(X2, X1) < 1e-12
    Xs, _, _, _ = o.ln_forward(7.0 * a, 7.0 * r, g, b, 1e-14)  # scale-free as eps -> 0
    Xt, _, _, _ = o.ln_forward(a, r, g, b, 1e-14)
    return bool(ok and _rel(Xs, Xt) < 1e-9)


def pin_ln_gradients_fd(o) -> bool:
    """ds, dgamma, dbeta against central differences of
    L = <dX, X> + <dres, s>; d(input) = d(residual) = ds."""
    T, h, eps = 3, 6, 1e-3
    a, r, g, b = _ln_inputs(T, h, 43)
    rng = np.random.default_rng(44)
    dX, dres = rng.standard_normal((T, h)), rng.standard_normal((T, h))
    p = dict(a=a, r=r, g=g, b=b)

    def loss(q):
        X, s, _, _ = o.ln_forward(q["a"], q["r"], q["g"], q["b"], eps)
        return float(np.sum(dX * X) + np.sum(dres * s))

    ds, dg, db = o.ln_backward(dX, dres, a, r, g, eps)
    step = 1e-6
    for key, an in (("a", ds), ("r", ds), ("g", dg), ("b", db)):
        fd = np.zeros_like(p[key])
        it = np.nditer(p[key], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            q = {k: v.copy() for k, v in p.items()}
            q[key][idx] += step
            lp = loss(q)
            q[key][idx] -= 2 * step
            fd[idx] = (lp - loss(q)) / (2 * step)
        if _rel(an, fd) > 1e-6:
            return False
    # without the residual-path gradient each row of ds sums to zero
    ds0, _, _ = o.ln_backward(dX, None, a, r, g, eps)
    return float(np.max(np.abs(ds0.sum(axis=1)))) < 1e-12


# -------------------------------------------------------------- dropout

def pin_philox_known_answers(o) -> bool:
    """The published Philox4x32-10 known-answer vectors
    (tests/golden/philox4x32_10_kat.txt)."""
    import os

    path = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")
    n = 0
    for line in open(path):
        if not line.strip() or line.startswith("#"):
            continue
        words = [int(x, 16) for x in line.split()]
        if o.philox4x32_10(words[0:4], words[4:6]) != words[6:10]:
            return False
        n += 1
    return n == 3


def pin_dropout_mask(o) -> bool:
    n = 200000
    ok = True
    for p in (0.1, 0.5):
        keep = o.dropout_mask(99, 7, n, p)
        drop = 1.0 - keep.mean()
        ok &= abs(drop - p) < 6.0 * math.sqrt(p * (1 - p) / n)
    ok &= bool(o.dropout_mask(99, 7, 1000, 0.0).all())
    # seed 0, offset 0: element e reads word e of the first known-answer
    # block (6627e8d5 e169c58d bc57ac4c 9b00dbd8); at p = 1/2 the first is
    # below 2^31 (dropped), the other three above (kept)
    ok &= o.dropout_mask(0, 0, 4, 0.5).tolist() == [0, 1, 1, 1]
    a = o.dropout_mask(99, 0, 4096, 0.5)
    ok &= bool((a[5:] == o.dropout_mask(99, 5, 4091, 0.5)).all())  # the counter is offset + e
    ok &= bool((a != o.dropout_mask(100, 0, 4096, 0.5)).any())      # the seed matters
    return bool(ok)


def pin_dropout_forward(o) -> bool:
    T, h, F, t, p = 6, 16, 32, 2, 0.25
    q = _rand_block(T, h, F, 51)
    Y0, _, _ = o.forward(q["X"], q["A"], q["b1"], q["B"], q["b2"], q["R"], t)
    Yp0, _, _ = o.forward_dropout(q["X"], q["A"], q["b1"], q["B"], q["b2"], q["R"], t, 0.0, 5)
    Yd, _, _ = o.forward_dropout(q["X"], q["A"], q["b1"], q["B"], q["b2"], q["R"], t, p, 5, 3)
    keep = o.dropout_mask(5, 3, T * h, p).reshape(T, h)
    expect = q["R"] + keep * (Y0 - q["R"]) / (1.0 - p)
    return _rel(Yp0, Y0) < 1e-13 and _rel(Yd, expect) < 1e-12


def pin_dropout_backward_fd(o) -> bool:
    """Gradients with dropout against central differences of <dY, Y>; the
    mask depends only on (seed, offset, position), so it stays fixed."""
    T, h, F, t, p = 3, 4, 8, 2, 0.3
    q = _rand_block(T, h, F, 52, scale_w=0.5)

    def loss(v):
        Y, _, _ = o.forward_dropout(v["X"], v["A"], v["b1"], v["B"], v["b2"], v["R"], t, p, 11)
        return float(np.sum(q["dY"] * Y))

    grads = o.backward_dropout(q["dY"], q["X"], q["A"], q["b1"], q["B"], t, p, 11)
    eps = 1e-6
    for key, an in zip(("X", "A", "B", "b1", "b2"), grads):
        fd = np.zeros_like(q[key])
        it = np.nditer(q[key], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            v = {k: w.copy() for k, w in q.items()}
            v[key][idx] += eps
            lp = loss(v)
            v[key][idx] -= 2 * eps
            fd[idx] = (lp - loss(v)) / (2 * eps)
        if _rel(an, fd) > 1e-6:
            return False
    return True


# ------------------------------------------------------------ attention

def _attn_inputs(nb, s, h, seed, scale_w=0.4):
    rng = np.random.default_rng(seed)
    return dict(X=rng.standard_normal((nb * s, h)),
                Wqkv=scale_w * rng.standard_normal((h, 3 * h)),
                bqkv=0.1 * rng.standard_normal(3 * h),
                Wo=scale_w * rng.standard_normal((h, h)),
                bo=0.1 * rng.standard_normal(h),
                R=rng.standard_normal((nb * s, h)),
                dY=rng.standard_normal((nb * s, h)))


def _attn_library(p, nb, nh):
    """The block from numpy float64 matmuls and scipy's softmax over each
    row's causal prefix: library routines composed by the definition."""
    from scipy.special import softmax

    T, h = p["X"].shape
    s, d = T // nb, h // nh
    QKV = p["X"] @ p["Wqkv"] + p["bqkv"]
    O = np.zeros((T, h))
    for n in range(nb):
        rows = slice(n * s, (n + 1) * s)
        for j in range(nh):
            q = QKV[rows, j * d:(j + 1) * d]
            k = QKV[rows, h + j * d:h + (j + 1) * d]
            v = QKV[rows, 2 * h + j * d:2 * h + (j + 1) * d]
            S = q @ k.T / math.sqrt(d)
            for r in range(s):
                pr = softmax(S[r, :r + 1])
                O[n * s + r, j * d:(j + 1) * d] = pr @ v[:r + 1]
    return O @ p["Wo"] + p["bo"] + p["R"], QKV, O


def pin_attn_vs_library(o) -> bool:
    ok = True
    for nb, s, h, nh, t in ((2, 5, 8, 2, 2), (1, 7, 12, 3, 3), (3, 1, 4, 1, 1), (0, 4, 8, 2, 1)):
        p = _attn_inputs(nb, s, h, 60 + s)
        Y, QKV, O = o.attn_forward(p["X"], p["Wqkv"], p["bqkv"], p["Wo"], p["bo"], p["R"], nb, nh, t)
        Yl, QKVl, Ol = _attn_library(p, nb, nh) if nb else (np.zeros((0, h)),) * 3
        ok &= _rel(Y, Yl) < 1e-12 and _rel(O, Ol) < 1e-12 and _rel(QKV, QKVl) < 1e-12
    return bool(ok)


def pin_attn_closed_forms(o) -> bool:
    """One token per sequence: each row attends only to itself, so
    O = V = X Wv + bv.  Zero query weights: every score is 0 and each row
    averages the values of its prefix (a running mean)."""
    nb, s, h, nh = 3, 1, 8, 2
    p = _attn_inputs(nb, s, h, 71)
    Y, _, O = o.attn_forward(p["X"], p["Wqkv"], p["bqkv"], p["Wo"], p["bo"], p["R"], nb, nh, 2)
    V = p["X"] @ p["Wqkv"][:, 2 * h:] + p["bqkv"][2 * h:]
    ok = _rel(O, V) < 1e-13 and _rel(Y, V @ p["Wo"] + p["bo"] + p["R"]) < 1e-13
    nb, s = 2, 6
    p = _attn_inputs(nb, s, h, 72)
    p["Wqkv"][:, :h] = 0.0
    p["bqkv"][:h] = 0.0
    _, QKV, O = o.attn_forward(p["X"], p["Wqkv"], p["bqkv"], p["Wo"], p["bo"], p["R"], nb, nh, 1)
    V = QKV[:, 2 * h:].reshape(nb, s, h)
    mean = np.cumsum(V, axis=1) / np.arange(1, s + 1)[None, :, None]
    return bool(ok and _rel(O, mean.reshape(nb * s, h)) < 1e-13)


def pin_attn_invariants(o) -> bool:
    """Causality, independence of the sequences, and the key bias: adding
    the same vector to every key shifts each score row by a constant, which
    softmax ignores, so Y and the other gradients do not see bk and its
    gradient vanishes."""
    nb, s, h, nh = 2, 5, 8, 2
    p = _attn_inputs(nb, s, h, 73)
    args = lambda q: (q["X"], q["Wqkv"], q["bqkv"], q["Wo"], q["bo"], q["R"], nb, nh, 2)  # noqa: E731
    Y0, _, _ = o.attn_forward(*args(p))
    q = {k: v.copy() for k, v in p.items()}
    q["X"][3:5] += 1.7             # tokens 3, 4 of sequence 0 and nothing else
    Y1, _, _ = o.attn_forward(*args(q))
    ok = np.array_equal(Y0[:3], Y1[:3]) and np.array_equal(Y0[5:], Y1[5:]) and not np.allclose(Y0[3:5], Y1[3:5])
    q = {k: v.copy() for k, v in p.items()}
    q["bqkv"][h:2 * h] += 0.9      # the key bias
    Y2, _, _ = o.attn_forward(*args(q))
    ok &= _rel(Y2, Y0) < 1e-13
    g = o.attn_backward(p["dY"], p["X"], p["Wqkv"], p["bqkv"], p["Wo"], nb, nh, 2)
    ok &= float(np.max(np.abs(g[2][h:2 * h]))) < 1e-12 * max(1.0, float(np.max(np.abs(g[2]))))
    return bool(ok)


def pin_attn_partition_invariant(o) -> bool:
    nb, s, h, nh = 2, 4, 16, 4
    p = _attn_inputs(nb, s, h, 74)
    base = None
    for t in (1, 2, 4):
        out = o.attn_forward(p["X"], p["Wqkv"], p["bqkv"], p["Wo"], p["bo"], p["R"], nb, nh, t)[:1] + \
            o.attn_backward(p["dY"], p["X"], p["Wqkv"], p["bqkv"], p["Wo"], nb, nh, t)
        if base is None:
            base = out
        elif not all(_rel(a, b) < 1e-12 for a, b in zip(out, base)):
            return False
    return True


def pin_attn_gradients_fd(o) -> bool:
    """dX, dWqkv, dbqkv, dWo, dbo against central differences of <dY, Y>."""
    nb, s, h, nh, t = 2, 3, 4, 2, 2
    p = _attn_inputs(nb, s, h, 75)

    def loss(q):
        Y, _, _ = o.attn_forward(q["X"], q["Wqkv"], q["bqkv"], q["Wo"], q["bo"], q["R"], nb, nh, t)
        return float(np.sum(p["dY"] * Y))

    grads = o.attn_backward(p["dY"], p["X"], p["Wqkv"], p["bqkv"], p["Wo"], nb, nh, t)
    eps = 1e-6
    for key, an in zip(("X", "Wqkv", "bqkv", "Wo", "bo"), grads):
        fd = np.zeros_like(p[key])
        it = np.nditer(p[key], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            q = {k: v.copy() for k, v in p.items()}
            q[key][idx] += eps
            lp = loss(q)
            q[key][idx] -= 2 * eps
            fd[idx] = (lp - loss(q)) / (2 * eps)
        if _rel(an, fd) > 1e-6:
            return False
    return True


def pin_attn_sampled_matches_full(o) -> bool:
    """The per-head entry points (bf16 inputs) against the full block."""
    nb, s, h, nh, t = 2, 6, 16, 4, 2
    rng = np.random.default_rng(76)
    bf = lambda *sh: torch.from_numpy(0.5 * rng.standard_normal(sh)).to(torch.bfloat16)  # noqa: E731
    inp = dict(X=bf(nb * s, h), Wqkv=bf(h, 3 * h), bqkv=bf(3 * h), Wo=bf(h, h), bo=bf(h),
               R=bf(nb * s, h), dY=bf(nb * s, h))
    f = {k: v.double().numpy() for k, v in inp.items()}
    _, _, O = o.attn_forward(f["X"], f["Wqkv"], f["bqkv"], f["Wo"], f["bo"], f["R"], nb, nh, t)
    dX, dW, db, dWo, dbo = o.attn_backward(f["dY"], f["X"], f["Wqkv"], f["bqkv"], f["Wo"], nb, nh, t)
    d = h // nh
    ok = True
    for j in range(nh):
        cols = np.r_[j * d:(j + 1) * d, h + j * d:h + (j + 1) * d, 2 * h + j * d:2 * h + (j + 1) * d]
        ok &= _rel(o.attn_head(inp, nb, nh, j), O[:, j * d:(j + 1) * d]) < 1e-13
        gW, gb, gWo = o.attn_head_grads(inp, nb, nh, j)
        ok &= _rel(gW, dW[:, cols]) < 1e-12 and _rel(gb, db[cols]) < 1e-12
        ok &= _rel(gWo, dWo[j * d:(j + 1) * d]) < 1e-12
    return bool(ok)


def pin_attn_rows_match_full(o) -> bool:
    """Sampled rows of Y and dX (bf16 inputs, several sequences, shards and
    heads, rows early and late in their sequences) against the full block."""
    rng = np.random.default_rng(77)
    ok = True
    for nb, s, h, nh, t, rows in ((2, 6, 16, 4, 2, [0, 5, 6, 11]), (3, 9, 24, 6, 3, [4, 17, 26]),
                                  (1, 7, 8, 1, 1, [6]), (2, 5, 12, 3, 1, [])):
        bf = lambda *sh: torch.from_numpy(0.5 * rng.standard_normal(sh)).to(torch.bfloat16)  # noqa: E731
        inp = dict(X=bf(nb * s, h), Wqkv=bf(h, 3 * h), bqkv=bf(3 * h), Wo=bf(h, h), bo=bf(h),
                   residual=bf(nb * s, h), dY=bf(nb * s, h))
        f = {k: v.double().numpy() for k, v in inp.items()}
        Y, _, _ = o.attn_forward(f["X"], f["Wqkv"], f["bqkv"], f["Wo"], f["bo"], f["residual"],
                                 nb, nh, t)
        dX = o.attn_backward(f["dY"], f["X"], f["Wqkv"], f["bqkv"], f["Wo"], nb, nh, t)[0]
        Yr, dXr = o.attn_rows(inp, nb, nh, t, rows)
        ok &= Yr.shape == (len(rows), h) and dXr.shape == (len(rows), h)
        if rows:
            ok &= _rel(Yr, Y[rows]) < 1e-12 and _rel(dXr, dX[rows]) < 1e-12
    return bool(ok)


ALL_PINS = [
    pin_gelu_identities,
    pin_gelu_asymptotes,
    pin_gelu_vs_erf,
    pin_gelu_known_values,
    pin_gelu_grad_fd,
    pin_forward_vs_numpy,
    pin_backward_vs_numpy,
    pin_gradients_fd,
    pin_partition_invariant,
    pin_special_cases,
    pin_sampled_matches_full,
    pin_ln_normalizes,
    pin_ln_affine_and_invariant,
    pin_ln_gradients_fd,
    pin_philox_known_answers,
    pin_dropout_mask,
    pin_dropout_forward,
    pin_dropout_backward_fd,
    pin_attn_vs_library,
    pin_attn_closed_forms,
    pin_attn_invariants,
    pin_attn_partition_invariant,
    pin_attn_gradients_fd,
    pin_attn_sampled_matches_full,
    pin_attn_rows_match_full,
]


def failing_pins(o):
    out = []
    for pin in ALL_PINS:
        try:
            ok = pin(o)
        except Exception:  # a mutant may also break an entry point outright
            ok = False
        if not ok:
            out.append(pin.__name__)
    return out
