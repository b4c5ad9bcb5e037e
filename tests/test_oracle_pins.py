"""The fp64 oracle against its pins, and the pins against planted mistakes."""

import os
import subprocess

import pytest

import oracle
from oracle import Oracle
from tests import oracle_pins as P

ORACLE_SRC = os.path.join(os.path.dirname(oracle.__file__), "tpmlp_oracle.c")


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    assert pin(orc)


# Plausible mistakes, each planted by a textual edit of the oracle's source:
# a wrong constant, a wrong sign, a dropped term, a transposed or shifted
# index, an operand swapped, a sum replaced by an overwrite.
MUTANTS = {
    "gelu_coefficient": ("0.5 * x * (1.0 + tanh(u));", "0.5 * x * (1.0 + tanh(1.05 * u));"),
    "gelu_sign": ("return 0.5 * x * (1.0 + tanh(u));", "return 0.5 * x * (1.0 - tanh(u));"),
    "gelu_grad_dropped_term": ("+ 0.5 * x * (1.0 - th * th) * du;", ";"),
    "gelu_grad_cubic_factor": ("(1.0 + 3.0 * 0.044715 * x * x)", "(1.0 + 0.044715 * x * x)"),
    "g_sum_overwrites": ("Y[e] += P[e]; /* g: sum of partials */", "Y[e] = P[e];"),
    "first_gemm_transposed": ("s += X[r * h + k] * A[k * F + c0 + j];",
                              "s += X[r * h + k] * A[(c0 + j) * h + k];"),
    "b2_dropped": ("Y[r * h + n] += b2[n] + R[r * h + n];", "Y[r * h + n] += R[r * h + n];"),
    "dB_uses_Z": ("s += H[r * F + c0 + j] * dY[r * h + n];", "s += Z[r * F + c0 + j] * dY[r * h + n];"),
    "db1_shard_offset": ("for (long r = 0; r < T; ++r) s += dZ[r * F + c0 + j];",
                         "for (long r = 0; r < T; ++r) s += dZ[r * F + j];"),
    "f_sum_overwrites": ("for (long e = 0; e < T * h; ++e) dX[e] += dXi[e];",
                         "for (long e = 0; e < T * h; ++e) dX[e] = dXi[e];"),
    "dA_wrong_operand": ("s += X[r * h + k] * dZ[r * F + c0 + j];",
                         "s += X[r * h + k] * H[r * F + c0 + j];"),
    "rows_g_sum_overwrites": ("y[n] += part[n - n0]; /* g sum */", "y[n] = part[n - n0];"),
    "rows_f_sum_overwrites": ("acc += s; /* f-operator sum */", "acc = s;"),
    "cols_gelu_instead_of_grad": ("dzc[r * ncols + q] = g * orc_gelu_grad(z);",
                                  "dzc[r * ncols + q] = g * orc_gelu(z);"),
    "cols_dB_wrong_row": ("sb += hc[r * ncols + q] * w16(dY[r * h + k]);",
                          "sb += hc[r * ncols + q] * w16(X[r * h + k]);"),
    "ln_unbiased_variance": ("double rs = 1.0 / sqrt(sq / (double)h + eps);\n        for (long j = 0; j < h; ++j) X[",
                             "double rs = 1.0 / sqrt(sq / (double)(h - 1) + eps);\n        for (long j = 0; j < h; ++j) X["),
    "ln_eps_outside_sqrt": ("double rs = 1.0 / sqrt(sq / (double)h + eps);\n        for (long j = 0; j < h; ++j) X[",
                            "double rs = 1.0 / (sqrt(sq / (double)h) + eps);\n        for (long j = 0; j < h; ++j) X["),
    "ln_bwd_drops_xhat_term": ("double v = rs * (g - mg - xhat[i * h + j] * mgx);",
                               "double v = rs * (g - mg);"),
    "ln_dgamma_uses_gamma": ("sg += dX[i * h + j] * xhat[i * h + j];",
                             "sg += dX[i * h + j] * gamma[j] * xhat[i * h + j];"),
    "ln_ds_drops_dres": ("ds[i * h + j] = v + (dres ? dres[i * h + j] : 0.0);", "ds[i * h + j] = v;"),
    "philox_multiplier": ("uint64_t p0 = (uint64_t)0xD2511F53u * c[0];", "uint64_t p0 = (uint64_t)0xD2511F55u * c[0];"),
    "philox_no_key_bump": ("k1 += 0xBB67AE85u;", "k1 += 0u;"),
    "dropout_no_rescale": ("Y[e] = R[e] + (keep[e] ? Y[e] / (1.0 - p) : 0.0);", "Y[e] = R[e] + (keep[e] ? Y[e] : 0.0);"),
    "dropout_bwd_ignores_mask": ("dP[e] = keep[e] ? dY[e] / (1.0 - p) : 0.0;", "dP[e] = dY[e] / (1.0 - p);"),
    "dropout_counter_word": ("keep[e] = w[g & 3] >= thr ? 1 : 0;", "keep[e] = w[0] >= thr ? 1 : 0;"),
    "attn_no_score_scale": ("row[c] = acc * scale;", "row[c] = acc;"),
    "attn_mask_open": ("c <= r; ++c) { /* causal: keys 0..r */", "c < s; ++c) { /* causal: keys 0..r */"),
    "attn_dS_drops_rowsum": ("P[r * s + c] * (dS[r * s + c] - D)", "P[r * s + c] * dS[r * s + c]"),
    "attn_dK_no_scale": ("dk[c * ldg + e] = a * scale;", "dk[c * ldg + e] = a;"),
    "attn_dV_uses_dS": ("b += P[r * s + c] * dO[r * ldo + e];", "b += dS[r * s + c] * dO[r * ldo + e];"),
    "attn_g_sum_overwrites": ("Y[r * h + n] += acc; /* g: sum of partials */", "Y[r * h + n] = acc;"),
    "attn_f_sum_overwrites": ("dX[r * h + k] += acc; /* f: sum of partials */", "dX[r * h + k] = acc;"),
    "attn_bo_dropped": ("Y[r * h + n] += bo[n] + R[r * h + n];", "Y[r * h + n] += R[r * h + n];"),
    "attn_k_v_swapped": ("attn_head_forward(base, base + h, base + 2 * h, 3 * h, s, d, O + n * s * h + j * d, h,",
                         "attn_head_forward(base, base + 2 * h, base + h, 3 * h, s, d, O + n * s * h + j * d, h,"),
    "attn_head_wrong_part_stride": ("out[part * d + e] += x * w16(wrow[part * h + e]);",
                                    "out[part * d + e] += x * w16(wrow[part * d + e]);"),
    "db2_drops_last_row": ("for (long r = 0; r < T; ++r) s += w16(dY[r * h + n]);",
                           "for (long r = 0; r + 1 < T; ++r) s += w16(dY[r * h + n]);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(ORACLE_SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} must occur exactly once"
    mut_c = tmp_path / "mutant.c"
    mut_c.write_text(src.replace(old, new))
    so = tmp_path / "mutant.so"
    r = subprocess.run(["gcc", "-O1", "-std=c11", "-D_DEFAULT_SOURCE", "-fPIC", "-shared",
                        str(mut_c), "-o", str(so), "-lm"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    failed = P.failing_pins(Oracle(str(so)))
    assert failed, f"no pin caught the planted mistake {name}"


# Planted mistakes in the sampled-row attention oracle (numpy), each loaded
# from an edited copy of its source.
ATTN_ROWS_SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_rows.py")
ROWS_MUTANTS = {
    "rows_mask_open": ("S = np.where(causal, Q @ K.T * scale, -np.inf)", "S = Q @ K.T * scale"),
    "rows_no_score_scale": ("S = np.where(causal, Q @ K.T * scale, -np.inf)",
                            "S = np.where(causal, Q @ K.T, -np.inf)"),
    "rows_dS_drops_rowsum": ("dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))", "dS = P * dP"),
    "rows_dQ_no_scale": ("dqkv[:, c] = dS[pos] @ K * scale", "dqkv[:, c] = dS[pos] @ K"),
    "rows_dK_transposed": ("dqkv[:, ck] = dS[:, pos].T @ Q * scale", "dqkv[:, ck] = dS[pos] @ Q * scale"),
    "rows_dV_uses_dS": ("dqkv[:, cv] = P[:, pos].T @ dOj", "dqkv[:, cv] = dS[:, pos].T @ dOj"),
    "rows_k_v_swapped": ("Q, K, V = qkv[:, c], qkv[:, ck], qkv[:, cv]",
                         "Q, K, V = qkv[:, c], qkv[:, cv], qkv[:, ck]"),
    "rows_g_sum_overwrites": ("Y[sel] += O[pos] @ Woi", "Y[sel] = O[pos] @ Woi"),
    "rows_f_sum_overwrites": ("dX[sel] += dqkv @ Wi.T", "dX[sel] = dqkv @ Wi.T"),
    "rows_bo_dropped": ('Y += _f64(inp["bo"]) + _f64(inp["residual"][torch.as_tensor(rows)])',
                        'Y += _f64(inp["residual"][torch.as_tensor(rows)])'),
    "rows_wrong_shard_columns": ("np.arange(p * h + i * w, p * h + (i + 1) * w)",
                                 "np.arange(p * w + i * w, p * w + (i + 1) * w)"),
}


@pytest.mark.parametrize("name", sorted(ROWS_MUTANTS))
def test_pins_catch_attn_rows_mutant(name):
    import types

    old, new = ROWS_MUTANTS[name]
    src = open(ATTN_ROWS_SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} must occur exactly once"
    mod = types.ModuleType("attn_rows_mutant")
    exec(compile(src.replace(old, new), "attn_rows_mutant.py", "exec"), mod.__dict__)
    failed = P.failing_pins(Oracle(attn_rows_impl=mod.attn_rows))
    assert failed, f"no pin caught the planted mistake {name}"
