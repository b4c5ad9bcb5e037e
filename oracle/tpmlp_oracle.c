/*
 * tpmlp_oracle.c -- plain, slow fp64 CPU oracle of the tensor-parallel
 * Transformer MLP block, forward and backward.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header
 * or constant with the CUDA path, and the product path never calls it.
 *
 * What it computes (row-major matrices, T tokens, hidden h, FFN width F,
 * t shards of width f = F / t):
 *
 *   shard i owns A_i = A[:, i f:(i+1) f], b1_i, B_i = B[i f:(i+1) f, :]
 *   Z_i = X A_i + b1_i                 column-parallel first GEMM
 *   H_i = GeLU(Z_i)                    local nonlinearity, no sync before it
 *   Y   = sum_i H_i B_i + b2 + R       row-parallel partials, the g-operator
 *                                      sum, then bias and residual
 *
 * following "Megatron-LM: Tensor Model Parallel" (charles2530.github.io),
 * section "MLP: Column Parallel first, then Row Parallel" (Figure 3a) and
 * section "f / g Operators" (Figure 4: g is a sum in the forward pass and the
 * identity in the backward pass; f is the identity forward and a sum
 * backward).  The backward pass is the chain rule of the same formula:
 *
 *   dH_i = dY B_i^T ;  dZ_i = dH_i * GeLU'(Z_i)
 *   dB_i = H_i^T dY ;  dA_i = X^T dZ_i ;  db1_i = sum_rows dZ_i
 *   dX   = sum_i dZ_i A_i^T            the f-operator sum
 *   db2  = sum_rows dY                 (d residual = dY, not returned)
 *
 * Readings where the pages are silent:
 *  - GeLU is named but never defined on the pages; the tanh approximation
 *    0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) is used.
 *  - The pages' MLP has no biases.  b1 is split with A's columns (it must be
 *    added before the local GeLU); b2 and the residual are added once, after
 *    the shard sum.
 *  - Nothing is rounded: inputs are widened exactly to double and every
 *    intermediate stays double.  The oracle recomputes Z and H itself in the
 *    backward pass.
 *
 * Each shard's partial product is formed on its own and then added to the
 * running sum, exactly as the pages' per-rank computation followed by the
 * all-reduce.  Loops are plain; OpenMP only splits independent output rows
 * or columns across threads, never a sum.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_SHAPE 2
#define ORC_ERR_ALLOC 8

static double gelu_c(void) { return sqrt(2.0 / M_PI); }

/* GeLU, tanh approximation (reading of the pages' unnamed "GeLU"). */
double orc_gelu(double x) {
    double u = gelu_c() * (x + 0.044715 * x * x * x);
    return 0.5 * x * (1.0 + tanh(u));
}

/* d/dx of orc_gelu, written out by the product and chain rules. */
double orc_gelu_grad(double x) {
    double u = gelu_c() * (x + 0.044715 * x * x * x);
    double th = tanh(u);
    double du = gelu_c() * (1.0 + 3.0 * 0.044715 * x * x);
    return 0.5 * (1.0 + th) + 0.5 * x * (1.0 - th * th) * du;
}

static int bad_shape(long T, long h, long F, long t) {
    return T < 0 || h < 1 || F < 1 || t < 1 || F % t != 0;
}

/* ---------------------------------------------------------------------- */
/* Full computation on fp64 inputs (small problems).                       */
/* ---------------------------------------------------------------------- */

/* Column-parallel step for shard i: Z_i = X A_i + b1_i, H_i = GeLU(Z_i).
 * Z and H are the full [T, F] arrays; shard i fills its column block. */
static void shard_forward_first(const double* X, const double* A, const double* b1,
                                long T, long h, long F, long f, long i,
                                double* Z, double* H) {
    long c0 = i * f;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < T; ++r) {
        for (long j = 0; j < f; ++j) {
            double s = 0.0;
            for (long k = 0; k < h; ++k) s += X[r * h + k] * A[k * F + c0 + j];
            double z = s + b1[c0 + j];
            Z[r * F + c0 + j] = z;
            H[r * F + c0 + j] = orc_gelu(z);
        }
    }
}

/* Row-parallel partial for shard i: P_i = H_i B_i  ([T, h]). */
static void shard_forward_second(const double* H, const double* B, long T, long h,
                                 long F, long f, long i, double* P) {
    long c0 = i * f;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < T; ++r) {
        for (long n = 0; n < h; ++n) {
            double s = 0.0;
            for (long j = 0; j < f; ++j) s += H[r * F + c0 + j] * B[(c0 + j) * h + n];
            P[r * h + n] = s;
        }
    }
}

/* Forward pass.  Y [T,h]; Z, H [T,F] (may be NULL when not wanted). */
int orc_forward(const double* X, const double* A, const double* b1, const double* B,
                const double* b2, const double* R, long T, long h, long F, long t,
                double* Y, double* Z, double* H) {
    if (bad_shape(T, h, F, t)) return ORC_ERR_SHAPE;
    long f = F / t;
    double* Zw = Z ? Z : (double*)malloc(sizeof(double) * (size_t)(T * F + 1));
    double* Hw = H ? H : (double*)malloc(sizeof(double) * (size_t)(T * F + 1));
    double* P = (double*)malloc(sizeof(double) * (size_t)(T * h + 1));
    if (!Zw || !Hw || !P) {
        if (!Z) free(Zw);
        if (!H) free(Hw);
        free(P);
        return ORC_ERR_ALLOC;
    }
    for (long e = 0; e < T * h; ++e) Y[e] = 0.0;
    for (long i = 0; i < t; ++i) {
        shard_forward_first(X, A, b1, T, h, F, f, i, Zw, Hw);
        shard_forward_second(Hw, B, T, h, F, f, i, P);
        for (long e = 0; e < T * h; ++e) Y[e] += P[e]; /* g: sum of partials */
    }
    for (long r = 0; r < T; ++r)
        for (long n = 0; n < h; ++n) Y[r * h + n] += b2[n] + R[r * h + n];
    if (!Z) free(Zw);
    if (!H) free(Hw);
    free(P);
    return ORC_OK;
}

/* Backward pass given the upstream gradient dY [T,h].
 * Outputs: dX [T,h], dA [h,F], dB [F,h], db1 [F], db2 [h]. */
int orc_backward(const double* dY, const double* X, const double* A, const double* b1,
                 const double* B, long T, long h, long F, long t, double* dX, double* dA,
                 double* dB, double* db1, double* db2) {
    if (bad_shape(T, h, F, t)) return ORC_ERR_SHAPE;
    long f = F / t;
    double* Z = (double*)malloc(sizeof(double) * (size_t)(T * F + 1));
    double* H = (double*)malloc(sizeof(double) * (size_t)(T * F + 1));
    double* dZ = (double*)malloc(sizeof(double) * (size_t)(T * F + 1));
    double* dXi = (double*)malloc(sizeof(double) * (size_t)(T * h + 1));
    if (!Z || !H || !dZ || !dXi) {
        free(Z); free(H); free(dZ); free(dXi);
        return ORC_ERR_ALLOC;
    }
    for (long e = 0; e < T * h; ++e) dX[e] = 0.0;
    for (long i = 0; i < t; ++i) {
        long c0 = i * f;
        shard_forward_first(X, A, b1, T, h, F, f, i, Z, H);
        /* dZ_i = (dY B_i^T) * GeLU'(Z_i) */
#pragma omp parallel for schedule(static)
        for (long r = 0; r < T; ++r) {
            for (long j = 0; j < f; ++j) {
                double s = 0.0;
                for (long n = 0; n < h; ++n) s += dY[r * h + n] * B[(c0 + j) * h + n];
                dZ[r * F + c0 + j] = s * orc_gelu_grad(Z[r * F + c0 + j]);
            }
        }
        /* dB_i = H_i^T dY */
#pragma omp parallel for schedule(static)
        for (long j = 0; j < f; ++j) {
            for (long n = 0; n < h; ++n) {
                double s = 0.0;
                for (long r = 0; r < T; ++r) s += H[r * F + c0 + j] * dY[r * h + n];
                dB[(c0 + j) * h + n] = s;
            }
        }
        /* dA_i = X^T dZ_i */
#pragma omp parallel for schedule(static)
        for (long k = 0; k < h; ++k) {
            for (long j = 0; j < f; ++j) {
                double s = 0.0;
                for (long r = 0; r < T; ++r) s += X[r * h + k] * dZ[r * F + c0 + j];
                dA[k * F + c0 + j] = s;
            }
        }
        /* db1_i = column sums of dZ_i */
        for (long j = 0; j < f; ++j) {
            double s = 0.0;
            for (long r = 0; r < T; ++r) s += dZ[r * F + c0 + j];
            db1[c0 + j] = s;
        }
        /* dX_i = dZ_i A_i^T, then the f-operator sum over shards */
#pragma omp parallel for schedule(static)
        for (long r = 0; r < T; ++r) {
            for (long k = 0; k < h; ++k) {
                double s = 0.0;
                for (long j = 0; j < f; ++j) s += dZ[r * F + c0 + j] * A[k * F + c0 + j];
                dXi[r * h + k] = s;
            }
        }
        for (long e = 0; e < T * h; ++e) dX[e] += dXi[e];
    }
    for (long n = 0; n < h; ++n) {
        double s = 0.0;
        for (long r = 0; r < T; ++r) s += dY[r * h + n];
        db2[n] = s;
    }
    free(Z); free(H); free(dZ); free(dXi);
    return ORC_OK;
}

/* ---------------------------------------------------------------------- */
/* Sampled computation on bf16 inputs (large problems).                     */
/* Inputs are raw bfloat16 bit patterns, widened exactly to double on read. */
/* Each sampled output is the same definition as above, evaluated alone.   */
/* ---------------------------------------------------------------------- */

static inline double w16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float v;
    memcpy(&v, &u, sizeof v);
    return (double)v;
}

/* Z and H for a set of rows: Zr, Hr are [nrows, F]. */
static void rows_first(const uint16_t* X, const uint16_t* A, const uint16_t* b1, long h,
                       long F, const long* rows, long nrows, double* Zr, double* Hr) {
    /* Each thread owns a block of columns and walks k in ascending order, so
     * every Z entry is b1 + sum_k X[r,k] A[k,j] summed from k = 0 upwards. */
#pragma omp parallel for schedule(static)
    for (long j0 = 0; j0 < F; j0 += 256) {
        long j1 = j0 + 256 < F ? j0 + 256 : F;
        for (long q = 0; q < nrows; ++q)
            for (long j = j0; j < j1; ++j) Zr[q * F + j] = 0.0;
        for (long k = 0; k < h; ++k) {
            const uint16_t* Ak = A + k * F;
            for (long q = 0; q < nrows; ++q) {
                double x = w16(X[rows[q] * h + k]);
                double* z = Zr + q * F;
                for (long j = j0; j < j1; ++j) z[j] += x * w16(Ak[j]);
            }
        }
        for (long q = 0; q < nrows; ++q)
            for (long j = j0; j < j1; ++j) {
                double z = Zr[q * F + j] + w16(b1[j]);
                Zr[q * F + j] = z;
                Hr[q * F + j] = orc_gelu(z);
            }
    }
}

/* Y rows: Y[r,:] = sum_i H_i[r,:] B_i + b2 + R[r,:].  Yr is [nrows, h];
 * Zr, Hr ([nrows, F]) receive the pre-activation and GeLU rows (may be NULL). */
int orc_forward_rows_bf16(const uint16_t* X, const uint16_t* A, const uint16_t* b1,
                          const uint16_t* B, const uint16_t* b2, const uint16_t* R,
                          long T, long h, long F, long t, const long* rows, long nrows,
                          double* Yr, double* Zr, double* Hr) {
    if (bad_shape(T, h, F, t)) return ORC_ERR_SHAPE;
    for (long q = 0; q < nrows; ++q)
        if (rows[q] < 0 || rows[q] >= T) return ORC_ERR_SHAPE;
    long f = F / t;
    double* Z = Zr ? Zr : (double*)malloc(sizeof(double) * (size_t)(nrows * F + 1));
    double* H = Hr ? Hr : (double*)malloc(sizeof(double) * (size_t)(nrows * F + 1));
    if (!Z || !H) {
        if (!Zr) free(Z);
        if (!Hr) free(H);
        return ORC_ERR_ALLOC;
    }
    rows_first(X, A, b1, h, F, rows, nrows, Z, H);
#pragma omp parallel for schedule(static)
    for (long n0 = 0; n0 < h; n0 += 64) {
        long n1 = n0 + 64 < h ? n0 + 64 : h;
        double part[64];
        for (long q = 0; q < nrows; ++q) {
            double* y = Yr + q * h;
            for (long n = n0; n < n1; ++n) y[n] = 0.0;
            for (long i = 0; i < t; ++i) {
                for (long n = n0; n < n1; ++n) part[n - n0] = 0.0;
                for (long j = i * f; j < (i + 1) * f; ++j) {
                    double hv = H[q * F + j];
                    const uint16_t* Bj = B + j * h;
                    for (long n = n0; n < n1; ++n) part[n - n0] += hv * w16(Bj[n]);
                }
                for (long n = n0; n < n1; ++n) y[n] += part[n - n0]; /* g sum */
            }
            for (long n = n0; n < n1; ++n) y[n] += w16(b2[n]) + w16(R[rows[q] * h + n]);
        }
    }
    if (!Zr) free(Z);
    if (!Hr) free(H);
    return ORC_OK;
}

/* dX rows: dX[r,:] = sum_i (dY[r,:] B_i^T * GeLU'(Z_i[r,:])) A_i^T.
 * dXr is [nrows, h]. */
int orc_backward_rows_bf16(const uint16_t* dY, const uint16_t* X, const uint16_t* A,
                           const uint16_t* b1, const uint16_t* B, long T, long h, long F,
                           long t, const long* rows, long nrows, double* dXr) {
    if (bad_shape(T, h, F, t)) return ORC_ERR_SHAPE;
    for (long q = 0; q < nrows; ++q)
        if (rows[q] < 0 || rows[q] >= T) return ORC_ERR_SHAPE;
    long f = F / t;
    double* Z = (double*)malloc(sizeof(double) * (size_t)(nrows * F + 1));
    double* H = (double*)malloc(sizeof(double) * (size_t)(nrows * F + 1));
    double* dZ = (double*)malloc(sizeof(double) * (size_t)(nrows * F + 1));
    if (!Z || !H || !dZ) {
        free(Z); free(H); free(dZ);
        return ORC_ERR_ALLOC;
    }
    rows_first(X, A, b1, h, F, rows, nrows, Z, H);
    /* dZ[r, j] = (sum_n dY[r,n] B[j,n]) * GeLU'(Z[r,j]) */
#pragma omp parallel for schedule(static)
    for (long j = 0; j < F; ++j) {
        const uint16_t* Bj = B + j * h;
        for (long q = 0; q < nrows; ++q) {
            const uint16_t* d = dY + rows[q] * h;
            double s = 0.0;
            for (long n = 0; n < h; ++n) s += w16(d[n]) * w16(Bj[n]);
            dZ[q * F + j] = s * orc_gelu_grad(Z[q * F + j]);
        }
    }
    /* dX[r, k] = sum_i sum_{j in shard i} dZ[r,j] A[k,j] */
#pragma omp parallel for schedule(static)
    for (long k = 0; k < h; ++k) {
        const uint16_t* Ak = A + k * F;
        for (long q = 0; q < nrows; ++q) {
            double acc = 0.0;
            for (long i = 0; i < t; ++i) {
                double s = 0.0;
                for (long j = i * f; j < (i + 1) * f; ++j) s += dZ[q * F + j] * w16(Ak[j]);
                acc += s; /* f-operator sum */
            }
            dXr[q * h + k] = acc;
        }
    }
    free(Z); free(H); free(dZ);
    return ORC_OK;
}

/* Sampled FFN columns j (global index into F):
 *   dA[:, j] ([h] per column) -> dAc is [h, ncols] (column q at dAc[k*ncols+q]);
 *   dB[j, :] ([h] per column) -> dBr is [ncols, h];
 *   db1[j]                    -> db1c is [ncols]. */
int orc_backward_cols_bf16(const uint16_t* dY, const uint16_t* X, const uint16_t* A,
                           const uint16_t* b1, const uint16_t* B, long T, long h, long F,
                           long t, const long* cols, long ncols, double* dAc, double* dBr,
                           double* db1c) {
    if (bad_shape(T, h, F, t)) return ORC_ERR_SHAPE;
    for (long q = 0; q < ncols; ++q)
        if (cols[q] < 0 || cols[q] >= F) return ORC_ERR_SHAPE;
    double* zc = (double*)malloc(sizeof(double) * (size_t)(T * ncols + 1));
    double* hc = (double*)malloc(sizeof(double) * (size_t)(T * ncols + 1));
    double* dzc = (double*)malloc(sizeof(double) * (size_t)(T * ncols + 1));
    if (!zc || !hc || !dzc) {
        free(zc); free(hc); free(dzc);
        return ORC_ERR_ALLOC;
    }
    /* Z[:, j], H[:, j], dZ[:, j] for every sampled column (row-major [T, ncols]) */
#pragma omp parallel for schedule(static)
    for (long r = 0; r < T; ++r) {
        const uint16_t* xr = X + r * h;
        const uint16_t* dr = dY + r * h;
        for (long q = 0; q < ncols; ++q) {
            long j = cols[q];
            double z = 0.0;
            for (long k = 0; k < h; ++k) z += w16(xr[k]) * w16(A[k * F + j]);
            z += w16(b1[j]);
            double g = 0.0;
            for (long n = 0; n < h; ++n) g += w16(dr[n]) * w16(B[j * h + n]);
            zc[r * ncols + q] = z;
            hc[r * ncols + q] = orc_gelu(z);
            dzc[r * ncols + q] = g * orc_gelu_grad(z);
        }
    }
    /* dA[k, j] = sum_r X[r,k] dZ[r,j] ; dB[j, n] = sum_r H[r,j] dY[r,n] */
#pragma omp parallel for schedule(static)
    for (long k = 0; k < h; ++k) {
        for (long q = 0; q < ncols; ++q) {
            double sa = 0.0, sb = 0.0;
            for (long r = 0; r < T; ++r) {
                sa += w16(X[r * h + k]) * dzc[r * ncols + q];
                sb += hc[r * ncols + q] * w16(dY[r * h + k]);
            }
            dAc[k * ncols + q] = sa;
            dBr[q * h + k] = sb;
        }
    }
    for (long q = 0; q < ncols; ++q) {
        double s = 0.0;
        for (long r = 0; r < T; ++r) s += dzc[r * ncols + q];
        db1c[q] = s;
    }
    free(zc); free(hc); free(dzc);
    return ORC_OK;
}

/* db2 = column sums of dY (all h entries). */
int orc_db2_bf16(const uint16_t* dY, long T, long h, double* db2) {
    if (T < 0 || h < 1) return ORC_ERR_SHAPE;
#pragma omp parallel for schedule(static)
    for (long n = 0; n < h; ++n) {
        double s = 0.0;
        for (long r = 0; r < T; ++r) s += w16(dY[r * h + n]);
        db2[n] = s;
    }
    return ORC_OK;
}

/* Threads the OpenMP runtime will use (1 without OpenMP). */
int orc_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------- */
/* Residual add + LayerNorm feeding the block's input X.                   */
/*                                                                         */
/* "Megatron-DeepSpeed to ZeRO-3" (seekfood.cn), section 4.3, gives only   */
/* the signature of a fused LayerNorm + residual kernel (output, input,    */
/* residual, gamma, beta, n); "Megatron-LM: Tensor Model Parallel",        */
/* Figure 2, places layer normalization and the residual connection around */
/* the MLP.  Reading: per row of n = h values                              */
/*   s = input + residual                (the residual stream)            */
/*   mu = mean(s), var = mean((s - mu)^2)  (biased), rstd = 1/sqrt(var+eps)*/
/*   X = (s - mu) * rstd * gamma + beta  (the MLP's input)                */
/* and the backward pass of the same formula, where ds also receives      */
/* dres, the gradient reaching s directly (the MLP's residual path):      */
/*   xhat = (s - mu) rstd ; g = dX * gamma                                */
/*   ds = rstd (g - mean(g) - xhat mean(g xhat)) + dres                   */
/*   dgamma = sum_rows dX xhat ; dbeta = sum_rows dX ; dinput = dres_in = ds */
/* ---------------------------------------------------------------------- */

int orc_ln_forward(const double* a, const double* r, const double* gamma, const double* beta,
                   long T, long h, double eps, double* X, double* s, double* mean, double* rstd) {
    if (T < 0 || h < 1) return ORC_ERR_SHAPE;
#pragma omp parallel for schedule(static)
    for (long i = 0; i < T; ++i) {
        const double* ai = a + i * h;
        const double* ri = r + i * h;
        double* si = s + i * h;
        double sum = 0.0;
        for (long j = 0; j < h; ++j) {
            si[j] = ai[j] + ri[j];
            sum += si[j];
        }
        double mu = sum / (double)h;
        double sq = 0.0;
        for (long j = 0; j < h; ++j) sq += (si[j] - mu) * (si[j] - mu);
        double rs = 1.0 / sqrt(sq / (double)h + eps);
        for (long j = 0; j < h; ++j) X[i * h + j] = (si[j] - mu) * rs * gamma[j] + beta[j];
        mean[i] = mu;
        rstd[i] = rs;
    }
    return ORC_OK;
}

/* dres may be NULL (no residual-path gradient). */
int orc_ln_backward(const double* dX, const double* dres, const double* a, const double* r,
                    const double* gamma, long T, long h, double eps, double* ds,
                    double* dgamma, double* dbeta) {
    if (T < 0 || h < 1) return ORC_ERR_SHAPE;
    double* xhat = (double*)malloc(sizeof(double) * (size_t)(T * h + 1));
    if (!xhat) return ORC_ERR_ALLOC;
#pragma omp parallel for schedule(static)
    for (long i = 0; i < T; ++i) {
        const double* ai = a + i * h;
        const double* ri = r + i * h;
        double sum = 0.0;
        for (long j = 0; j < h; ++j) sum += ai[j] + ri[j];
        double mu = sum / (double)h;
        double sq = 0.0;
        for (long j = 0; j < h; ++j) {
            double c = ai[j] + ri[j] - mu;
            sq += c * c;
        }
        double rs = 1.0 / sqrt(sq / (double)h + eps);
        double mg = 0.0, mgx = 0.0;
        for (long j = 0; j < h; ++j) {
            double xh = (ai[j] + ri[j] - mu) * rs;
            double g = dX[i * h + j] * gamma[j];
            xhat[i * h + j] = xh;
            mg += g;
            mgx += g * xh;
        }
        mg /= (double)h;
        mgx /= (double)h;
        for (long j = 0; j < h; ++j) {
            double g = dX[i * h + j] * gamma[j];
            double v = rs * (g - mg - xhat[i * h + j] * mgx);
            ds[i * h + j] = v + (dres ? dres[i * h + j] : 0.0);
        }
    }
#pragma omp parallel for schedule(static)
    for (long j = 0; j < h; ++j) {
        double sg = 0.0, sb = 0.0;
        for (long i = 0; i < T; ++i) {
            sg += dX[i * h + j] * xhat[i * h + j];
            sb += dX[i * h + j];
        }
        dgamma[j] = sg;
        dbeta[j] = sb;
    }
    free(xhat);
    return ORC_OK;
}

/* ---------------------------------------------------------------------- */
/* Dropout before the residual add ("bias-dropout-add").                   */
/*                                                                         */
/* "Megatron-LM: Tensor Model Parallel", section "Hybrid MP + DP" (the     */
/* random-number paragraph): the dropout in front of the residual lies     */
/* outside the model-parallel region and uses the same pattern on every    */
/* TP rank; the training-recipe table sets dropout 0.1.  Reading:          */
/*   Y = R + keep * (sum_i H_i B_i + b2) / (1 - p)                         */
/* with keep(e) for element e = row * h + col decided by a counter-based    */
/* generator shared by every shard: Philox4x32 with 10 rounds (Salmon et   */
/* al., "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11).  Counter    */
/* g = offset + e: word g % 4 of Philox(counter = (lo g/4, hi g/4, 0, 0),   */
/* key = (lo seed, hi seed)); keep iff word >= floor(p * 2^32).            */
/* ---------------------------------------------------------------------- */

/* One Philox4x32-10 block: 10 rounds of the multiply-hi/lo bijection with
 * multipliers 0xD2511F53 (word 0) and 0xCD9E8D57 (word 2), the key bumped by
 * the Weyl constants 0x9E3779B9, 0xBB67AE85 between rounds. */
void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    uint32_t c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c[1] ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c[3] ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c[0] = n0; c[1] = n1; c[2] = n2; c[3] = n3;
    }
    out[0] = c[0]; out[1] = c[1]; out[2] = c[2]; out[3] = c[3];
}

/* keep[e] for the n elements e = 0 .. n-1 (1 = kept). */
int orc_dropout_mask(uint64_t seed, uint64_t offset, long n, double p, uint8_t* keep) {
    if (n < 0 || !(p >= 0.0 && p < 1.0)) return ORC_ERR_SHAPE;
    uint32_t thr = (uint32_t)(p * 4294967296.0);
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
#pragma omp parallel for schedule(static)
    for (long e = 0; e < n; ++e) {
        uint64_t g = offset + (uint64_t)e;
        uint64_t blk = g >> 2;
        uint32_t ctr[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), 0u, 0u};
        uint32_t w[4];
        orc_philox4x32_10(ctr, key, w);
        keep[e] = w[g & 3] >= thr ? 1 : 0;
    }
    return ORC_OK;
}

/* Forward with dropout: Y = R + keep * (sum_i H_i B_i + b2) / (1 - p). */
int orc_forward_dropout(const double* X, const double* A, const double* b1, const double* B,
                        const double* b2, const double* R, long T, long h, long F, long t,
                        double p, uint64_t seed, uint64_t offset, double* Y, double* Z,
                        double* H) {
    if (bad_shape(T, h, F, t)) return ORC_ERR_SHAPE;
    double* zero = (double*)calloc((size_t)(T * h + 1), sizeof(double));
    uint8_t* keep = (uint8_t*)malloc((size_t)(T * h + 1));
    if (!zero || !keep) {
        free(zero); free(keep);
        return ORC_ERR_ALLOC;
    }
    /* the MLP's output before the residual: sum_i H_i B_i + b2 */
    int rc = orc_forward(X, A, b1, B, b2, zero, T, h, F, t, Y, Z, H);
    if (rc == ORC_OK) rc = orc_dropout_mask(seed, offset, T * h, p, keep);
    if (rc == ORC_OK)
        for (long e = 0; e < T * h; ++e) Y[e] = R[e] + (keep[e] ? Y[e] / (1.0 - p) : 0.0);
    free(zero); free(keep);
    return rc;
}

/* Backward with dropout: the MLP sees dP = keep * dY / (1 - p) (the residual
 * still receives dY).  Outputs as orc_backward. */
int orc_backward_dropout(const double* dY, const double* X, const double* A, const double* b1,
                         const double* B, long T, long h, long F, long t, double p, uint64_t seed,
                         uint64_t offset, double* dX, double* dA, double* dB, double* db1,
                         double* db2) {
    if (bad_shape(T, h, F, t)) return ORC_ERR_SHAPE;
    double* dP = (double*)malloc(sizeof(double) * (size_t)(T * h + 1));
    uint8_t* keep = (uint8_t*)malloc((size_t)(T * h + 1));
    if (!dP || !keep) {
        free(dP); free(keep);
        return ORC_ERR_ALLOC;
    }
    int rc = orc_dropout_mask(seed, offset, T * h, p, keep);
    if (rc == ORC_OK) {
        for (long e = 0; e < T * h; ++e) dP[e] = keep[e] ? dY[e] / (1.0 - p) : 0.0;
        rc = orc_backward(dP, X, A, b1, B, T, h, F, t, dX, dA, dB, db1, db2);
    }
    free(dP); free(keep);
    return rc;
}

/* ------------------------------------------------------------------ */
/* Head-parallel self-attention block                                  */
/* ------------------------------------------------------------------ */
/*
 * "Megatron-LM: Tensor Model Parallel", section "Attention: split Q/K/V by
 * head" (Figure 3b): the Q, K and V projections are split by columns so that
 * each rank holds a subset of the heads; a head's scores, softmax and value
 * sum are computed locally; the output projection is split by rows and its
 * per-rank partials meet in the g-operator sum before the residual.
 *
 * Layout (readings; the page fixes only the split):
 *  - X, R, Y [T, h] with T = nb sequences of s tokens (token = n s + pos);
 *  - Wqkv [h, 3h], columns [Q | K | V], head j at columns j d .. j d + d - 1
 *    of each part, d = h / nh; bqkv [3h] likewise; Wo [h, h] with the rows
 *    of head j at j d ..; bo [h];
 *  - shard i owns heads i nh/t .. (i+1) nh/t - 1: their Wqkv columns, bqkv
 *    entries and Wo rows.
 * Scores are scaled by 1/sqrt(d) and causal: a token attends to itself and
 * the earlier tokens of its own sequence (the GPT models of the pages).
 *
 *   QKV = X Wqkv + bqkv
 *   each sequence n, head j:  S = Q_j K_j^T / sqrt(d), masked,
 *                             P = softmax over each row, O_j = P V_j
 *   Y = sum_i O_i Wo_i + bo + R
 * Backward (chain rule of the same formula, forward recomputed from X):
 *   dbo = sum_rows dY ; dWo_i = O_i^T dY ; dO_i = dY Wo_i^T
 *   dV = P^T dO_j ; dP = dO_j V_j^T ; dS = P * (dP - rowsum(P * dP))
 *   dQ = dS K_j / sqrt(d) ; dK = dS^T Q_j / sqrt(d)
 *   dWqkv = X^T dQKV ; dbqkv = sum_rows dQKV ; dX = sum_i dQKV_i Wqkv_i^T
 */

static int attn_bad(long nb, long s, long h, long nh, long t) {
    if (nb < 0 || s < 1 || h < 1 || nh < 1 || t < 1) return 1;
    if (h % nh != 0 || nh % t != 0) return 1;
    return 0;
}

/* One head of one sequence.  q, k, v: s x d with row stride ld; writes the
 * s x d output o (row stride ldo) and, when P is not NULL, the s x s
 * probabilities (zero above the diagonal). */
static void attn_head_forward(const double* q, const double* k, const double* v, long ld,
                              long s, long d, double* o, long ldo, double* P) {
    double scale = 1.0 / sqrt((double)d);
    double* row = (double*)malloc(sizeof(double) * (size_t)s);
    for (long r = 0; r < s; ++r) {
        double m = -INFINITY;
        for (long c = 0; c <= r; ++c) { /* causal: keys 0..r */
            double acc = 0.0;
            for (long e = 0; e < d; ++e) acc += q[r * ld + e] * k[c * ld + e];
            row[c] = acc * scale;
            if (row[c] > m) m = row[c];
        }
        double sum = 0.0;
        for (long c = 0; c <= r; ++c) {
            row[c] = exp(row[c] - m);
            sum += row[c];
        }
        for (long c = 0; c <= r; ++c) row[c] /= sum;
        for (long e = 0; e < d; ++e) {
            double acc = 0.0;
            for (long c = 0; c <= r; ++c) acc += row[c] * v[c * ld + e];
            o[r * ldo + e] = acc;
        }
        if (P)
            for (long c = 0; c < s; ++c) P[r * s + c] = c <= r ? row[c] : 0.0;
    }
    free(row);
}

/* Backward of one head of one sequence: given dO (s x d, stride ldo) writes
 * dq, dk, dv (s x d, stride ldg). */
static void attn_head_backward(const double* q, const double* k, const double* v, long ld,
                               long s, long d, const double* dO, long ldo, double* dq,
                               double* dk, double* dv, long ldg) {
    double scale = 1.0 / sqrt((double)d);
    double* P = (double*)malloc(sizeof(double) * (size_t)(s * s));
    double* dS = (double*)malloc(sizeof(double) * (size_t)(s * s));
    double* o = (double*)malloc(sizeof(double) * (size_t)(s * d));
    attn_head_forward(q, k, v, ld, s, d, o, d, P);
    for (long r = 0; r < s; ++r) {
        double D = 0.0;
        for (long c = 0; c <= r; ++c) {
            double dp = 0.0;
            for (long e = 0; e < d; ++e) dp += dO[r * ldo + e] * v[c * ld + e];
            dS[r * s + c] = dp;
            D += P[r * s + c] * dp;
        }
        for (long c = 0; c < s; ++c)
            dS[r * s + c] = c <= r ? P[r * s + c] * (dS[r * s + c] - D) : 0.0;
    }
    for (long r = 0; r < s; ++r)
        for (long e = 0; e < d; ++e) {
            double a = 0.0;
            for (long c = 0; c <= r; ++c) a += dS[r * s + c] * k[c * ld + e];
            dq[r * ldg + e] = a * scale;
        }
    for (long c = 0; c < s; ++c)
        for (long e = 0; e < d; ++e) {
            double a = 0.0, b = 0.0;
            for (long r = c; r < s; ++r) {
                a += dS[r * s + c] * q[r * ld + e];
                b += P[r * s + c] * dO[r * ldo + e];
            }
            dk[c * ldg + e] = a * scale;
            dv[c * ldg + e] = b;
        }
    free(P); free(dS); free(o);
}

/* QKV columns of shard i (its Q, K and V blocks of width h/t): out = X W + b. */
static void attn_qkv_shard(const double* X, const double* Wqkv, const double* bqkv, long T,
                           long h, long t, long i, double* QKV) {
    long w = h / t;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < T; ++r)
        for (long part = 0; part < 3; ++part)
            for (long c = part * h + i * w; c < part * h + (i + 1) * w; ++c) {
                double acc = bqkv[c];
                for (long k = 0; k < h; ++k) acc += X[r * h + k] * Wqkv[k * 3 * h + c];
                QKV[r * 3 * h + c] = acc;
            }
}

/* Attention of shard i's heads for every sequence: O columns of shard i. */
static void attn_shard_core(const double* QKV, long nb, long s, long h, long nh, long t, long i,
                            double* O) {
    long d = h / nh, hs = nh / t;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (long n = 0; n < nb; ++n)
        for (long jj = 0; jj < hs; ++jj) {
            long j = i * hs + jj;
            const double* base = QKV + n * s * 3 * h + j * d;
            attn_head_forward(base, base + h, base + 2 * h, 3 * h, s, d, O + n * s * h + j * d, h,
                              NULL);
        }
}

int orc_attn_forward(const double* X, const double* Wqkv, const double* bqkv, const double* Wo,
                     const double* bo, const double* R, long nb, long s, long h, long nh, long t,
                     double* Y, double* QKV, double* O) {
    if (attn_bad(nb, s, h, nh, t)) return ORC_ERR_SHAPE;
    long T = nb * s, w = h / t;
    for (long e = 0; e < T * h; ++e) Y[e] = 0.0;
    for (long i = 0; i < t; ++i) {
        attn_qkv_shard(X, Wqkv, bqkv, T, h, t, i, QKV);
        attn_shard_core(QKV, nb, s, h, nh, t, i, O);
        /* the shard's partial of the row-parallel output projection, added
         * to the running sum (the g operator) */
#pragma omp parallel for schedule(static)
        for (long r = 0; r < T; ++r)
            for (long n = 0; n < h; ++n) {
                double acc = 0.0;
                for (long c = i * w; c < (i + 1) * w; ++c) acc += O[r * h + c] * Wo[c * h + n];
                Y[r * h + n] += acc; /* g: sum of partials */
            }
    }
#pragma omp parallel for schedule(static)
    for (long r = 0; r < T; ++r)
        for (long n = 0; n < h; ++n) Y[r * h + n] += bo[n] + R[r * h + n];
    return ORC_OK;
}

int orc_attn_backward(const double* dY, const double* X, const double* Wqkv, const double* bqkv,
                      const double* Wo, long nb, long s, long h, long nh, long t, double* dX,
                      double* dWqkv, double* dbqkv, double* dWo, double* dbo) {
    if (attn_bad(nb, s, h, nh, t)) return ORC_ERR_SHAPE;
    long T = nb * s, w = h / t, d = h / nh, hs = nh / t;
    double* QKV = (double*)calloc((size_t)(T * 3 * h + 1), sizeof(double));
    double* O = (double*)calloc((size_t)(T * h + 1), sizeof(double));
    double* dO = (double*)calloc((size_t)(T * h + 1), sizeof(double));
    double* dQKV = (double*)calloc((size_t)(T * 3 * h + 1), sizeof(double));
    if (!QKV || !O || !dO || !dQKV) {
        free(QKV); free(O); free(dO); free(dQKV);
        return ORC_ERR_ALLOC;
    }
    for (long n = 0; n < h; ++n) {
        double acc = 0.0;
        for (long r = 0; r < T; ++r) acc += dY[r * h + n];
        dbo[n] = acc; /* g backward: the identity */
    }
    for (long e = 0; e < T * h; ++e) dX[e] = 0.0;
    for (long i = 0; i < t; ++i) {
        attn_qkv_shard(X, Wqkv, bqkv, T, h, t, i, QKV);
        attn_shard_core(QKV, nb, s, h, nh, t, i, O);
        /* dO_i = dY Wo_i^T ; dWo_i = O_i^T dY */
#pragma omp parallel for schedule(static)
        for (long r = 0; r < T; ++r)
            for (long c = i * w; c < (i + 1) * w; ++c) {
                double acc = 0.0;
                for (long n = 0; n < h; ++n) acc += dY[r * h + n] * Wo[c * h + n];
                dO[r * h + c] = acc;
            }
#pragma omp parallel for schedule(static)
        for (long c = i * w; c < (i + 1) * w; ++c)
            for (long n = 0; n < h; ++n) {
                double acc = 0.0;
                for (long r = 0; r < T; ++r) acc += O[r * h + c] * dY[r * h + n];
                dWo[c * h + n] = acc;
            }
        /* local attention backward of the shard's heads */
#pragma omp parallel for collapse(2) schedule(dynamic)
        for (long n = 0; n < nb; ++n)
            for (long jj = 0; jj < hs; ++jj) {
                long j = i * hs + jj;
                const double* base = QKV + n * s * 3 * h + j * d;
                double* g = dQKV + n * s * 3 * h + j * d;
                attn_head_backward(base, base + h, base + 2 * h, 3 * h, s, d,
                                   dO + n * s * h + j * d, h, g, g + h, g + 2 * h, 3 * h);
            }
        /* dWqkv_i = X^T dQKV_i ; dbqkv_i = sum_rows dQKV_i */
#pragma omp parallel for schedule(static)
        for (long part = 0; part < 3; ++part)
            for (long c = part * h + i * w; c < part * h + (i + 1) * w; ++c) {
                double acc = 0.0;
                for (long r = 0; r < T; ++r) acc += dQKV[r * 3 * h + c];
                dbqkv[c] = acc;
            }
#pragma omp parallel for schedule(static)
        for (long k = 0; k < h; ++k)
            for (long part = 0; part < 3; ++part)
                for (long c = part * h + i * w; c < part * h + (i + 1) * w; ++c) {
                    double acc = 0.0;
                    for (long r = 0; r < T; ++r) acc += X[r * h + k] * dQKV[r * 3 * h + c];
                    dWqkv[k * 3 * h + c] = acc;
                }
        /* dX += dQKV_i Wqkv_i^T : the shard's partial of the f-operator sum */
#pragma omp parallel for schedule(static)
        for (long r = 0; r < T; ++r)
            for (long k = 0; k < h; ++k) {
                double acc = 0.0;
                for (long part = 0; part < 3; ++part)
                    for (long c = part * h + i * w; c < part * h + (i + 1) * w; ++c)
                        acc += dQKV[r * 3 * h + c] * Wqkv[k * 3 * h + c];
                dX[r * h + k] += acc; /* f: sum of partials */
            }
    }
    free(QKV); free(O); free(dO); free(dQKV);
    return ORC_OK;
}

/* Sampled entry points for full-size workloads: everything of one head j,
 * from the bf16 inputs.  QKV_j [T, 3d] holds head j's Q, K, V columns. */
static void attn_head_qkv_bf16(const uint16_t* X, const uint16_t* Wqkv, const uint16_t* bqkv,
                               long T, long h, long d, long j, double* QKVj) {
#pragma omp parallel for schedule(static)
    for (long r = 0; r < T; ++r) {
        double* out = QKVj + r * 3 * d;
        for (long part = 0; part < 3; ++part)
            for (long e = 0; e < d; ++e) out[part * d + e] = w16(bqkv[part * h + j * d + e]);
        for (long k = 0; k < h; ++k) {
            double x = w16(X[r * h + k]);
            const uint16_t* wrow = Wqkv + k * 3 * h + j * d;
            for (long part = 0; part < 3; ++part)
                for (long e = 0; e < d; ++e) out[part * d + e] += x * w16(wrow[part * h + e]);
        }
    }
}

/* O_j [T, d]: head j's attention output for every sequence. */
int orc_attn_head_bf16(const uint16_t* X, const uint16_t* Wqkv, const uint16_t* bqkv, long nb,
                       long s, long h, long nh, long j, double* Oj) {
    if (attn_bad(nb, s, h, nh, 1) || j < 0 || j >= nh) return ORC_ERR_SHAPE;
    long T = nb * s, d = h / nh;
    double* QKVj = (double*)malloc(sizeof(double) * (size_t)(T * 3 * d + 1));
    if (!QKVj) return ORC_ERR_ALLOC;
    attn_head_qkv_bf16(X, Wqkv, bqkv, T, h, d, j, QKVj);
#pragma omp parallel for schedule(dynamic)
    for (long n = 0; n < nb; ++n) {
        const double* base = QKVj + n * s * 3 * d;
        attn_head_forward(base, base + d, base + 2 * d, 3 * d, s, d, Oj + n * s * d, d, NULL);
    }
    free(QKVj);
    return ORC_OK;
}

/* Head j's parameter gradients: dWqkv_j [h, 3d] (its Q, K, V columns),
 * dbqkv_j [3d] and dWo_j [d, h] (its rows of Wo). */
int orc_attn_head_grads_bf16(const uint16_t* dY, const uint16_t* X, const uint16_t* Wqkv,
                             const uint16_t* bqkv, const uint16_t* Wo, long nb, long s, long h,
                             long nh, long j, double* dWqkvj, double* dbqkvj, double* dWoj) {
    if (attn_bad(nb, s, h, nh, 1) || j < 0 || j >= nh) return ORC_ERR_SHAPE;
    long T = nb * s, d = h / nh;
    double* QKVj = (double*)malloc(sizeof(double) * (size_t)(T * 3 * d + 1));
    double* Oj = (double*)malloc(sizeof(double) * (size_t)(T * d + 1));
    double* dOj = (double*)malloc(sizeof(double) * (size_t)(T * d + 1));
    double* G = (double*)malloc(sizeof(double) * (size_t)(T * 3 * d + 1));
    if (!QKVj || !Oj || !dOj || !G) {
        free(QKVj); free(Oj); free(dOj); free(G);
        return ORC_ERR_ALLOC;
    }
    attn_head_qkv_bf16(X, Wqkv, bqkv, T, h, d, j, QKVj);
#pragma omp parallel for schedule(dynamic)
    for (long n = 0; n < nb; ++n) {
        const double* base = QKVj + n * s * 3 * d;
        attn_head_forward(base, base + d, base + 2 * d, 3 * d, s, d, Oj + n * s * d, d, NULL);
    }
#pragma omp parallel for schedule(static)
    for (long r = 0; r < T; ++r)
        for (long e = 0; e < d; ++e) {
            double acc = 0.0;
            for (long n = 0; n < h; ++n) acc += w16(dY[r * h + n]) * w16(Wo[(j * d + e) * h + n]);
            dOj[r * d + e] = acc;
        }
#pragma omp parallel for schedule(static)
    for (long e = 0; e < d; ++e) {
        double* out = dWoj + e * h;
        for (long n = 0; n < h; ++n) out[n] = 0.0;
        for (long r = 0; r < T; ++r) {
            double o = Oj[r * d + e];
            for (long n = 0; n < h; ++n) out[n] += o * w16(dY[r * h + n]);
        }
    }
#pragma omp parallel for schedule(dynamic)
    for (long n = 0; n < nb; ++n) {
        const double* base = QKVj + n * s * 3 * d;
        double* g = G + n * s * 3 * d;
        attn_head_backward(base, base + d, base + 2 * d, 3 * d, s, d, dOj + n * s * d, d, g,
                           g + d, g + 2 * d, 3 * d);
    }
    for (long c = 0; c < 3 * d; ++c) {
        double acc = 0.0;
        for (long r = 0; r < T; ++r) acc += G[r * 3 * d + c];
        dbqkvj[c] = acc;
    }
#pragma omp parallel for schedule(static)
    for (long k = 0; k < h; ++k) {
        double* out = dWqkvj + k * 3 * d;
        for (long c = 0; c < 3 * d; ++c) out[c] = 0.0;
        for (long r = 0; r < T; ++r) {
            double x = w16(X[r * h + k]);
            for (long c = 0; c < 3 * d; ++c) out[c] += x * G[r * 3 * d + c];
        }
    }
    free(QKVj); free(Oj); free(dOj); free(G);
    return ORC_OK;
}
