/*
 * oracle/swiglu_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU statement of what the fused gate-up
 * SwiGLU computes.  It exists to check the CUDA library against; nothing in the
 * product path may link or call it (only the tests, the smoke check and the
 * bench's CPU-baseline leg do).  It shares no code, header or constant with the
 * CUDA side.
 *
 * Source of each step (Liger-Kernel Megatron SwiGLU page):
 *   - layout, §Background: Megatron's linear_fc1 emits one [tokens, 2n] buffer,
 *     gate in columns [0, n), up in [n, 2n); the fused kernel reads both halves
 *     through a column offset, input row stride 2n, output row stride n.
 *   - activation, §Summary / §Background: SwiGLU as Megatron's bias_swiglu_impl
 *     computes it with bias=None, y = silu(gate) * up, silu(g) = g * sigmoid(g).
 *   - backward, §What's added / §Optional in_place: the backward works from the
 *     saved fc1 buffer (recomputing sigmoid) and writes d(gate) into [0, n) and
 *     d(up) into [n, 2n).  The page prints no formula; the one used is the
 *     analytic derivative of silu(g) * u:
 *        d(gate) = dy * u * s * (1 + g * (1 - s)),   d(up) = dy * g * s,
 *     with s = 1 / (1 + exp(-g)).
 *
 * Arithmetic: every input is widened exactly to double (bf16 -> fp32 -> double
 * are exact), the formulas above are evaluated in double with libm exp, and each
 * result is rounded once to the storage type, round-to-nearest-even.  The bf16
 * rounding is done directly from the double (no intermediate fp32 rounding).
 * No blocking, fusion or reordering: one loop over rows, one over columns.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no fast-math, no
 * FMA contraction, so x86 and Arm hosts give the same bits).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F64 2

#define ORACLE_OK 0
#define ORACLE_BAD_ARG -1

/* ---- storage types ------------------------------------------------------ */

static double bf16_bits_to_double(uint16_t h) {
    uint32_t bits = ((uint32_t)h) << 16; /* bf16 is the top half of an fp32 */
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (8 exponent bits, 8 significand bits
 * including the hidden one), ties to even, in one step.  The spacing of bf16
 * numbers in [2^k, 2^(k+1)) is 2^(k-7) for k >= -126, and 2^-133 in the
 * subnormal range below 2^-126. */
uint16_t oracle_bf16_from_double(double v) {
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v)) return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(v);
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e); /* a in [2^(e-1), 2^e) */
    int k = e - 1;
    if (k < -126) k = -126;
    double spacing = ldexp(1.0, k - 7);
    double q = nearbyint(a / spacing); /* a / spacing is exact; ties to even */
    double r = q * spacing;
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u); /* overflow */
    float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

static double load_elem(const void *base, int64_t idx, int dtype) {
    const char *p = (const char *)base;
    if (dtype == ORACLE_F32) {
        float f;
        memcpy(&f, p + idx * 4, 4);
        return (double)f;
    }
    if (dtype == ORACLE_BF16) {
        uint16_t h;
        memcpy(&h, p + idx * 2, 2);
        return bf16_bits_to_double(h);
    }
    double d;
    memcpy(&d, p + idx * 8, 8);
    return d;
}

static void store_elem(void *base, int64_t idx, int dtype, double v) {
    char *p = (char *)base;
    if (dtype == ORACLE_F32) {
        float f = (float)v; /* IEEE conversion, round to nearest even */
        memcpy(p + idx * 4, &f, 4);
    } else if (dtype == ORACLE_BF16) {
        uint16_t h = oracle_bf16_from_double(v);
        memcpy(p + idx * 2, &h, 2);
    } else {
        memcpy(p + idx * 8, &v, 8);
    }
}

/* ---- the method, one element pair at a time ------------------------------ */

static double sigmoid(double g) { return 1.0 / (1.0 + exp(-g)); }

/* forward: y = silu(g) * u = g * s * u */
static double swiglu_fwd_pair(double g, double u) {
    double s = sigmoid(g);
    return g * s * u;
}

/* backward: the derivative of g * s(g) * u with respect to g and to u, times dy */
static void swiglu_bwd_pair(double dy, double g, double u, double *dgate, double *dup) {
    double s = sigmoid(g);
    *dgate = dy * u * s * (1.0 + g * (1.0 - s));
    *dup = dy * g * s;
}

/* ---- the layouts ----------------------------------------------------------- */

static int check_args(int64_t rows, int64_t n, int dtype) {
    if (rows < 0 || n < 0) return ORACLE_BAD_ARG;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F64) return ORACLE_BAD_ARG;
    return ORACLE_OK;
}

/* x: [rows, 2n] with row stride sx (elements); y: [rows, n] with row stride sy. */
int oracle_swiglu_fwd(const void *x, void *y, int64_t rows, int64_t n, int64_t sx, int64_t sy,
                      int dtype) {
    if (check_args(rows, n, dtype)) return ORACLE_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < n; ++j) {
            double g = load_elem(x, r * sx + j, dtype);
            double u = load_elem(x, r * sx + n + j, dtype);
            store_elem(y, r * sy + j, dtype, swiglu_fwd_pair(g, u));
        }
    }
    return ORACLE_OK;
}

/* dy: [rows, n] (stride sdy); x: [rows, 2n] (stride sx); dx: [rows, 2n] (stride
 * sdx) receives d(gate) in [0, n) and d(up) in [n, 2n).  dx may be x itself (the
 * in-place backward): each pair is read before it is written. */
int oracle_swiglu_bwd(const void *dy, const void *x, void *dx, int64_t rows, int64_t n,
                      int64_t sdy, int64_t sx, int64_t sdx, int dtype) {
    if (check_args(rows, n, dtype)) return ORACLE_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < n; ++j) {
            double d = load_elem(dy, r * sdy + j, dtype);
            double g = load_elem(x, r * sx + j, dtype);
            double u = load_elem(x, r * sx + n + j, dtype);
            double dg, du;
            swiglu_bwd_pair(d, g, u, &dg, &du);
            store_elem(dx, r * sdx + j, dtype, dg);
            store_elem(dx, r * sdx + n + j, dtype, du);
        }
    }
    return ORACLE_OK;
}

/* ---- the two-tensor formulation ------------------------------------------- */
/* Liger-Kernel Megatron SwiGLU page, §Background: Liger's earlier SwiGLU takes
 * the gate a and the up projection b as two separate tensors, as HuggingFace
 * models produce them.  Same arithmetic, separate buffers:
 *   c[r, j] = silu(a[r, j]) * b[r, j]
 *   da[r, j] = dc * b * s * (1 + a (1 - s)),   db[r, j] = dc * a * s.
 * da may be a and db may be b (each pair is read before it is written). */
int oracle_silu_mul_fwd(const void *a, const void *b, void *c, int64_t rows, int64_t n,
                        int64_t sa, int64_t sb, int64_t sc, int dtype) {
    if (check_args(rows, n, dtype)) return ORACLE_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < n; ++j) {
            double g = load_elem(a, r * sa + j, dtype);
            double u = load_elem(b, r * sb + j, dtype);
            store_elem(c, r * sc + j, dtype, swiglu_fwd_pair(g, u));
        }
    }
    return ORACLE_OK;
}

int oracle_silu_mul_bwd(const void *dc, const void *a, const void *b, void *da, void *db,
                        int64_t rows, int64_t n, int64_t sdc, int64_t sa, int64_t sb,
                        int64_t sda, int64_t sdb, int dtype) {
    if (check_args(rows, n, dtype)) return ORACLE_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < n; ++j) {
            double d = load_elem(dc, r * sdc + j, dtype);
            double g = load_elem(a, r * sa + j, dtype);
            double u = load_elem(b, r * sb + j, dtype);
            double dg, du;
            swiglu_bwd_pair(d, g, u, &dg, &du);
            store_elem(da, r * sda + j, dtype, dg);
            store_elem(db, r * sdb + j, dtype, du);
        }
    }
    return ORACLE_OK;
}

/* ---- per-token weights and bias ------------------------------------------ */
/* Liger-Kernel Megatron SwiGLU page, §Known issues 2: Megatron's MoE routed
 * experts scale each token's activation by its routing weight
 * (weighted_bias_swiglu_impl needs a per_token_scale-aware kernel); §Scope:
 * the fused path has no bias and falls back when one is given.  Both are
 * stated here by their plain definitions:
 *
 *   weighted:  y[r, j] = w[r] * silu(g) * u
 *              d gate = dy * w[r] * u * s * (1 + g (1 - s)),  d up = dy * w[r] * g * s
 *              dw[r]  = sum_j dy[r, j] * silu(g[r, j]) * u[r, j]
 *   bias:      z_g = g + bias[j], z_u = u + bias[n + j];  y = silu(z_g) * z_u
 *              dx = the plain backward evaluated at (z_g, z_u)
 *              dbias[k] = sum_r dx[r, k]   (k < 2n, the exact dx before rounding)
 *
 * w and dw are fp32 [rows] (unit stride); bias and dbias have x's dtype, [2n].
 * Sums are accumulated in double and rounded once. */

int oracle_swiglu_weighted_fwd(const void *x, const float *w, void *y, int64_t rows, int64_t n,
                               int64_t sx, int64_t sy, int dtype) {
    if (check_args(rows, n, dtype)) return ORACLE_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        double wr = (double)w[r];
        for (int64_t j = 0; j < n; ++j) {
            double g = load_elem(x, r * sx + j, dtype);
            double u = load_elem(x, r * sx + n + j, dtype);
            store_elem(y, r * sy + j, dtype, wr * swiglu_fwd_pair(g, u));
        }
    }
    return ORACLE_OK;
}

int oracle_swiglu_weighted_bwd(const void *dy, const void *x, const float *w, void *dx, float *dw,
                               int64_t rows, int64_t n, int64_t sdy, int64_t sx, int64_t sdx,
                               int dtype) {
    if (check_args(rows, n, dtype)) return ORACLE_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        double wr = (double)w[r];
        double acc = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            double d = load_elem(dy, r * sdy + j, dtype);
            double g = load_elem(x, r * sx + j, dtype);
            double u = load_elem(x, r * sx + n + j, dtype);
            double dg, du;
            acc += d * swiglu_fwd_pair(g, u);
            swiglu_bwd_pair(d * wr, g, u, &dg, &du);
            store_elem(dx, r * sdx + j, dtype, dg);
            store_elem(dx, r * sdx + n + j, dtype, du);
        }
        dw[r] = (float)acc;
    }
    return ORACLE_OK;
}

int oracle_swiglu_bias_fwd(const void *x, const void *bias, void *y, int64_t rows, int64_t n,
                           int64_t sx, int64_t sy, int dtype) {
    if (check_args(rows, n, dtype)) return ORACLE_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < n; ++j) {
            double g = load_elem(x, r * sx + j, dtype) + load_elem(bias, j, dtype);
            double u = load_elem(x, r * sx + n + j, dtype) + load_elem(bias, n + j, dtype);
            store_elem(y, r * sy + j, dtype, swiglu_fwd_pair(g, u));
        }
    }
    return ORACLE_OK;
}

/* dbias needs the unrounded dx of every row; `acc` is caller-provided
 * scratch of 2n doubles (the oracle keeps its own arithmetic simple rather
 * than allocate). */
int oracle_swiglu_bias_bwd(const void *dy, const void *x, const void *bias, void *dx, void *dbias,
                           double *acc, int64_t rows, int64_t n, int64_t sdy, int64_t sx,
                           int64_t sdx, int dtype) {
    if (check_args(rows, n, dtype)) return ORACLE_BAD_ARG;
    for (int64_t k = 0; k < 2 * n; ++k) acc[k] = 0.0;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < n; ++j) {
            double d = load_elem(dy, r * sdy + j, dtype);
            double g = load_elem(x, r * sx + j, dtype) + load_elem(bias, j, dtype);
            double u = load_elem(x, r * sx + n + j, dtype) + load_elem(bias, n + j, dtype);
            double dg, du;
            swiglu_bwd_pair(d, g, u, &dg, &du);
            acc[j] += dg;
            acc[n + j] += du;
            store_elem(dx, r * sdx + j, dtype, dg);
            store_elem(dx, r * sdx + n + j, dtype, du);
        }
    }
    for (int64_t k = 0; k < 2 * n; ++k) store_elem(dbias, k, dtype, acc[k]);
    return ORACLE_OK;
}

/* ---- linear_fc1 followed by the activation -------------------------------- */
/* Liger-Kernel Megatron SwiGLU page, §Background: the [s, b, 2n] buffer is the
 * output of Megatron's linear_fc1 (a ColumnParallelLinear), i.e. fc1 = X W^T with
 * W the [2n, K] weight whose rows [0, n) produce the gate and [n, 2n) the up
 * projection.  Stated plainly (bias-free, as the fused path requires):
 *   fc1[m, c] = sum_k X[m, k] * W[c, k]        (c < 2n, exact sum in double)
 *   y[m, j]   = silu(fc1[m, j]) * fc1[m, n + j]
 * y is rounded once to the storage type; when x_out is not NULL the
 * pre-activation fc1 is also returned (rounded once), as a training step saves
 * it for the backward.  X: [M, K], W: [2n, K], both row-major with unit column
 * stride; `acc` is caller scratch of 2n doubles. */
int oracle_fc1_swiglu_fwd(const void *X, const void *W, void *y, void *x_out, double *acc,
                          int64_t M, int64_t n, int64_t K, int dtype) {
    if (check_args(M, n, dtype) || K < 0) return ORACLE_BAD_ARG;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t c = 0; c < 2 * n; ++c) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k)
                s += load_elem(X, m * K + k, dtype) * load_elem(W, c * K + k, dtype);
            acc[c] = s;
        }
        for (int64_t j = 0; j < n; ++j) {
            store_elem(y, m * n + j, dtype, swiglu_fwd_pair(acc[j], acc[n + j]));
            if (x_out != NULL) {
                store_elem(x_out, m * 2 * n + j, dtype, acc[j]);
                store_elem(x_out, m * 2 * n + n + j, dtype, acc[n + j]);
            }
        }
    }
    return ORACLE_OK;
}

/* ---- per-token weights and bias together ------------------------------------ */
/* Megatron's routed-expert activation with a bias (the weighted_bias_swiglu_impl
 * the page names in §Known issues 2, bias given): both of the above at once,
 *   y = w[r] * silu(g + bias[j]) * (u + bias[n + j])
 *   dx = the plain backward at the shifted values with dy scaled by w[r]
 *   dw[r] = sum_j dy * silu(g + bias[j]) * (u + bias[n + j])
 *   dbias[k] = sum_r dx[r, k]   (exact, before rounding)
 * `acc` is caller scratch of 2n doubles. */
int oracle_swiglu_weighted_bias_fwd(const void *x, const void *bias, const float *w, void *y,
                                    int64_t rows, int64_t n, int64_t sx, int64_t sy, int dtype) {
    if (check_args(rows, n, dtype)) return ORACLE_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        double wr = (double)w[r];
        for (int64_t j = 0; j < n; ++j) {
            double g = load_elem(x, r * sx + j, dtype) + load_elem(bias, j, dtype);
            double u = load_elem(x, r * sx + n + j, dtype) + load_elem(bias, n + j, dtype);
            store_elem(y, r * sy + j, dtype, wr * swiglu_fwd_pair(g, u));
        }
    }
    return ORACLE_OK;
}

int oracle_swiglu_weighted_bias_bwd(const void *dy, const void *x, const void *bias,
                                    const float *w, void *dx, void *dbias, float *dw, double *acc,
                                    int64_t rows, int64_t n, int64_t sdy, int64_t sx, int64_t sdx,
                                    int dtype) {
    if (check_args(rows, n, dtype)) return ORACLE_BAD_ARG;
    for (int64_t k = 0; k < 2 * n; ++k) acc[k] = 0.0;
    for (int64_t r = 0; r < rows; ++r) {
        double wr = (double)w[r];
        double sum = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            double d = load_elem(dy, r * sdy + j, dtype);
            double g = load_elem(x, r * sx + j, dtype) + load_elem(bias, j, dtype);
            double u = load_elem(x, r * sx + n + j, dtype) + load_elem(bias, n + j, dtype);
            double dg, du;
            sum += d * swiglu_fwd_pair(g, u);
            swiglu_bwd_pair(d * wr, g, u, &dg, &du);
            acc[j] += dg;
            acc[n + j] += du;
            store_elem(dx, r * sdx + j, dtype, dg);
            store_elem(dx, r * sdx + n + j, dtype, du);
        }
        dw[r] = (float)sum;
    }
    for (int64_t k = 0; k < 2 * n; ++k) store_elem(dbias, k, dtype, acc[k]);
    return ORACLE_OK;
}
