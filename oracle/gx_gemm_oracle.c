/*
 * CPU oracle of the gx_gemm step update -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the bench's CPU-baseline leg use this file. The CUDA library never links,
 * loads or calls it, and it shares no code with the library.
 *
 * What it computes (sparse_delta_memory/cuda/gx_gemm_cuda.py, the module docstring's step formula, and the kernel's
 * fixed chain and epilogue in gx_gemm_kernel): for one step ti, every chunk n = ti*P + p (p < P), every row i < C and
 * every column c < hd:
 *
 *     acc = +0;  for j = 0, 1, .., C-1:  acc = fmaf(x[n, j, i], d_dv[n, j, c], acc);
 *     d_u[n, i, c] = d_u[n, i, c] + acc            (one more IEEE round-to-nearest-even rounding)
 *
 * It is the definition written out: a plain loop nest with no blocking, no reordering and no vectorisation.
 * Compile flags: -O2 -ffp-contract=off, no fast-math, so that `+` stays a separately rounded add and no FTZ/DAZ mode
 * is switched on. fmaf() is C99's correctly rounded fused multiply-add. Both properties are checked at run time
 * (oracle_fp_env_ok) before any result is trusted.
 *
 * Strides are in elements: x[n, j, i] is at x[n*x_sn + j*x_sj + i]; d_dv[n, j, c] at d_dv[n*dv_sn + j*dv_sj + c];
 * d_u[n, i, c] at d_u[n*du_sn + i*du_si + c].
 */
#include <math.h>
#include <stdint.h>

/* 1 if this thread computes with gradual underflow (no FTZ / DAZ) and fmaf is a fused, singly rounded operation. */
int oracle_fp_env_ok(void) {
    volatile float tiny = 1e-38f, scale = 1e-3f;
    volatile float den = tiny * scale;                 /* ~1e-41: a subnormal, zero under FTZ */
    if (!(den > 0.0f)) return 0;
    volatile float d2 = den;                           /* a subnormal operand must not be read as zero (DAZ) */
    if (!(d2 + d2 > 0.0f)) return 0;
    /* fused: (1 + 2^-23) * (1 - 2^-23) - 1 = -2^-46 exactly; an unfused product rounds to 1 and gives 0 */
    volatile float a = 1.0f + 0x1p-23f, b = 1.0f - 0x1p-23f, m1 = -1.0f;
    if (fmaf(a, b, m1) != -0x1p-46f) return 0;
    /* the chain starts from +0: a -0 product plus +0 is +0 under round-to-nearest */
    volatile float nz = -1.0f, z = 0.0f;
    float r = fmaf(nz, z, 0.0f);
    if (signbit(r)) return 0;
    return 1;
}

/* One output element: the fixed j-order chain from +0, then the separately rounded add to the old d_u value. */
float oracle_gx_gemm_element(const float *x, const float *d_dv, float du_old, int64_t n, int64_t i, int64_t c,
                             int64_t C, int64_t x_sn, int64_t x_sj, int64_t dv_sn, int64_t dv_sj) {
    float acc = 0.0f;
    for (int64_t j = 0; j < C; ++j) {
        acc = fmaf(x[n * x_sn + j * x_sj + i], d_dv[n * dv_sn + j * dv_sj + c], acc);
    }
    return du_old + acc;
}

/* One step ti over chunks ti*P .. ti*P + P - 1, in place on d_u. Returns 0, or -1 if the FP environment is wrong. */
int oracle_gx_gemm_step(float *d_u, const float *x, const float *d_dv, int64_t ti, int64_t P, int64_t C, int64_t hd,
                        int64_t x_sn, int64_t x_sj, int64_t dv_sn, int64_t dv_sj, int64_t du_sn, int64_t du_si) {
    if (!oracle_fp_env_ok()) return -1;
    for (int64_t p = 0; p < P; ++p) {
        const int64_t n = ti * P + p;
        for (int64_t i = 0; i < C; ++i) {
            for (int64_t c = 0; c < hd; ++c) {
                float *o = &d_u[n * du_sn + i * du_si + c];
                *o = oracle_gx_gemm_element(x, d_dv, *o, n, i, c, C, x_sn, x_sj, dv_sn, dv_sj);
            }
        }
    }
    return 0;
}

/* Selected outputs only (parity at full size): for k < count, out[k] = the updated value of d_u[n[k], i[k], c[k]]
 * (d_u itself is not modified). */
int oracle_gx_gemm_points(float *out, const float *d_u, const float *x, const float *d_dv, const int64_t *pn,
                          const int64_t *pi, const int64_t *pc, int64_t count, int64_t C, int64_t x_sn, int64_t x_sj,
                          int64_t dv_sn, int64_t dv_sj, int64_t du_sn, int64_t du_si) {
    if (!oracle_fp_env_ok()) return -1;
    for (int64_t k = 0; k < count; ++k) {
        const float old = d_u[pn[k] * du_sn + pi[k] * du_si + pc[k]];
        out[k] = oracle_gx_gemm_element(x, d_dv, old, pn[k], pi[k], pc[k], C, x_sn, x_sj, dv_sn, dv_sj);
    }
    return 0;
}
