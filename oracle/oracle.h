/*
 * oracle.h -- plain, slow, scalar C restatement of the F16-weight products.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this code: only tests/, the smoke check and the bench's CPU-baseline leg
 * do.  It shares no header, helper, table or constant with the CUDA library.
 *
 * What it restates (page "docs/modules/f16.md", bankML):
 *   - to_f16        : section "Design notes", bullet "Activation" -- f32 rounded
 *                     to f16 with round-to-nearest-even before any product.
 *   - widen         : section "Technical usage" -- exact f16 -> f32.
 *   - vec_dot_ref   : section "Design notes", bullet "vec_dot" -- four 8-lane
 *                     f32 accumulators over 32-element steps, reduced
 *                     (a0+a2)+(a1+a3), low half + high half, two horizontal
 *                     adds, then the n%32 tail added in double.
 *   - sgemm_dot_ref : section "Design notes", bullet "sgemm_dot" -- one 8-lane
 *                     FMA chain over the row, hsum ((l0+l4)+(l2+l6))+((l1+l5)+(l3+l7)).
 *   - takes_sgemm   : section "Technical usage" -- n>=2 && rows%4==0 && k%8==0.
 *   - matvec, matvec_multi, matmul : section "Matrix products"
 *                     (out[c*rows + r]; sgemm_dot when takes_sgemm, else vec_dot).
 *
 * and (page "docs/modules/forward.md", bankML):
 *   - rms_norm_mul  : section "Technical usage", "Other public pieces" -- rms_norm
 *                     then mul, the sum of squares in double, no FMA (the readings
 *                     of the steps the page leaves open are listed in oracle.c).
 *
 * Every f16 x f16 product is exact in f32 (11-bit significands, exponents well
 * inside the f32 normal range), so an FMA and a multiply-then-add give the same
 * bits; this file uses plain '*' and '+' and is built with -ffp-contract=off.
 *
 * Parity with the shipped ggml binary itself is unpinned (no such binary or
 * recorded vectors exist here); each function is pinned instead by the tests in
 * tests/test_oracle_*.py against closed forms, hand-derived examples and exact
 * rational brute force.
 */
#ifndef BM_ORACLE_H
#define BM_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

uint16_t or_to_f16(float x);
float    or_widen(uint16_t h);
float    or_vec_dot_ref(const uint16_t *w, const uint16_t *a, int64_t k);
float    or_sgemm_dot_ref(const uint16_t *w, const uint16_t *a, int64_t k);
int      or_takes_sgemm(int64_t rows, int64_t k, int64_t n);
double   or_abs_dot(const uint16_t *w, const uint16_t *a, int64_t k);

void or_to_f16_array(const float *x, uint16_t *h, int64_t n);
void or_widen_array(const uint16_t *h, float *x, int64_t n);
void or_matvec(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *x, float *y);
void or_matvec_multi(int nmat, const uint16_t *const *W, const int64_t *rows, int64_t k,
                     const uint16_t *x, float *const *y);
void or_matmul(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols,
               float *Y);
/* Elements (r_idx[i], c_idx[i]) of the product W(rows x k) . X(ncols x k) with the
 * path the full product's shape selects; also returns sum |w.a| per element. */
void or_matmul_sample(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X,
                      int64_t ncols, const int64_t *r_idx, const int64_t *c_idx, int64_t n,
                      float *out, double *absdot);
/* Sum |w.a| in double for every element, laid out as out[c*rows + r]. */
void or_abs_matmul(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X,
                   int64_t ncols, double *out);

/* rms_norm then mul: out = (x * (1 / sqrt(mean(x^2) + eps))) * w, one row of n
 * values, or `rows` rows of n values laid out one after another. */
void or_rms_norm_mul(const float *x, const float *w, int64_t n, float eps, float *out);
void or_rms_norm_mul_rows(const float *X, const float *w, int64_t rows, int64_t n, float eps,
                          float *out);

/* The attention-side accumulator helpers (page "docs/modules/f16.md", Technical usage:
 * `mad` is ggml_vec_mad_f16, flash attention's V accumulator; `scale` is
 * ggml_vec_scale_f16).  In place on acc[0..n):
 *   or_f16_mad:   acc[i] = to_f16(fmaf(widen(v[i]), w, widen(acc[i])))
 *   or_f16_scale: acc[i] = to_f16(widen(acc[i]) * s)
 * Reading where the page is silent: mad rounds once in f32 (a fused multiply-add, as
 * ggml's F16C + FMA path does), then to f16 nearest-even. */
void or_f16_mad(uint16_t *acc, const uint16_t *v, float w, int64_t n);
void or_f16_scale(uint16_t *acc, float s, int64_t n);

/* Exhaustive self-checks over every f32 bit pattern in [lo, hi): returns the
 * number of non-NaN inputs whose or_to_f16 differs from the C compiler's own
 * _Float16 conversion, and stores the first such pattern in *first_bad. */
int64_t or_check_to_f16_vs_compiler(uint64_t lo, uint64_t hi, uint32_t *first_bad);
int     or_threads(void);
/* Threads the row loops use from now on (n < 1 counts as 1); timing only, never results. */
void    or_set_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
