/*
 * oracle.c -- scalar C restatement of the F16-weight products (test
 * infrastructure only; see oracle.h for the scope and the citations).
 *
 * Built with: -O2 -std=c11 -ffp-contract=off -fno-fast-math -fopenmp.
 * OpenMP splits whole output elements between threads and never a sum, so the
 * bits do not depend on the thread count.
 */
#include "oracle.h"

#include <math.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#if defined(__BYTE_ORDER__) && (__BYTE_ORDER__ != __ORDER_LITTLE_ENDIAN__)
#error "f16 data is read as little-endian bytes (f16.md, Limitations): little-endian hosts only"
#endif

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/*
 * f32 -> f16, IEEE-754 round to nearest, ties to even, by integer operations on
 * the bit pattern (f16.md, Design notes, "Activation").  Overflow (|x| >= 65520)
 * gives +-inf, f16 subnormal results are kept, f32 subnormals round to +-0.
 * NaN keeps its sign and upper payload and is made quiet (outside the contract).
 */
uint16_t or_to_f16(float x)
{
    uint32_t u = f32_bits(x);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7fffffffu;
    if (a >= 0x7f800000u) {                      /* inf or NaN */
        if (a == 0x7f800000u) return sign | 0x7c00u;
        return (uint16_t)(sign | 0x7e00u | ((a & 0x007fffffu) >> 13));
    }
    if (a >= 0x477ff000u) return sign | 0x7c00u; /* 65520 and above round to inf */
    uint32_t e = a >> 23;                        /* biased f32 exponent */
    uint32_t m = a & 0x007fffffu;
    if (e >= 113) {                              /* result is a normal f16 (>= 2^-14) */
        uint32_t h = ((e - 112) << 10) | (m >> 13);
        uint32_t rem = m & 0x1fffu;
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1; /* carry may bump the exponent */
        return (uint16_t)(sign | h);
    }
    /* subnormal f16 result, counted in units of 2^-24: value = M * 2^(e-150) */
    if (e < 102) return sign;                    /* below 2^-25: rounds to zero */
    uint32_t M = m | 0x00800000u;
    uint32_t shift = 126 - e;                    /* 14 .. 24 */
    uint32_t q = M >> shift;
    uint32_t rem = M & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1u))) q += 1; /* may become 0x400, the least normal */
    return (uint16_t)(sign | q);
}

/* f16 -> f32, exact (f16.md, Technical usage, "widen"). */
float or_widen(uint16_t h)
{
    uint32_t s = (uint32_t)(h >> 15) & 1u;
    uint32_t e = (uint32_t)(h >> 10) & 0x1fu;
    uint32_t m = (uint32_t)h & 0x3ffu;
    if (e == 0) {
        float v = (float)m * 0x1p-24f;           /* m < 2^10: exact, includes +-0 */
        return s ? -v : v;
    }
    if (e == 31) return bits_f32((s << 31) | 0x7f800000u | (m << 13));
    return bits_f32((s << 31) | ((e + 112u) << 23) | (m << 13));
}

/*
 * ggml_vec_dot_f16 as the page states it (f16.md, Design notes, "vec_dot"):
 * element i < 32*floor(k/32) goes to accumulator j = (i%32)/8, lane l = i%8, and
 * each of those 32 chains adds its products in increasing i from +0.0f.  The four
 * accumulators are combined lane-wise as (a0+a2)+(a1+a3); the low four lanes are
 * added to the high four; two horizontal adds leave (t0+t1)+(t2+t3).  That f32
 * value is widened to double and the k%32 tail products are added to it in
 * order, in double; the double is rounded once to f32.
 */
float or_vec_dot_ref(const uint16_t *w, const uint16_t *a, int64_t k)
{
    float acc[4][8];
    for (int j = 0; j < 4; j++)
        for (int l = 0; l < 8; l++) acc[j][l] = 0.0f;
    int64_t k32 = k - k % 32;
    for (int64_t s = 0; s < k32; s += 32)
        for (int j = 0; j < 4; j++)
            for (int l = 0; l < 8; l++) {
                int64_t i = s + 8 * j + l;
                acc[j][l] = acc[j][l] + or_widen(w[i]) * or_widen(a[i]);
            }
    float v[8];
    for (int l = 0; l < 8; l++) v[l] = (acc[0][l] + acc[2][l]) + (acc[1][l] + acc[3][l]);
    float t[4];
    for (int m = 0; m < 4; m++) t[m] = v[m] + v[m + 4];     /* low half + high half */
    float h0 = t[0] + t[1];                                 /* first horizontal add */
    float h1 = t[2] + t[3];
    float r = h0 + h1;                                      /* second horizontal add */
    double sumf = (double)r;
    for (int64_t i = k32; i < k; i++) sumf += (double)(or_widen(w[i]) * or_widen(a[i]));
    return (float)sumf;
}

/*
 * One tinyBLAS element (f16.md, Design notes, "sgemm_dot"): lane q = i%8 adds the
 * products of elements q, q+8, q+16, ... in increasing order from +0.0f; then
 * hsum ((l0+l4)+(l2+l6))+((l1+l5)+(l3+l7)).  Requires k%8 == 0 (returns NaN
 * otherwise: the path is never taken for such k).
 */
float or_sgemm_dot_ref(const uint16_t *w, const uint16_t *a, int64_t k)
{
    if (k % 8 != 0) return NAN;
    float l[8];
    for (int q = 0; q < 8; q++) l[q] = 0.0f;
    for (int64_t i = 0; i < k; i += 8)
        for (int q = 0; q < 8; q++) l[q] = l[q] + or_widen(w[i + q]) * or_widen(a[i + q]);
    return ((l[0] + l[4]) + (l[2] + l[6])) + ((l[1] + l[5]) + (l[3] + l[7]));
}

/* ggml's path selector (f16.md, Technical usage). */
int or_takes_sgemm(int64_t rows, int64_t k, int64_t n)
{
    return n >= 2 && rows % 4 == 0 && k % 8 == 0;
}

/* sum |w_i * a_i| in double: the scale of the tensor-core tolerance. */
double or_abs_dot(const uint16_t *w, const uint16_t *a, int64_t k)
{
    double s = 0.0;
    for (int64_t i = 0; i < k; i++) s += fabs((double)or_widen(w[i]) * (double)or_widen(a[i]));
    return s;
}

void or_to_f16_array(const float *x, uint16_t *h, int64_t n)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) h[i] = or_to_f16(x[i]);
}

void or_widen_array(const uint16_t *h, float *x, int64_t n)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) x[i] = or_widen(h[i]);
}

/* One column: vec_dot per row (f16.md, Matrix products, "mat_vec_par"). */
void or_matvec(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *x, float *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) y[r] = or_vec_dot_ref(W + r * k, x, k);
}

/* Several matrices by one column: every output row is still one vec_dot
 * (f16.md, Matrix products, "mat_vec_multi_par"). */
void or_matvec_multi(int nmat, const uint16_t *const *W, const int64_t *rows, int64_t k,
                     const uint16_t *x, float *const *y)
{
    for (int m = 0; m < nmat; m++) or_matvec(W[m], rows[m], k, x, y[m]);
}

/* Several columns: out[c*rows + r], sgemm_dot when takes_sgemm, else vec_dot
 * (f16.md, Matrix products, "mat_mul_par"). */
void or_matmul(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols,
               float *Y)
{
    int sg = or_takes_sgemm(rows, k, ncols);
    int64_t total = rows * ncols;
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < total; e++) {
        int64_t c = e / rows, r = e % rows;
        const uint16_t *w = W + r * k, *a = X + c * k;
        Y[e] = sg ? or_sgemm_dot_ref(w, a, k) : or_vec_dot_ref(w, a, k);
    }
}

void or_matmul_sample(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X,
                      int64_t ncols, const int64_t *r_idx, const int64_t *c_idx, int64_t n,
                      float *out, double *absdot)
{
    int sg = or_takes_sgemm(rows, k, ncols);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) {
        const uint16_t *w = W + r_idx[i] * k, *a = X + c_idx[i] * k;
        out[i] = sg ? or_sgemm_dot_ref(w, a, k) : or_vec_dot_ref(w, a, k);
        if (absdot) absdot[i] = or_abs_dot(w, a, k);
    }
}

void or_abs_matmul(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X,
                   int64_t ncols, double *out)
{
    int64_t total = rows * ncols;
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < total; e++) {
        int64_t c = e / rows, r = e % rows;
        out[e] = or_abs_dot(W + r * k, X + c * k, k);
    }
}

int64_t or_check_to_f16_vs_compiler(uint64_t lo, uint64_t hi, uint32_t *first_bad)
{
    int64_t bad = 0;
    uint64_t first = UINT64_MAX;
#pragma omp parallel for schedule(static) reduction(+ : bad) reduction(min : first)
    for (uint64_t p = lo; p < hi; p++) {
        float x = bits_f32((uint32_t)p);
        if (isnan(x)) continue;
        _Float16 hc = (_Float16)x;
        uint16_t hb;
        memcpy(&hb, &hc, 2);
        if (hb != or_to_f16(x)) {
            bad++;
            if (p < first) first = p;
        }
    }
    if (first_bad) *first_bad = (first == UINT64_MAX) ? 0u : (uint32_t)first;
    return bad;
}

/*
 * rms_norm then mul of one row of n f32 values by an f32 weight (page
 * "docs/modules/forward.md", Technical usage, "Other public pieces": the sum of
 * squares in double, no FMA; Design notes, step three: the first RMS norm with its
 * weight gives attn_norm-0).  Readings where the page is silent:
 *   - each square is one f32 multiply (the row's own type), widened to double and
 *     added in index order to a double sum that starts at +0;
 *   - the mean is sum / n divided in double, then rounded to f32;
 *   - scale = 1 / sqrt(mean + eps): an f32 add, a correctly rounded f32 square root
 *     and an f32 division;
 *   - out[i] = (x[i] * scale) * w[i]: two f32 multiplies, each rounded.
 * A zero row with eps == 0 gives 0 * inf = NaN, as the formula does.
 */
void or_rms_norm_mul(const float *x, const float *w, int64_t n, float eps, float *out)
{
    double sum = 0.0;
    for (int64_t i = 0; i < n; i++) {
        float sq = x[i] * x[i];
        sum += (double)sq;
    }
    float mean = (float)(sum / (double)n);
    float scale = 1.0f / sqrtf(mean + eps);
    for (int64_t i = 0; i < n; i++) {
        float y = x[i] * scale;
        out[i] = y * w[i];
    }
}

void or_rms_norm_mul_rows(const float *X, const float *w, int64_t rows, int64_t n, float eps, float *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) or_rms_norm_mul(X + r * n, w, n, eps, out + r * n);
}

/* mad and scale (page "docs/modules/f16.md", Technical usage: `mad` is
 * ggml_vec_mad_f16, the V accumulator of flash attention; `scale` is
 * ggml_vec_scale_f16), element by element in index order.  mad's product and sum
 * round once together (C99 fmaf is correctly rounded); scale is one f32 multiply
 * (this file is compiled with -ffp-contract=off, so nothing else is fused).  Both
 * results go to f16 by or_to_f16 (nearest-even). */
void or_f16_mad(uint16_t *acc, const uint16_t *v, float w, int64_t n)
{
    for (int64_t i = 0; i < n; i++) acc[i] = or_to_f16(fmaf(or_widen(v[i]), w, or_widen(acc[i])));
}

void or_f16_scale(uint16_t *acc, float s, int64_t n)
{
    for (int64_t i = 0; i < n; i++) acc[i] = or_to_f16(or_widen(acc[i]) * s);
}

int or_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void or_set_threads(int n)
{
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : 1);
#else
    (void)n;
#endif
}
