// bm_norm.cuh -- rms_norm then mul (page "docs/modules/forward.md", Technical
// usage, "Other public pieces": rms_norm, then a multiply by the norm weight,
// the sum of squares in double, no FMA), the device steps every kernel that
// normalises a row shares.
//
//   q_i   = x_i * x_i                          (f32 multiply)
//   mean  = the mean of the q_i, rounded once to f32 (below)
//   scale = 1 / sqrt(mean + eps)               (f32 add, square root, divide; IEEE)
//   out_i = (x_i * scale) * g_i                (two f32 multiplies)
//
// The mean.  The page sums the squares in double; an index-order double sum of k
// terms lies within (k - 1) * 2^-53 (relative) of the exact sum, and the f32 mean
// taken from it can differ from the exact one only when the exact mean is that
// close to an f32 rounding boundary.  Here the mean is the exact one, up to a
// much smaller error, rounded once: no FP64 arithmetic at all (this part's FP64
// pipe retires about one operation per clock per SM, microseconds for a row in
// every CTA that needs the scale).
//   - Each q_i (24 significant bits) is added exactly into a 128-bit integer in
//     fixed point anchored at the largest square: with E the largest biased
//     exponent among the q_i, q_i = m_i * 2^(e_i - 150) enters as m_i << s_i,
//     s_i = e_i - E + 63, so the integer counts units of 2^(E - 213).  A square
//     with s_i < 0 is more than 2^63 below the largest one and is left out: all of
//     them together are below k * 2^-63 of the sum.
//   - Each thread keeps two 64-bit columns (bits 0 and 32 of the integer); a
//     square adds m << (s mod 32), below 2^55, to column s / 32.  The columns hold
//     2^8 terms (rows of up to 65536 values over 256 threads) without overflow.
//     Integer addition is exact, so the total is the same for every thread layout,
//     CTA and kernel.  These steps are issue-bound (every CTA on an SM runs them at
//     once), so they are kept short, and chunk slots past the row's end are skipped.
//   - mean = total * 2^(E - 213) / k: the top 64 bits of the total times a 64-bit
//     fixed-point reciprocal of k (made on the host) give the quotient to 2^-62
//     (relative), rounded to f32 to nearest even by integer steps.
// A NaN square makes the mean NaN, an infinite one +inf, as a double sum would.
#pragma once

#include <cstdint>

namespace bm {
namespace norm {

constexpr int kNormThreads = 256;  // eight warps take part in every reduction
constexpr int kNormWarps = kNormThreads / 32;
constexpr uint32_t kInfBits = 0x7f800000u;
constexpr int kWindow = 63;  // squares more than 2^63 below the largest are left out

// 1/k for the mean: recip = ceil(2^(63 + p) / k) with 2^(p-1) < k <= 2^p, so that
// recip lies in [2^63, 2^64).  Made on the host by reciprocal_of().
struct Recip {
    unsigned long long recip;
    int p;
};

inline Recip reciprocal_of(int64_t k)
{
    int p = 0;
    while (((int64_t)1 << p) < k) p++;
    const unsigned __int128 num = ((unsigned __int128)1 << (63 + p)) + (unsigned __int128)(k - 1);
    return Recip{(unsigned long long)(num / (unsigned __int128)k), p};
}

// 128-bit integer as four 32-bit limbs (least significant first).
struct Acc {
    uint32_t w0, w1, w2, w3;
};

__device__ __forceinline__ void add128(Acc &a, uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3)
{
    asm("add.cc.u32 %0, %0, %4;\n\taddc.cc.u32 %1, %1, %5;\n\taddc.cc.u32 %2, %2, %6;\n\taddc.u32 %3, %3, %7;"
        : "+r"(a.w0), "+r"(a.w1), "+r"(a.w2), "+r"(a.w3)
        : "r"(x0), "r"(x1), "r"(x2), "r"(x3));
}
__device__ __forceinline__ void add128(Acc &a, const Acc &b) { add128(a, b.w0, b.w1, b.w2, b.w3); }

struct Scratch {
    uint32_t mx[kNormWarps];
    Acc part[kNormWarps];
    float scale;
};

__device__ __forceinline__ uint32_t square_bits(float v) { return __float_as_uint(__fmul_rn(v, v)); }

__device__ __forceinline__ uint32_t max4(uint32_t mb, const float4 &v)
{
    return max(max(mb, square_bits(v.x)), max(max(square_bits(v.y), square_bits(v.z)), square_bits(v.w)));
}

struct Cols {
    unsigned long long c0, c1;
};

// Adds the square with bits b (finite, >= 0); base = kWindow - E.  When E > kWindow + 1
// every subnormal square lies below the window, so every square kept is normal and
// carries the hidden bit (fast == true); otherwise subnormal squares are handled too.
template <bool fast>
__device__ __forceinline__ void accumulate(Cols &a, uint32_t b, int base)
{
    const int e = (int)(b >> 23);  // biased exponent, 0 for a subnormal square or zero
    uint32_t m;
    int s;
    if (fast) {
        m = (b & 0x7fffffu) | 0x800000u;
        s = e + base;  // negative for zero and subnormal squares: left out
    } else {
        m = (b & 0x7fffffu) | ((uint32_t)min(e, 1) << 23);
        s = max(e, 1) + base;
    }
    const unsigned long long v = (unsigned long long)m << (s & 31);
    if ((uint32_t)s < 32u)
        a.c0 += v;  // 0 <= s < 32
    else if ((uint32_t)s < 64u)
        a.c1 += v;  // 32 <= s < 64 (a negative s wraps above both)
}

__device__ __forceinline__ Acc fold(const Cols &a)
{
    Acc r = {(uint32_t)a.c0, (uint32_t)(a.c0 >> 32), 0u, 0u};
    add128(r, 0u, (uint32_t)a.c1, (uint32_t)(a.c1 >> 32), 0u);
    return r;
}

// Largest of the group's square bit patterns (bit patterns of non-negative floats
// order as the values); sync() is the group's barrier.
template <class Sync>
__device__ __forceinline__ uint32_t group_max(uint32_t mb, int t, Scratch &sh, Sync sync)
{
    mb = __reduce_max_sync(0xffffffffu, mb);
    if ((t & 31) == 0) sh.mx[t >> 5] = mb;
    sync();
    mb = sh.mx[0];
#pragma unroll
    for (int w = 1; w < kNormWarps; w++) mb = max(mb, sh.mx[w]);
    return mb;
}

// total * 2^(E - 213) / k rounded to f32 (nearest even), total != 0.  Returns false
// when the result would not be a normal float (a mean below 2^-126).
__device__ __forceinline__ bool mean_f32(const Acc &a, int E, const Recip &rk, float &mean)
{
    const unsigned long long lo = ((unsigned long long)a.w1 << 32) | a.w0;
    const unsigned long long hi = ((unsigned long long)a.w3 << 32) | a.w2;
    unsigned long long T;
    int sh;  // total ~ T * 2^sh, T in [2^63, 2^64) (the bits below T are dropped: 2^-63)
    if (hi) {
        const int lz = __clzll((long long)hi);
        T = (hi << lz) | (lz ? lo >> (64 - lz) : 0ull);
        sh = 64 - lz;
    } else {
        const int lz = __clzll((long long)lo);
        T = lo << lz;
        sh = -lz;
    }
    const unsigned long long Q = __umul64hi(T, rk.recip);  // (T / k) * 2^(p - 1), in [2^62, 2^64)
    int d = 40 - __clzll((long long)Q);                    // bits to drop to keep 24
    uint32_t mant = (uint32_t)(Q >> d);
    const unsigned long long rem = Q & ((1ull << d) - 1), half = 1ull << (d - 1);
    if (rem > half || (rem == half && (mant & 1u))) mant++;
    if (mant >> 24) {
        mant >>= 1;
        d++;
    }
    const int field = d + 1 - rk.p + sh + E - 213 + 23 + 127;  // biased exponent of mant * 2^(d + 1 - p + sh + E - 213)
    if (field < 1 || field > 254) return false;
    mean = __uint_as_float(((uint32_t)field << 23) | (mant & 0x7fffffu));
    return true;
}

// The same mean through doubles, for a mean below the normal f32 range (rows whose
// values are all below about 1e-19): the total rounded to double, divided by k.
__device__ __forceinline__ float mean_tiny(const Acc &a, int E, int64_t k)
{
    const double lo = __ull2double_rn(((unsigned long long)a.w1 << 32) | a.w0);
    const double hi = __ull2double_rn(((unsigned long long)a.w3 << 32) | a.w2);
    const double total = __dadd_rn(__dmul_rn(hi, 18446744073709551616.0), lo);  // hi * 2^64 + lo
    const double unit = __longlong_as_double((long long)(E - 213 + 1023) << 52);  // 2^(E - 213), a normal double
    return __double2float_rn(__ddiv_rn(__dmul_rn(total, unit), (double)k));
}

__device__ __forceinline__ float scale_of_mean(float mean, float eps)
{
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
}

// The scale from the group's 128-bit totals: one thread adds the eight warp totals
// and takes mean and scale, then every thread reads it.
template <class Sync>
__device__ __forceinline__ float group_scale(Acc a, int E, int64_t k, const Recip &rk, float eps, int t, Scratch &sh,
                                             Sync sync)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        add128(a, __shfl_xor_sync(0xffffffffu, a.w0, o), __shfl_xor_sync(0xffffffffu, a.w1, o),
               __shfl_xor_sync(0xffffffffu, a.w2, o), __shfl_xor_sync(0xffffffffu, a.w3, o));
    if ((t & 31) == 0) sh.part[t >> 5] = a;
    sync();
    if (t == 0) {
        a = sh.part[0];
#pragma unroll
        for (int w = 1; w < kNormWarps; w++) add128(a, sh.part[w]);
        float mean = 0.0f;
        if ((a.w0 | a.w1 | a.w2 | a.w3) && !mean_f32(a, E, rk, mean)) mean = mean_tiny(a, E, k);
        sh.scale = scale_of_mean(mean, eps);
    }
    sync();
    return sh.scale;
}

// The scale when a square is infinite (mean +inf) or NaN (mean NaN).
__device__ __forceinline__ float special_scale(uint32_t mb, float eps)
{
    return scale_of_mean(__uint_as_float(mb == kInfBits ? kInfBits : 0x7fc00000u), eps);
}

// scale = 1 / sqrt(mean(x^2) + eps) of x[0..k) over the kNormThreads threads of one
// group (thread index t), reading x from memory twice; sync() is the group's barrier.
// vec: x is 16-byte aligned.  Every thread returns the same value.
template <class Sync>
__device__ __forceinline__ float row_scale(const float *__restrict__ x, int64_t k, const Recip &rk, float eps,
                                           bool vec, int t, Scratch &sh, Sync sync)
{
    const int64_t n4 = vec ? (k >> 2) : 0;
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    uint32_t mb = 0;
    for (int64_t c = t; c < n4; c += kNormThreads) mb = max4(mb, __ldg(x4 + c));
    for (int64_t i = 4 * n4 + t; i < k; i += kNormThreads) mb = max(mb, square_bits(__ldg(x + i)));
    mb = group_max(mb, t, sh, sync);
    if (mb >= kInfBits) return special_scale(mb, eps);
    const int E = max((int)(mb >> 23), 1);
    const int base = kWindow - E;
    Cols a = {0, 0}, b = {0, 0};  // two chains; integer sums in any grouping agree
    if (E > kWindow + 1) {
        for (int64_t c = t; c < n4; c += kNormThreads) {
            const float4 v = __ldg(x4 + c);
            accumulate<true>(a, square_bits(v.x), base);
            accumulate<true>(b, square_bits(v.y), base);
            accumulate<true>(a, square_bits(v.z), base);
            accumulate<true>(b, square_bits(v.w), base);
        }
        for (int64_t i = 4 * n4 + t; i < k; i += kNormThreads) accumulate<true>(a, square_bits(__ldg(x + i)), base);
    } else {
        for (int64_t c = t; c < n4; c += kNormThreads) {
            const float4 v = __ldg(x4 + c);
            accumulate<false>(a, square_bits(v.x), base);
            accumulate<false>(b, square_bits(v.y), base);
            accumulate<false>(a, square_bits(v.z), base);
            accumulate<false>(b, square_bits(v.w), base);
        }
        for (int64_t i = 4 * n4 + t; i < k; i += kNormThreads) accumulate<false>(a, square_bits(__ldg(x + i)), base);
    }
    Acc r = fold(a);
    add128(r, fold(b));
    return group_scale(r, E, k, rk, eps, t, sh, sync);
}

template <bool fast, int NC>
__device__ __forceinline__ void accumulate_held(Cols &a, Cols &b, const float4 (&v)[NC], int n4, int warp0, int base)
{
#pragma unroll
    for (int i = 0; i < NC; i++) {
        if (warp0 + i * kNormThreads < n4) {
            accumulate<fast>(a, square_bits(v[i].x), base);
            accumulate<fast>(b, square_bits(v[i].y), base);
            accumulate<fast>(a, square_bits(v[i].z), base);
            accumulate<fast>(b, square_bits(v[i].w), base);
        }
    }
}

// As row_scale for a row of k = 4 * n4 values, with thread t's chunks x[4c..4c+3],
// c = t + kNormThreads * i, already in registers (v[i]; zeros past the row's end):
// one read of x in all.  Slots past the row's end for the whole warp are skipped.
template <int NC, class Sync>
__device__ __forceinline__ float row_scale_held(const float4 (&v)[NC], int n4, const Recip &rk, float eps, int t,
                                                Scratch &sh, Sync sync)
{
    const int warp0 = t & ~31;  // the warp's first thread
    uint32_t mb = 0;
#pragma unroll
    for (int i = 0; i < NC; i++)
        if (warp0 + i * kNormThreads < n4) mb = max4(mb, v[i]);
    mb = group_max(mb, t, sh, sync);
    if (mb >= kInfBits) return special_scale(mb, eps);
    const int E = max((int)(mb >> 23), 1);
    Cols a = {0, 0}, b = {0, 0};  // two independent chains
    if (E > kWindow + 1)
        accumulate_held<true>(a, b, v, n4, warp0, kWindow - E);
    else
        accumulate_held<false>(a, b, v, n4, warp0, kWindow - E);
    Acc r = fold(a);
    add128(r, fold(b));
    return group_scale(r, E, (int64_t)n4 * 4, rk, eps, t, sh, sync);
}

__device__ __forceinline__ float apply(float x, float scale, float g) { return __fmul_rn(__fmul_rn(x, scale), g); }

}  // namespace norm
}  // namespace bm
