// k_vecdot.cu -- ggml_vec_dot_f16, bit for bit, for one or many rows and columns.
//
// The order restated from the page "docs/modules/f16.md" (Design notes,
// "vec_dot"): a row of k elements is cut into 32-element steps; element
// 32s + 8j + l feeds accumulator j (0..3), lane l (0..7), so there are 32
// independent f32 chains, each adding its products in increasing s from +0.
// The accumulators are combined lane-wise (a0+a2)+(a1+a3); lanes 0..3 are
// added to lanes 4..7; two horizontal adds leave (t0+t1)+(t2+t3).  The k%32
// tail is added to that value in double, in order, and the double is rounded
// once to f32.  Each f16 x f16 product is exact in f32, so the FMA of the page
// and the mixed-precision FMA below (f16 operands, f32 addend, one rounding)
// give identical bits.  No split of a chain is ever made; the thread layout
// decides only who computes a chain, never its order.
//
// This file holds the two kernels of the multi-column vec_dot fallback.  For short
// rows (32 <= k <= 256) the tile kernel gives each thread whole outputs of a
// 64-row x 64-column tile staged in shared memory: an output's 32 chains live in
// the thread's registers and take 16-byte reads (like the one-column kernels'
// accumulators), so the page's reduction is a few register adds; the tile leaves
// through shared memory as runs of consecutive rows.  Otherwise the lane-per-chain
// kernel: lane c of a warp owns chain c (element 32s + c) for a tile of R rows x C
// columns, with 2-byte loads and five warp shuffles per output.  One-column
// products go to k_gemv_stream.cu (k % 8 == 0) and k_gemv_bulk.cu (rows not
// 16-byte aligned).
#include "../../include/bm.h"
#include "bm_internal.h"

#include <cuda_fp16.h>

#include <mutex>

namespace bm {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void fma1(float &a, uint16_t w, uint16_t x)
{
    asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(a) : "h"(w), "h"(x));
}

// Weights are read once: no L1 allocation, and a 256-byte L2 prefetch so the
// next steps of the row are already on their way.
__device__ __forceinline__ uint16_t ld_weights2(const uint16_t *p)
{
    uint16_t v;
    asm("ld.global.nc.L1::no_allocate.L2::256B.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float widen(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// The k%32 tail of row w against activation x, added in double to r in order.
__device__ __forceinline__ float add_tail(float r, const uint16_t *w, const uint16_t *x, int64_t k32, int64_t k)
{
    if (k32 == k) return r;
    double sum = (double)r;
    for (int64_t i = k32; i < k; i++) sum += (double)__fmul_rn(widen(w[i]), widen(x[i]));
    return (float)sum;
}

__device__ __forceinline__ int matrix_of(const VecdotJob &job, int64_t g)
{
    int m = 0;
#pragma unroll
    for (int q = 1; q < 4; q++)
        if (q < job.nmat && g >= job.gbeg[q]) m = q;
    return m;
}

// ---------------------------------------------------------------------------
// lanes: any k, R rows x C columns per warp, lane c owns chain c.
// The 1-D grid enumerates (row block, column group) with the column group
// fastest, so consecutive blocks reuse the same weight rows from L2.
template <int R, int C, int U>
__global__ void __launch_bounds__(kThreads) k_vecdot_lanes(const __grid_constant__ VecdotJob job, int64_t ncg)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t cg = (int64_t)blockIdx.x % ncg;
    const int64_t g = ((int64_t)blockIdx.x / ncg) * kWarps + warp;
    if (g >= job.gbeg[job.nmat]) return;
    const int m = matrix_of(job, g);
    const int64_t rows = job.rows[m], k = job.k, ncols = job.ncols;
    const int64_t r0 = (g - job.gbeg[m]) * R, c0 = cg * C;

    const uint16_t *wr[R];
    const uint16_t *xc[C];
#pragma unroll
    for (int i = 0; i < R; i++) wr[i] = job.W[m] + min(r0 + i, rows - 1) * k + lane;
#pragma unroll
    for (int q = 0; q < C; q++) xc[q] = job.X + min(c0 + q, ncols - 1) * k + lane;

    float acc[R][C];
#pragma unroll
    for (int i = 0; i < R; i++)
#pragma unroll
        for (int q = 0; q < C; q++) acc[i][q] = 0.0f;

    const int64_t nsteps = k >> 5;
    int64_t s = 0;
    for (; s + U <= nsteps; s += U) {
        uint16_t wv[U][R], xv[U][C];
#pragma unroll
        for (int u = 0; u < U; u++) {
#pragma unroll
            for (int i = 0; i < R; i++) wv[u][i] = ld_weights2(wr[i] + 32 * (s + u));
#pragma unroll
            for (int q = 0; q < C; q++) xv[u][q] = __ldg(xc[q] + 32 * (s + u));
        }
#pragma unroll
        for (int u = 0; u < U; u++)
#pragma unroll
            for (int i = 0; i < R; i++)
#pragma unroll
                for (int q = 0; q < C; q++) fma1(acc[i][q], wv[u][i], xv[u][q]);
    }
    for (; s < nsteps; s++) {
        uint16_t wv[R], xv[C];
#pragma unroll
        for (int i = 0; i < R; i++) wv[i] = ld_weights2(wr[i] + 32 * s);
#pragma unroll
        for (int q = 0; q < C; q++) xv[q] = __ldg(xc[q] + 32 * s);
#pragma unroll
        for (int i = 0; i < R; i++)
#pragma unroll
            for (int q = 0; q < C; q++) fma1(acc[i][q], wv[i], xv[q]);
    }

    // Lane 8j + l holds chain (j, l).  Partners: lane^16 is j^2, lane^8 is j^1,
    // lane^4 is l^4, then lane^1 and lane^2 are the two horizontal adds.
    float mine = 0.0f;
#pragma unroll
    for (int i = 0; i < R; i++)
#pragma unroll
        for (int q = 0; q < C; q++) {
            float v = acc[i][q];
            v += __shfl_xor_sync(kFull, v, 16);
            v += __shfl_xor_sync(kFull, v, 8);
            v += __shfl_xor_sync(kFull, v, 4);
            v += __shfl_xor_sync(kFull, v, 1);
            v += __shfl_xor_sync(kFull, v, 2);
            v = __shfl_sync(kFull, v, 0);
            if (lane == q * R + i) mine = v;
        }
    if (lane < R * C) {
        const int i = lane % R, q = lane / R;
        const int64_t r = r0 + i, c = c0 + q;
        if (r < rows && c < ncols) {
            const float out = add_tail(mine, job.W[m] + r * k, job.X + c * k, nsteps << 5, k);
            job.y[m][c * rows + r] = out;
        }
    }
}

// ---------------------------------------------------------------------------
// tiles: short rows (32 <= k <= 256), ncols >= 2, whole outputs per thread.

constexpr int kShortMaxK = 256;  // the whole row is staged at once
constexpr int kStageBatch = 8;   // staging loads issued before their stores

__device__ __forceinline__ void fma2t(float &a0, float &a1, uint32_t w, uint32_t x)
{
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "mov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.f16 %0, wl, xl, %0;\n\t"
        "fma.rn.f32.f16 %1, wh, xh, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(w), "r"(x));
}

// A 64-row x 64-column tile per block, its rows and columns staged whole at once;
// warp w computes rows 8w..8w+7 and lane l columns l and l + 32, one output after
// another (its 32 chains in registers, as above), so a warp's weight reads are
// broadcasts and its activation reads fall in distinct banks (rows of an odd number
// of 16-byte chunks apart); the tile leaves through shared memory as runs of 64 rows.
constexpr int kBig = 64;

__global__ void __launch_bounds__(256) k_vecdot_tile_short(const __grid_constant__ VecdotJob job, int64_t nct,
                                                           int pitch)
{
    extern __shared__ __align__(16) uint8_t tsm[];
    uint16_t *ws = reinterpret_cast<uint16_t *>(tsm);            // [64][pitch]
    uint16_t *xs = ws + kBig * pitch;                            // [64][pitch]
    float *yt = reinterpret_cast<float *>(xs + kBig * pitch);    // [64 columns][65]
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int64_t ct = (int64_t)blockIdx.x % nct, rt = (int64_t)blockIdx.x / nct;
    const int64_t rows = job.rows[0], k = job.k, ncols = job.ncols;
    const int64_t r0 = rt * kBig, c0 = ct * kBig;
    const uint16_t *W = job.W[0];
    for (int i0 = t; i0 < kBig * pitch; i0 += 256 * kStageBatch) {  // eight loads in flight per thread
        uint16_t wv[kStageBatch], xv[kStageBatch];
#pragma unroll
        for (int u = 0; u < kStageBatch; u++) {
            const int i = i0 + 256 * u, rr = i / pitch, e = i % pitch;
            const int64_t r = r0 + rr, c = c0 + rr;
            wv[u] = (i < kBig * pitch && e < k && r < rows) ? W[r * k + e] : (uint16_t)0;
            xv[u] = (i < kBig * pitch && e < k && c < ncols) ? job.X[c * k + e] : (uint16_t)0;
        }
#pragma unroll
        for (int u = 0; u < kStageBatch; u++) {
            const int i = i0 + 256 * u;
            if (i < kBig * pitch) {
                ws[i] = wv[u];
                xs[i] = xv[u];
            }
        }
    }
    __syncthreads();
    const int nsteps = (int)(k >> 5);
    for (int o = 0; o < 16; o++) {
        const int rr = 8 * warp + (o & 7), cc = lane + 32 * (o >> 3);
        const uint4 *w4 = reinterpret_cast<const uint4 *>(ws + rr * pitch);
        const uint4 *x4 = reinterpret_cast<const uint4 *>(xs + cc * pitch);
        float a[4][8];
#pragma unroll
        for (int j = 0; j < 4; j++)
#pragma unroll
            for (int l = 0; l < 8; l++) a[j][l] = 0.0f;
        for (int st = 0; st < nsteps; st++) {
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const uint4 w = w4[4 * st + j], x = x4[4 * st + j];
                fma2t(a[j][0], a[j][1], w.x, x.x);
                fma2t(a[j][2], a[j][3], w.y, x.y);
                fma2t(a[j][4], a[j][5], w.z, x.z);
                fma2t(a[j][6], a[j][7], w.w, x.w);
            }
        }
        float v[8];
#pragma unroll
        for (int l = 0; l < 8; l++) v[l] = (a[0][l] + a[2][l]) + (a[1][l] + a[3][l]);
        const float t0 = v[0] + v[4], t1 = v[1] + v[5], t2 = v[2] + v[6], t3 = v[3] + v[7];
        float out = (t0 + t1) + (t2 + t3);
        if (32 * nsteps < k) {
            double sum = (double)out;
            for (int e = 32 * nsteps; e < k; e++)
                sum += (double)__fmul_rn(widen(ws[rr * pitch + e]), widen(xs[cc * pitch + e]));
            out = (float)sum;
        }
        yt[cc * (kBig + 1) + rr] = out;
    }
    __syncthreads();
    for (int i = t; i < kBig * kBig; i += 256) {
        const int cc = i / kBig, rr = i % kBig;
        const int64_t r = r0 + rr, c = c0 + cc;
        if (r < rows && c < ncols) job.y[0][c * rows + r] = yt[cc * (kBig + 1) + rr];
    }
}

int finish(const char *what)
{
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(BM_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
    return BM_OK;
}

// Row groups of `per` rows for each matrix of the job.
int64_t set_groups(VecdotJob &job, int per)
{
    job.gbeg[0] = 0;
    for (int m = 0; m < job.nmat; m++) job.gbeg[m + 1] = job.gbeg[m] + (job.rows[m] + per - 1) / per;
    for (int m = job.nmat; m < 4; m++) job.gbeg[m + 1] = job.gbeg[job.nmat];
    return job.gbeg[job.nmat];
}

template <int R, int C>
int launch_lanes(VecdotJob job, cudaStream_t s)
{
    const int64_t groups = set_groups(job, R);
    const int64_t ncg = (job.ncols + C - 1) / C;
    const int64_t blocks = ((groups + kWarps - 1) / kWarps) * ncg;
    if (blocks > 0x7fffffffLL) return fail(BM_ERR_INVALID_ARG, "vec_dot: product too large for one launch");
    constexpr int U = (R * C >= 16) ? 2 : 4;
    k_vecdot_lanes<R, C, U><<<(unsigned)blocks, kThreads, 0, s>>>(job, ncg);
    return finish("vec_dot (lanes)");
}

}  // namespace

int launch_vecdot_1col(const VecdotJob &job_in, cudaStream_t s, const DeviceInfo &dev)
{
    VecdotJob job = job_in;
    job.ncols = 1;
    if (job.k % 8 != 0) return launch_gemv_bulk(job, s, dev);
    return launch_gemv_stream(job, nullptr, nullptr, s, dev);
}

int launch_tile_short(VecdotJob job, cudaStream_t s)
{
    // rows of an odd number of 16-byte chunks, at least k elements
    int chunks = (int)((job.k + 7) / 8);
    if (chunks % 2 == 0) chunks++;
    const int pitch = 8 * chunks;
    const size_t smem = (size_t)2 * kBig * pitch * 2 + (size_t)kBig * (kBig + 1) * 4;  // <= 84 KB
    static std::once_flag attr_once[64];
    int d = 0;
    cudaGetDevice(&d);
    std::call_once(attr_once[d & 63], [] {
        cudaFuncSetAttribute(k_vecdot_tile_short, cudaFuncAttributeMaxDynamicSharedMemorySize, 100 * 1024);
    });
    const int64_t nct = (job.ncols + kBig - 1) / kBig, nrt = (job.rows[0] + kBig - 1) / kBig;
    if (nrt > 0x7fffffffLL / nct) return fail(BM_ERR_INVALID_ARG, "vec_dot: product too large for one launch");
    k_vecdot_tile_short<<<(unsigned)(nrt * nct), 256, smem, s>>>(job, nct, pitch);
    return finish("vec_dot (short tiles)");
}

int launch_vecdot_ncol(const VecdotJob &job, cudaStream_t s, const DeviceInfo &)
{
    // short rows: whole outputs per thread (measured 3.3x faster at 4096 x 33 x 512); longer
    // rows, fewer than 16 rows, or rows under one 32-element step (all of it the double
    // tail): the lane-per-chain kernel, which measured faster there
    if (job.nmat == 1 && job.ncols >= 2 && job.rows[0] >= 16 && job.k >= 32 && job.k <= kShortMaxK)
        return launch_tile_short(job, s);
    if (job.ncols == 1) return launch_lanes<8, 1>(job, s);
    if (job.ncols == 2) return launch_lanes<8, 2>(job, s);
    if (job.ncols <= 4) return launch_lanes<8, 4>(job, s);
    return launch_lanes<4, 8>(job, s);
}

}  // namespace bm
