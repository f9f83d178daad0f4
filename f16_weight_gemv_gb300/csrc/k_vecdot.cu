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
// This file holds the lane-per-chain kernel of the multi-column vec_dot fallback:
// lane c of a warp owns chain c (element 32s + c) for a tile of R rows x C
// columns, with 2-byte loads; the reduction is five warp shuffles per output, and
// lane q*R + i stores output (row i, column q), so a warp's stores are runs of
// consecutive rows.  One-column products go to k_gemv_stream.cu (k % 8 == 0) and
// k_gemv_bulk.cu (rows not 16-byte aligned).
#include "../../include/bm.h"
#include "bm_internal.h"

#include <cuda_fp16.h>

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

int launch_vecdot_ncol(const VecdotJob &job, cudaStream_t s, const DeviceInfo &)
{
    if (job.ncols == 1) return launch_lanes<8, 1>(job, s);
    if (job.ncols == 2) return launch_lanes<8, 2>(job, s);
    if (job.ncols <= 4) return launch_lanes<8, 4>(job, s);
    return launch_lanes<4, 8>(job, s);
}

}  // namespace bm
