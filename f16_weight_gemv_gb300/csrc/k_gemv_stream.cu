// k_gemv_stream.cu -- the one-column product (ggml_vec_dot_f16 per row, bit for
// bit) for rows of k % 8 == 0 elements, streamed through shared memory by TMA.
//
// The order is that of the page "docs/modules/f16.md" (Design notes, "vec_dot"):
// 32 f32 chains per row (element 32s + c feeds chain c = 8j + l, accumulator j,
// lane l), each adding its products in increasing s from +0; then
// (a0+a2)+(a1+a3) lane-wise, low four lanes + high four lanes, two horizontal
// adds, and the k%32 tail added in double in order.  Optionally the activation
// arrives in f32 and is first rounded to f16, nearest-even (Design notes,
// "Activation"), once per CTA -- the same bits bm_to_f16 gives -- and, before
// that, optionally normalised: rms_norm then mul by the norm weight (page
// "docs/modules/forward.md", Technical usage, "Other public pieces"), with the
// steps of bm_norm.cuh (an exact integer sum of the squares and an integer
// mean), so every CTA reaches the same scale and the same bits as the
// standalone norm kernel.
//
// Layout on the GPU.  Each matrix's rows are cut into groups of 8; the groups
// of all (up to four) matrices are split evenly between the CTAs (CTA b owns
// groups [G*b/n, G*(b+1)/n)), so every SM streams the same number of rows at any
// product size.  A CTA walks its groups in sub-blocks of up to four groups of
// one matrix, and each sub-block in k-slices: a stage holds up to 32 TMA boxes
// of 8 rows x 64 elements, floor(32 / groups) boxes per group (slices of 512 to
// 2048 elements; with 3 groups the stage is fuller than with a power of two per
// group).  The boxes of a stage are issued in parallel by 16 threads in four
// producer warps, two TMA instructions each (one issuing thread cannot keep HBM
// busy with 1 KB boxes; issue spreads best across warps), each thread arriving on
// the stage's barrier with its own byte count.  Boxes are stored with the
// 128-byte swizzle (16-byte chunk c of row r lands at chunk c ^ (r % 8)).  Rows
// past the matrix and columns past k are zero-filled and never used.  Two
// consumer warps serve each group, eight threads per row: thread q holds lanes
// 4(q & 1) .. +3 of accumulator q >> 1 (chains 4q..4q+3) and reads the 8 bytes at
// element 32s + 4q of each step, the activation's matching 8 bytes as a
// broadcast.  Warp w serves four rows of group w / 2, lanes 8r..8r+7 row
// (r >> 1) | ((w & 1) << 1) | ((r & 1) << 2), so the two rows of every 16-lane
// phase differ in bit 2 and their swizzled chunks fall in disjoint banks.  The
// reduction is three xor-shuffles across the row's eight threads (the partners
// holding accumulator j^2, then j^1, then the high four lanes), then the two
// horizontal adds in registers.  Eight threads per row measured faster than four
// (each holding a whole accumulator) on every product; CTAs of one or two groups of
// rows up to 4096 elements (the short products of a decode step) take sixteen, two
// chains and 4 bytes per step each, four warps per group, rows w % 4 and w % 4 + 4
// of group w / 4 in warp w, the reduction starting at the partner of accumulator
// j^2 (xor 8), so that every consumer warp has rows.
//
// Programmatic dependent launch: the producer issues its first ring's worth of
// weight copies at once -- the weights are not written by the kernel ahead of
// this one -- while the consumers wait for that kernel (griddepcontrol.wait)
// before they read the activation; all output writes follow.
//
// Every mbarrier wait is bounded; on a give-up the CTA records BM_ERR_TIMEOUT,
// drains the copies it issued (bounded) and exits.
#include "../../include/bm.h"
#include "bm_device.cuh"
#include "bm_internal.h"
#include "bm_norm.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

namespace bm {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kProducerWarps = 4;
constexpr int kIssuersPerWarp = 4;  // lanes of a producer warp that issue TMA copies
constexpr int kIssuers = kProducerWarps * kIssuersPerWarp;
constexpr int kThreads = 32 * (kConsumerWarps + kProducerWarps);
constexpr int kGroupRows = 8;                   // rows per TMA box
// Consumer layouts: TPR threads per row, each holding 32 / TPR of the row's 32 chains.
// TPR = 8: 4 rows per warp, two warps a group, sub-blocks of up to 4 groups.  TPR = 16
// (CTAs of one or two groups of short rows): 2 rows per warp, four warps a group,
// sub-blocks of up to 2 groups, so every consumer warp has rows.
template <int TPR>
__host__ __device__ constexpr int groups_per_block() { return kConsumerWarps * (32 / TPR) / kGroupRows; }
constexpr int kBoxCols = 64;                    // 128 bytes: one swizzle row
constexpr uint32_t kBoxBytes = kGroupRows * kBoxCols * 2;  // 1 KB
constexpr int kBoxesPerStage = 32;
constexpr uint32_t kStageBytes = kBoxesPerStage * kBoxBytes;  // 32 KB
constexpr int kMaxStages = 8;
constexpr unsigned long long kTimeoutNs = 2000000000ull;
constexpr unsigned kFull = 0xffffffffu;
static_assert(kConsumerWarps == norm::kNormWarps, "the norm's reductions run over the eight consumer warps");
constexpr int kNormThreadsC = norm::kNormThreads;
constexpr int kHeldChunks = 4;  // rows of up to 4 * 4 * 256 = 4096 values keep x and g in registers

// Boxes per group in one stage for a sub-block of ng (1..8) groups: floor(32 / ng),
// so every stage is (nearly) full and a sub-block of few groups takes a wider k-slice
// (a byte table instead of a division: the consumers compute it on a small product's
// critical path).
__host__ __device__ __forceinline__ int boxes_per_group(int ng)
{
    return (int)((0x04040506080A1020ull >> (8 * (ng - 1))) & 0xffu);
}

struct StreamJob {
    CUtensorMap map[4];  // W[m] as [rows[m]][k] 16-bit elements, box 64 x 8, 128-byte swizzle
    float *y[4];
    int rows[4];         // each below 2^31 (checked on the host)
    int gbeg[5];         // first 8-row group of matrix m; gbeg[nmat] = total groups (below 2^30)
    const void *x;       // activation: f16 bits, or f32 when x_is_f32
    uint16_t *h_out;     // optional: the rounded activation (written by CTA 0)
    const float *g;      // with x_is_f32: rms_norm then mul by g first (null: no norm)
    float *n_out;        // optional with g: the normalised f32 row (written by CTA 0)
    norm::Recip rk;      // 1 / k in fixed point (the norm's mean)
    float eps;
    int x_is_f32;
    int nmat;
    int k;
    int stages;
    unsigned int *err;
    unsigned long long timeout_ns;
};

// a0 += w.lo * x.lo, a1 += w.hi * x.hi: the mixed-precision FMA takes the f16
// operands as their exact values and rounds once to f32 -- the page's FMA step,
// since an f16 x f16 product is exact in f32.
__device__ __forceinline__ void fma2(float &a0, float &a1, uint32_t w, uint32_t x)
{
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "mov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.f16 %0, wl, xl, %0;\n\t"
        "fma.rn.f32.f16 %1, wh, xh, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(w), "r"(x));
}

// Lanes 4h .. 4h+3 of one accumulator: elements 8j + 4h .. 8j + 4h + 3 of a step.
__device__ __forceinline__ void fma4(float (&acc)[4], const uint2 &w, const uint2 &x)
{
    fma2(acc[0], acc[1], w.x, x.x);
    fma2(acc[2], acc[3], w.y, x.y);
}

// A thread's chains of one step from its bytes of W and x: 4 chains (8 bytes, TPR 8) or
// 2 chains (4 bytes, TPR 16).
template <int TPR>
__device__ __forceinline__ void fma_step(float (&acc)[32 / TPR], const uint8_t *w, const uint16_t *x)
{
    if constexpr (TPR == 8) {
        fma4(acc, *reinterpret_cast<const uint2 *>(w), *reinterpret_cast<const uint2 *>(x));
    } else {
        fma2(acc[0], acc[1], *reinterpret_cast<const uint32_t *>(w), *reinterpret_cast<const uint32_t *>(x));
    }
}

__device__ __forceinline__ float widen(uint16_t h) { return __half2float(__ushort_as_half(h)); }

__device__ __forceinline__ uint32_t pack_rn(float lo, float hi)
{
    __half2 p = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

__device__ __forceinline__ int matrix_of(const StreamJob &job, int g)
{
    int m = 0;
#pragma unroll
    for (int q = 1; q < 4; q++)
        if (q < job.nmat && g >= job.gbeg[q]) m = q;
    return m;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int32_t c0, int32_t c1,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// Named barrier of the eight consumer warps (the producer warp never joins it).
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps)); }

template <int TPR>
__global__ void __launch_bounds__(kThreads, 2) k_gemv_stream(const __grid_constant__ StreamJob job)
{
    constexpr int kGroupsPerBlock = groups_per_block<TPR>();
    constexpr int kChains = 32 / TPR;  // chains per thread
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ int abort_flag;
    __shared__ int issued_slot;
    __shared__ norm::Scratch norm_sh;
    __shared__ int first_sub[4];  // the first sub-block: matrix, groups, slices, group within the matrix

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k = job.k;
    const int S = job.stages;
    const uint32_t xbytes = (uint32_t)((2 * k + 1023) / 1024 * 1024);
    // 1024-byte alignment: the swizzle pattern of the TMA boxes repeats every 1024 bytes.
    // (Offsetting the __shared__ array itself keeps the pointer in the shared window, so
    // the reads below compile to shared-memory loads, not generic ones.)
    uint8_t *smem = smem_raw + ((1024u - (dev::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem);  // the f16 activation
    const uint32_t ring_u = dev::smem_u32(smem) + xbytes;
    volatile int *abort_v = &abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            dev::mbar_init(dev::smem_u32(&full_bar[s]), kIssuers);
            dev::mbar_init(dev::smem_u32(&empty_bar[s]), kConsumerWarps);
        }
        abort_flag = 0;
        issued_slot = 0;
        dev::fence_barrier_init();
    }
    __syncthreads();
    dev::pdl_trigger();  // the next kernel may start its own weight copies

    const int G = job.gbeg[job.nmat];
    const int glo = (int)((int64_t)G * blockIdx.x / gridDim.x), ghi = (int)((int64_t)G * (blockIdx.x + 1) / gridDim.x);
    const int nsteps = k >> 5;

    if (warp >= kConsumerWarps) {
        // ------------------------------------------------------------ producers
        int t = 0;
        bool ok = true;
        for (int g = glo; g < ghi && ok;) {
            const int m = matrix_of(job, g);
            const int ng = min(kGroupsPerBlock, min(ghi, job.gbeg[m + 1]) - g);
            const int bpg = boxes_per_group(ng);
            const int sw = bpg * kBoxCols;  // slice width in elements
            const int nslices = (k + sw - 1) / sw;
            const int32_t row0 = (int32_t)((g - job.gbeg[m]) * kGroupRows);
            for (int sl = 0; sl < nslices; sl++, t++) {
                const int slot = t % S;
                const uint32_t ph = (uint32_t)(t / S) & 1u;
                if (!dev::mbar_wait_warp(dev::smem_u32(&empty_bar[slot]), ph ^ 1u, abort_v, job.timeout_ns, job.err)) {
                    ok = false;
                    break;
                }
                const int kc0 = sl * sw;
                const int nb = min(bpg, (k - kc0 + kBoxCols - 1) / kBoxCols);  // boxes per group in this slice
                if (lane < kIssuersPerWarp) {
                    // each of the 16 issuers arrives once per stage, announcing the bytes of its own boxes
                    const int me = (warp - kConsumerWarps) * kIssuersPerWarp + lane;
                    const uint32_t fb = dev::smem_u32(&full_bar[slot]);
                    const uint32_t dst = ring_u + (uint32_t)slot * kStageBytes;
                    const int nbox = ng * nb;  // <= 32 boxes per stage, two per issuer at most
                    const int mine = (me < nbox ? 1 : 0) + (me + kIssuers < nbox ? 1 : 0);
                    dev::mbar_expect_tx(fb, (uint32_t)mine * kBoxBytes);
                    for (int i = me; i < nbox; i += kIssuers) {
                        const int q = i / nb, b = i % nb;
                        tma_load_2d(dst + (uint32_t)(q * bpg + b) * kBoxBytes, &job.map[m], kc0 + b * kBoxCols,
                                    row0 + q * kGroupRows, fb);
                    }
                }
                if (warp == kConsumerWarps && lane == 0) issued_slot = t + 1;
            }
            g += ng;
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ consumers
        const bool held = job.g && k <= 4 * kHeldChunks * kNormThreadsC;
        const int n4 = k >> 2;
        float4 w[kHeldChunks];
        if (held) {
            // the norm weight is a constant, not the previous kernel's output: read this
            // thread's chunks of it while that kernel finishes
#pragma unroll
            for (int i = 0; i < kHeldChunks; i++) {
                const int c = threadIdx.x + i * kNormThreadsC;
                w[i] = c < n4 ? __ldg(reinterpret_cast<const float4 *>(job.g) + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        if (threadIdx.x == 0 && glo < ghi) {
            // The first sub-block's set-up depends on the parameters alone: done here, before
            // the wait, it stays off a small product's critical path (read after the barrier
            // that follows the activation's conversion).
            const int m = matrix_of(job, glo);
            const int ng = min(kGroupsPerBlock, min(ghi, job.gbeg[m + 1]) - glo);
            const int sw = boxes_per_group(ng) * kBoxCols;
            first_sub[0] = m;
            first_sub[1] = ng;
            first_sub[2] = (k + sw - 1) / sw;
            first_sub[3] = glo - job.gbeg[m];
        }
        dev::pdl_wait();  // the activation is the previous kernel's output; outputs follow too
        if (held) {
            // the norm with this thread's chunks of x held in registers: one read of x
            const int t = threadIdx.x;
            const float4 *xf = reinterpret_cast<const float4 *>(job.x);
            float4 v[kHeldChunks];
#pragma unroll
            for (int i = 0; i < kHeldChunks; i++) {
                const int c = t + i * kNormThreadsC;
                v[i] = c < n4 ? __ldg(xf + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            const float scale = norm::row_scale_held(v, n4, job.rk, job.eps, t, norm_sh, [] { consumers_sync(); });
            uint2 *xo = reinterpret_cast<uint2 *>(xs);
#pragma unroll
            for (int i = 0; i < kHeldChunks; i++) {
                const int c = t + i * kNormThreadsC;
                if (c < n4) {
                    const float4 o = make_float4(norm::apply(v[i].x, scale, w[i].x), norm::apply(v[i].y, scale, w[i].y),
                                                 norm::apply(v[i].z, scale, w[i].z), norm::apply(v[i].w, scale, w[i].w));
                    if (job.n_out && blockIdx.x == 0) reinterpret_cast<float4 *>(job.n_out)[c] = o;
                    const uint2 p = make_uint2(pack_rn(o.x, o.y), pack_rn(o.z, o.w));
                    xo[c] = p;
                    if (job.h_out && blockIdx.x == 0) reinterpret_cast<uint2 *>(job.h_out)[c] = p;
                }
            }
        } else if (job.x_is_f32 && !job.g && k <= 4 * kHeldChunks * kNormThreadsC) {
            // every load of this thread in flight before the first conversion
            const float4 *xf = reinterpret_cast<const float4 *>(job.x);
            uint2 *xo = reinterpret_cast<uint2 *>(xs);
            float4 v[kHeldChunks];
#pragma unroll
            for (int i = 0; i < kHeldChunks; i++) {
                const int c = threadIdx.x + i * kNormThreadsC;
                v[i] = c < n4 ? __ldg(xf + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int i = 0; i < kHeldChunks; i++) {
                const int c = threadIdx.x + i * kNormThreadsC;
                if (c < n4) {
                    const uint2 p = make_uint2(pack_rn(v[i].x, v[i].y), pack_rn(v[i].z, v[i].w));
                    xo[c] = p;
                    if (job.h_out && blockIdx.x == 0) reinterpret_cast<uint2 *>(job.h_out)[c] = p;
                }
            }
        } else if (job.x_is_f32 && !job.g) {
            // longer rows, no norm: this thread's loads in batches of eight, each batch in flight
            // before its first conversion (a load, convert, store loop made one L2 round trip per
            // 16 bytes: 14 in a row at k = 14336)
            const float4 *xf = reinterpret_cast<const float4 *>(job.x);
            uint2 *xo = reinterpret_cast<uint2 *>(xs);
            constexpr int kBatch = 8;
            for (int i0 = threadIdx.x; i0 < n4; i0 += kBatch * kNormThreadsC) {
                float4 v[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; u++) {
                    const int i = i0 + u * kNormThreadsC;
                    v[u] = i < n4 ? __ldg(xf + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < kBatch; u++) {
                    const int i = i0 + u * kNormThreadsC;
                    if (i < n4) {
                        const uint2 p = make_uint2(pack_rn(v[u].x, v[u].y), pack_rn(v[u].z, v[u].w));
                        xo[i] = p;
                        if (job.h_out && blockIdx.x == 0) reinterpret_cast<uint2 *>(job.h_out)[i] = p;
                    }
                }
            }
        } else if (job.x_is_f32) {
            // longer rows with the norm: x read once for the sum, once more for the values, the
            // second pass in batches of four (x and g) in flight before their first use
            const float4 *xf = reinterpret_cast<const float4 *>(job.x);
            const float4 *gf = reinterpret_cast<const float4 *>(job.g);
            uint2 *xo = reinterpret_cast<uint2 *>(xs);
            const float scale = norm::row_scale(static_cast<const float *>(job.x), k, job.rk, job.eps, true,
                                                threadIdx.x, norm_sh, [] { consumers_sync(); });
            constexpr int kBatch = 4;
            for (int i0 = threadIdx.x; i0 < n4; i0 += kBatch * kNormThreadsC) {
                float4 v[kBatch], w[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; u++) {
                    const int i = i0 + u * kNormThreadsC;
                    v[u] = i < n4 ? __ldg(xf + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                    w[u] = i < n4 ? __ldg(gf + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < kBatch; u++) {
                    const int i = i0 + u * kNormThreadsC;
                    if (i < n4) {
                        const float4 o = make_float4(norm::apply(v[u].x, scale, w[u].x), norm::apply(v[u].y, scale, w[u].y),
                                                     norm::apply(v[u].z, scale, w[u].z), norm::apply(v[u].w, scale, w[u].w));
                        if (job.n_out && blockIdx.x == 0) reinterpret_cast<float4 *>(job.n_out)[i] = o;
                        const uint2 p = make_uint2(pack_rn(o.x, o.y), pack_rn(o.z, o.w));
                        xo[i] = p;
                        if (job.h_out && blockIdx.x == 0) reinterpret_cast<uint2 *>(job.h_out)[i] = p;
                    }
                }
            }
        } else {
            const uint4 *xg = reinterpret_cast<const uint4 *>(job.x);
            uint4 *xo = reinterpret_cast<uint4 *>(xs);
#pragma unroll 4
            for (int i = threadIdx.x; i < (k >> 3); i += 32 * kConsumerWarps) xo[i] = __ldg(xg + i);
        }
        consumers_sync();

        // Thread q of a row holds chains c = C q .. C q + C - 1 (C = 32 / TPR): lanes
        // c % 8 .. of accumulator j = c / 8; it reads the 2C bytes at element 32s + C q.
        // TPR = 8: warp w serves 4 rows of group w / 2, lanes 8r..8r+7 row
        // (r >> 1) | ((w & 1) << 1) | ((r & 1) << 2).  TPR = 16: warp w serves rows w % 4 and
        // w % 4 + 4 of group w / 4 (lanes 0-15, 16-31).  Either way the two rows of a
        // shared-memory phase differ in bit 2, so their swizzled chunks fall in disjoint
        // banks.
        const int tq = lane % TPR;                                  // thread within the row
        const int tr = lane / TPR;                                  // row slot within the warp
        const int gw = TPR == 8 ? warp >> 1 : warp >> 2;            // the warp's group in the sub-block
        const int rho = TPR == 8 ? (tr >> 1) | ((warp & 1) << 1) | ((tr & 1) << 2)
                                 : (warp & 3) | (tr << 2);           // row in the group
        const int j = tq * kChains / 8;                             // accumulator
        const int lb = 2 * ((tq * kChains) % 8);                    // byte of its first lane in a chunk
        const uint16_t *xq = xs + tq * kChains;                     // x[32s + C q] at xq[32 s]
        bool ok = true;
        int t = 0;
        for (int g = glo; g < ghi && ok;) {
            int m, ng, nslices, g_in_m;
            if (g == glo) {
                m = first_sub[0];
                ng = first_sub[1];
                nslices = first_sub[2];
                g_in_m = first_sub[3];
            } else {
                m = matrix_of(job, g);
                ng = min(kGroupsPerBlock, min(ghi, job.gbeg[m + 1]) - g);
                const int sw0 = boxes_per_group(ng) * kBoxCols;
                nslices = (k + sw0 - 1) / sw0;
                g_in_m = g - job.gbeg[m];
            }
            const int bpg = boxes_per_group(ng);
            const int sw = bpg * kBoxCols;
            const int row = (g_in_m + gw) * kGroupRows + rho;  // this thread's row (< 2^31)
            const bool active = gw < ng;                                       // warp-uniform
            float acc[kChains];  // this thread's lanes of accumulator j
#pragma unroll
            for (int e = 0; e < kChains; e++) acc[e] = 0.0f;
            for (int sl = 0; sl < nslices; sl++, t++) {
                const int slot = t % S;
                const uint32_t ph = (uint32_t)(t / S) & 1u;
                if (!dev::mbar_wait_warp(dev::smem_u32(&full_bar[slot]), ph, abort_v, job.timeout_ns, job.err)) {
                    ok = false;
                    break;
                }
                const int kc0 = sl * sw;
                // this thread's row inside the stage: group gw, box b at +b KB, 128-byte rows
                const uint8_t *rbase = smem + xbytes + (size_t)slot * kStageBytes +
                                       (size_t)(gw * bpg) * kBoxBytes + rho * 128;
                if (active) {
                    const int nst = min(2 * bpg, nsteps - kc0 / 32);  // chain steps in this slice
                    int s = 0;
                    for (; s + 2 <= nst; s += 2) {  // one 64-element box: two steps
                        const uint8_t *bx = rbase + (s >> 1) * kBoxBytes;
                        const int S0 = kc0 / 32 + s;
                        fma_step<TPR>(acc, bx + ((j) ^ rho) * 16 + lb, xq + 32 * S0);
                        fma_step<TPR>(acc, bx + ((4 + j) ^ rho) * 16 + lb, xq + 32 * S0 + 32);
                    }
                    if (s < nst) {
                        const uint8_t *bx = rbase + (s >> 1) * kBoxBytes;
                        const int S0 = kc0 / 32 + s;
                        fma_step<TPR>(acc, bx + ((j) ^ rho) * 16 + lb, xq + 32 * S0);
                    }
                }
                if (sl == nslices - 1) {
                    // (a0 + a2) + (a1 + a3) lane by lane: the partners holding accumulator j^2,
                    // then j^1, at the same lanes; then low four lanes + high four lanes, then the
                    // two horizontal adds.  Thread 0 of the row ends with the row's sum.
                    constexpr int P = 8 / kChains;  // threads per accumulator: thread q^(2P) holds j^2
#pragma unroll
                    for (int e = 0; e < kChains; e++) acc[e] += __shfl_xor_sync(kFull, acc[e], 2 * P);
#pragma unroll
                    for (int e = 0; e < kChains; e++) acc[e] += __shfl_xor_sync(kFull, acc[e], P);
                    float red;
                    if constexpr (TPR == 8) {
                        // lanes 0-3 in thread 0, 4-7 in thread 1
                        float hi[4];
#pragma unroll
                        for (int e = 0; e < 4; e++) hi[e] = __shfl_xor_sync(kFull, acc[e], 1);
                        const float t0 = acc[0] + hi[0], t1 = acc[1] + hi[1], t2 = acc[2] + hi[2], t3 = acc[3] + hi[3];
                        red = (t0 + t1) + (t2 + t3);
                    } else {
                        // lanes 2i, 2i+1 in thread i: thread 0 takes 0+4 and 1+5, thread 1 2+6 and 3+7
                        const float h0 = __shfl_xor_sync(kFull, acc[0], 2), h1 = __shfl_xor_sync(kFull, acc[1], 2);
                        const float ta = acc[0] + h0, tb = acc[1] + h1;
                        const float tc = __shfl_xor_sync(kFull, ta, 1), td = __shfl_xor_sync(kFull, tb, 1);
                        red = (ta + tb) + (tc + td);
                    }
                    if (active && tq == 0 && row < job.rows[m]) {
                        float out = red;
                        if (32 * nsteps < k) {
                            double sum = (double)red;
                            for (int e = 32 * nsteps; e < k; e++) {
                                const int cc = e - kc0;  // column inside the slice
                                const int b = cc >> 6, c = ((cc & 63) >> 3) ^ rho;
                                const uint16_t w = *reinterpret_cast<const uint16_t *>(rbase + b * kBoxBytes + c * 16 +
                                                                                       (cc & 7) * 2);
                                sum += (double)__fmul_rn(widen(w), widen(xs[e]));
                            }
                            out = (float)sum;
                        }
                        job.y[m][row] = out;
                    }
                }
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(dev::smem_u32(&empty_bar[slot]));
            }
            g += ng;
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncthreads();
    if (*abort_v && threadIdx.x == 0) {
        // every copy issued must land before this CTA's shared memory is released
        const int issued = issued_slot;
        for (int s = 0; s < S && s < issued; s++) {
            const int last = issued - 1 - ((issued - 1 - s) % S);  // last stage issued into slot s
            dev::mbar_drain(dev::smem_u32(&full_bar[s]), (uint32_t)(last / S) & 1u, job.timeout_ns);
        }
    }
    __syncthreads();
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool encoder()
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

bool make_row_map(CUtensorMap *map, const uint16_t *W, int64_t rows, int64_t k)
{
    cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)k * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBoxCols, (cuuint32_t)kGroupRows};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t *>(W), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encoding a tensor map is a driver call on every product; a decode step makes the
// same products with the same weights over and over.  A small direct-mapped cache per
// host thread keeps the maps made: a map depends only on the base address and the
// sizes it was made from, so an entry is valid for as long as its key matches.
struct RowMapEntry {
    CUtensorMap map;
    const void *W;
    int64_t rows, k;
    bool valid;
};
constexpr int kRowMapCache = 64;
thread_local RowMapEntry g_row_maps[kRowMapCache];

bool row_map_cached(CUtensorMap *map, const uint16_t *W, int64_t rows, int64_t k)
{
    const uint64_t h = (reinterpret_cast<uint64_t>(W) >> 8) * 0x9E3779B97F4A7C15ull ^ (uint64_t)rows * 0xC2B2AE3Dull ^
                       (uint64_t)k;
    RowMapEntry &e = g_row_maps[(h >> 32) & (kRowMapCache - 1)];
    if (e.valid && e.W == W && e.rows == rows && e.k == k) {
        *map = e.map;
        return true;
    }
    if (!make_row_map(map, W, rows, k)) return false;
    e.map = *map;
    e.W = W;
    e.rows = rows;
    e.k = k;
    e.valid = true;
    return true;
}

constexpr int kMaxDevices = 64;
std::once_flag g_attr_once[kMaxDevices][2];

}  // namespace

int launch_gemv_stream(const VecdotJob &vj, const float *x_f32, uint16_t *h_out, cudaStream_t s,
                       const DeviceInfo &dev, const ActNorm *nrm)
{
    if (!encoder()) return fail(BM_ERR_CUDA, "vec_dot: cuTensorMapEncodeTiled unavailable");
    if (vj.k > 0x7fffffffLL) return fail(BM_ERR_INVALID_ARG, "vec_dot: k too large");
    StreamJob job{};
    job.nmat = vj.nmat;
    job.k = (int)vj.k;
    job.x = x_f32 ? static_cast<const void *>(x_f32) : static_cast<const void *>(vj.X);
    job.x_is_f32 = x_f32 != nullptr;
    job.h_out = h_out;
    if (nrm) {
        if (!x_f32) return fail(BM_ERR_INVALID_ARG, "vec_dot: the norm needs the f32 activation");
        job.g = nrm->g;
        job.eps = nrm->eps;
        job.rk = norm::reciprocal_of(vj.k);
        job.n_out = nrm->n_out;
    }
    job.gbeg[0] = 0;
    for (int m = 0; m < vj.nmat; m++) {
        if (vj.rows[m] > 0x7fffffffLL) return fail(BM_ERR_INVALID_ARG, "vec_dot: rows must be below 2^31");
        if (!row_map_cached(&job.map[m], vj.W[m], vj.rows[m], vj.k))
            return fail(BM_ERR_CUDA, "vec_dot: tensor map encoding failed");
        job.y[m] = vj.y[m];
        job.rows[m] = (int)vj.rows[m];
        job.gbeg[m + 1] = job.gbeg[m] + (int)((vj.rows[m] + kGroupRows - 1) / kGroupRows);  // 4 x 2^28 at most
    }
    for (int m = vj.nmat; m < 4; m++) job.gbeg[m + 1] = job.gbeg[vj.nmat];
    const int64_t G = job.gbeg[vj.nmat];
    job.err = device_error_word();
    if (!job.err) return fail(BM_ERR_CUDA, "vec_dot: device error word unavailable");
    job.timeout_ns = kTimeoutNs;

    const uint32_t xbytes = (uint32_t)((2 * job.k + 1023) / 1024 * 1024);
    // Two CTAs per SM, each with a ring as deep as its share of the work needs (2..8
    // stages of 32 boxes); when the activation leaves no room for two stages at two
    // CTAs per SM (very long rows), one CTA per SM.
    int64_t grid = std::min<int64_t>((int64_t)dev.sm_count * 2, G);
    const int64_t groups_per_cta = (G + grid - 1) / grid;
    const int64_t boxes_per_cta = groups_per_cta * ((job.k + kBoxCols - 1) / kBoxCols);
    const int64_t stages_needed = (boxes_per_cta + kBoxesPerStage - 1) / kBoxesPerStage + 1;
    const int64_t want = std::max<int64_t>(2, std::min<int64_t>(kMaxStages, stages_needed));
    int64_t room = ((int64_t)dev.max_smem_optin / 2 - 2048 - 1024 - (int64_t)xbytes) / kStageBytes;
    if (room < 2) {
        grid = std::min<int64_t>(grid, dev.sm_count);
        room = ((int64_t)dev.max_smem_optin - 2048 - 1024 - (int64_t)xbytes) / kStageBytes;  // >= 5 for k <= BM_MAX_K
    }
    const int stages = (int)std::min<int64_t>(want, room);
    job.stages = stages;
    const size_t smem = xbytes + (size_t)stages * kStageBytes + 1024;
    // CTAs of one or two groups of rows up to 4096 elements take sixteen threads per row,
    // the rest eight (same-GPU A/B, same bits: Qwen3-0.6B down 7 %, Q 3 %, Llama-3-8B Q 2 %
    // faster, the SmolLM2 step 2 %; Llama-3-8B down, k = 14336, 1 % slower, within noise).
    const bool tpr16 = (G + grid - 1) / grid <= groups_per_block<16>() && job.k <= 4096;
    auto kern = tpr16 ? k_gemv_stream<16> : k_gemv_stream<8>;

    int dev_id = 0;
    cudaGetDevice(&dev_id);
    std::call_once(g_attr_once[dev_id & (kMaxDevices - 1)][tpr16 ? 1 : 0], [&] {
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.max_smem_optin - 1024);
    });

    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, job);
    if (e != cudaSuccess) return fail(BM_ERR_CUDA, "vec_dot (stream): launch failed: %s", cudaGetErrorString(e));
    return BM_OK;
}

}  // namespace bm
