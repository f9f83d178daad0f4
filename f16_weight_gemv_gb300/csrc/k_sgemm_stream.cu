// k_sgemm_stream.cu -- products of 2..8 columns on tinyBLAS's path, bit for bit,
// for the shapes bm_takes_sgemm accepts (rows % 4 == 0, k % 8 == 0) whose activation
// is too long to stage whole in shared memory (k_sgemm_ring.cu takes the others: it
// streams like the one-column product and is faster); here the activation travels
// with the weights, slice by slice.
//
// Page "docs/modules/f16.md" (Design notes, "sgemm_dot"): every output
// Y[c*rows + r] is eight f32 chains -- lane l adds W[r][8t+l] * X[c][8t+l] in
// increasing t, from +0 -- folded as ((l0+l4)+(l2+l6))+((l1+l5)+(l3+l7)).  With a
// few columns the product is bound by streaming W from HBM (2..8 flops per
// weight byte), where tensor cores buy nothing; on the CUDA cores the chains keep
// their order, so the result is tinyBLAS's bit pattern.
//
// Layout on the GPU.  One CTA per SM.  Groups of 8 weight rows are split evenly
// between the CTAs; a CTA walks its groups in sub-blocks (R groups per consumer
// warp) and each sub-block in k-slices of bps 64-element blocks.  A ring slot
// holds one slice: a TMA box of 8 rows x 64 elements per group and block (128-byte
// swizzle: 16-byte chunk c of a 128-byte row r lands at c ^ (r % 8)), one box of
// NCP columns x 64 elements of X per block (NCP = ncols rounded up to even; columns
// past ncols and elements past k are zero-filled and never stored), and the f32
// copy of those X boxes.  The slot layout is fixed per launch from the number of
// groups a CTA owns, so that the ring holds as many weight bytes in flight as
// shared memory allows (the streaming rate follows the bytes in flight).
// Warp roles:
//   - eight issue warps, four lanes each, load the weight boxes of a slot (each of the
//     32 lanes arrives on the slot's barrier with its own byte count) and, on a
//     barrier of their own, its X boxes -- as far ahead as the ring allows.  One lane
//     cannot issue 1 KB boxes fast enough to keep HBM busy, and issue spreads over
//     warps, not over lanes of one warp (measured);
//   - two convert warps, alternating slots, widen a slot's X boxes to f32 once they
//     have landed and signal the slot; the products then read f32 operands only;
//   - eight consumer warps in CS column sets (CS = 1 or 2) of 8/CS warps; warp w
//     takes columns (w % CS) * NCP/CS .. of R groups of the sub-block.  Lane
//     4*rs + lp holds row rs of each of its warp's R groups and chains 2lp, 2lp+1 of
//     each of the warp's columns: 2*R*NCP/CS accumulators.  Each 8-element step
//     reads 4 bytes of each of its R rows (eight rows per warp and group: one
//     conflict-free wavefront by the swizzle), widens them once, and for each of its
//     columns reads 8 bytes of widened X (four addresses per warp), which then feed
//     R rows from registers through paired f32 FMAs (fma.rn.f32x2: chains 2lp and
//     2lp+1).  The launch picks R and CS from the groups a CTA owns and the columns:
//     with a few groups per CTA (Llama Q: 3-4) a single column set would leave most
//     warps idle while the busy ones wait on their loads.  Every operand is an exactly widened f16, so every product is
//     exact and every FMA rounds once, as tinyBLAS's does.  (The mixed-precision
//     f16 x f16 + f32 FMA would give the same bits but issues at half the f32 FMA
//     rate, which a kernel doing up to 8 FMAs per weight element cannot afford.)
//     At the end of a sub-block the four lane pairs of each row meet by two
//     shuffles: xor 2 forms (l0+l4, l1+l5) and (l2+l6, l3+l7), xor 1 brings the
//     other pair, and the lane with lp == c % 4 stores column c.
//
// Programmatic dependent launch: the weight boxes are issued without waiting for
// the kernel ahead (weights are constants); the X boxes, which read that kernel's
// output, and every output write come after griddepcontrol.wait.
//
// Every mbarrier wait is bounded; on a give-up the CTA records BM_ERR_TIMEOUT,
// drains the copies it issued (bounded) and exits.
#include "../../include/bm.h"
#include "bm_device.cuh"
#include "bm_internal.h"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

namespace bm {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kIssueWarps = 8;  // weight boxes: four lanes of each issue TMA copies
constexpr int kIssuersPerWarp = 4;
constexpr int kIssuers = kIssueWarps * kIssuersPerWarp;
constexpr int kConvertWarps = 2;  // X: widen to f32, signal (alternate slots)
constexpr int kIssueWarp0 = kConsumerWarps;
constexpr int kConvertWarp0 = kConsumerWarps + kIssueWarps;
constexpr int kThreads = 32 * (kConsumerWarps + kIssueWarps + kConvertWarps);
constexpr int kGroupRows = 8;
constexpr int kBoxCols = 64;                                // 128 bytes: one swizzle row
constexpr uint32_t kWBoxBytes = kGroupRows * kBoxCols * 2;  // 1 KB
constexpr int kMaxWBoxes = 32;                              // weight boxes per slot
constexpr int kMaxBlocks = 8;                               // 64-element blocks per slot
constexpr int kMaxStages = 16;
constexpr unsigned long long kTimeoutNs = 2000000000ull;

// Bytes between consecutive X boxes of a slot: NCP 128-byte rows, padded to whole
// 1 KB swizzle periods so that column c of every box is swizzle row c % 8.
__host__ __device__ constexpr uint32_t x16_slot(int ncp) { return ncp <= 8 ? 1024u : 2048u; }

// Consumer layouts (R groups per warp, CS column sets): each widened X value feeds R
// rows from registers, each widened weight value the warp's NCP/CS columns; at most
// 2 * R * NCP / CS <= 32 accumulators keep the 576-thread CTA within its registers.
struct Layout {
    int R, CS;
};
constexpr Layout kLayouts[] = {{2, 1}, {1, 2}, {2, 2}, {3, 2}};

struct SgemmJob {
    CUtensorMap wmap;  // W as [rows][k] 16-bit elements, box 64 x 8, 128-byte swizzle
    CUtensorMap xmap;  // X as [ncols][k] 16-bit elements, box 64 x NCP, 128-byte swizzle
    float *Y;
    int64_t rows;
    int64_t groups;       // ceil(rows / 8)
    int ncols;
    int k;
    int stages;
    int sub;              // groups per sub-block (<= 8 * R)
    int bps;              // 64-element blocks per slot (sub * bps <= 32)
    uint32_t x16_off;     // slot offsets: X boxes, widened X; slot size
    uint32_t x32_off;
    uint32_t slot_bytes;
    unsigned int *err;
    unsigned long long timeout_ns;
};

// Widens the eight f16 of a 16-byte chunk to f32 (exact).
__device__ __forceinline__ void widen8(float (&f)[8], const uint4 &h)
{
    asm("{\n\t.reg .b16 a, b, c, d, e, f, g, h;\n\t"
        "mov.b32 {a, b}, %8;\n\tmov.b32 {c, d}, %9;\n\tmov.b32 {e, f}, %10;\n\tmov.b32 {g, h}, %11;\n\t"
        "cvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\tcvt.f32.f16 %2, c;\n\tcvt.f32.f16 %3, d;\n\t"
        "cvt.f32.f16 %4, e;\n\tcvt.f32.f16 %5, f;\n\tcvt.f32.f16 %6, g;\n\tcvt.f32.f16 %7, h;\n\t}"
        : "=f"(f[0]), "=f"(f[1]), "=f"(f[2]), "=f"(f[3]), "=f"(f[4]), "=f"(f[5]), "=f"(f[6]), "=f"(f[7])
        : "r"(h.x), "r"(h.y), "r"(h.z), "r"(h.w));
}

// Widens the two f16 of a 4-byte word to f32 (exact).
__device__ __forceinline__ void widen2(float &lo, float &hi, uint32_t h)
{
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h));
}

// (a0, a1) = (w0 * x0 + a0, w1 * x1 + a1), each rounded once to f32: with f16 operands
// widened exactly, the product is exact and this is tinyBLAS's FMA step.
__device__ __forceinline__ void fma_x2(float &a0, float &a1, float w0, float w1, float x0, float x1)
{
    asm("{\n\t.reg .b64 A, W, X;\n\t"
        "mov.b64 A, {%0, %1};\n\tmov.b64 W, {%2, %3};\n\tmov.b64 X, {%4, %5};\n\t"
        "fma.rn.f32x2 A, W, X, A;\n\t"
        "mov.b64 {%0, %1}, A;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(w0), "f"(w1), "f"(x0), "f"(x1));
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

// The walk every role takes: sub-blocks of up to job.sub groups of the CTA's range,
// each in k-slices of job.bps 64-element blocks; step t of the walk uses ring slot
// t % stages.  f(t, first group, groups, first column, blocks in the slice, last
// slice of the sub-block) returns false to stop.
template <typename F>
__device__ __forceinline__ void walk(const SgemmJob &job, int64_t glo, int64_t ghi, F &&f)
{
    const int k = job.k, sw = job.bps * kBoxCols;
    const int nslices = (k + sw - 1) / sw;
    int t = 0;
    for (int64_t g = glo; g < ghi;) {
        const int ng = (int)min((int64_t)job.sub, ghi - g);
        for (int sl = 0; sl < nslices; sl++, t++)
            if (!f(t, g, ng, sl * sw, min(job.bps, (k - sl * sw + kBoxCols - 1) / kBoxCols), sl == nslices - 1))
                return;
        g += ng;
    }
}

template <int NCP, int R, int CS>
__global__ void __launch_bounds__(kThreads, 1) k_sgemm_stream(const __grid_constant__ SgemmJob job)
{
    constexpr int CW = NCP / CS;  // columns per warp
    constexpr uint32_t kX16Slot = x16_slot(NCP);
    constexpr uint32_t kX16BoxBytes = NCP * 128u;
    constexpr uint32_t kX32Block = NCP * 256u;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t wfull_bar[kMaxStages];   // weight boxes landed (16 issuer arrivals + bytes)
    __shared__ __align__(8) uint64_t xfull_bar[kMaxStages];   // X boxes landed (1 arrival + bytes)
    __shared__ __align__(8) uint64_t xready_bar[kMaxStages];  // X widened (1 arrival)
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];   // slot consumed (8 consumer warps)
    __shared__ int abort_flag;
    __shared__ int w_issued;            // walk steps whose weight boxes were issued
    __shared__ int x_last[kMaxStages];  // last walk step whose X boxes were issued into slot s

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = job.stages;
    const int bps = job.bps;
    // 1024-byte alignment: the swizzle pattern of the TMA boxes repeats every 1024 bytes.
    // (Offsetting the __shared__ array itself keeps the pointer in the shared window, so
    // the reads below compile to shared-memory loads, not generic ones.)
    uint8_t *smem = smem_raw + ((1024u - (dev::smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t ring_u = dev::smem_u32(smem);
    volatile int *abort_v = &abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            dev::mbar_init(dev::smem_u32(&wfull_bar[s]), kIssuers);
            dev::mbar_init(dev::smem_u32(&xfull_bar[s]), 1);
            dev::mbar_init(dev::smem_u32(&xready_bar[s]), 1);
            dev::mbar_init(dev::smem_u32(&empty_bar[s]), kConsumerWarps);
            x_last[s] = -1;
        }
        abort_flag = 0;
        w_issued = 0;
        dev::fence_barrier_init();
    }
    __syncthreads();
    dev::pdl_trigger();

    const int64_t G = job.groups;
    const int64_t glo = G * blockIdx.x / gridDim.x, ghi = G * (blockIdx.x + 1) / gridDim.x;

    if (warp >= kConvertWarp0) {
        // ------------------------------------------------------------ X: widen to f32, signal
        const int cw = warp - kConvertWarp0;
        walk(job, glo, ghi, [&](int t, int64_t, int, int, int nb, bool) {
            if (t % kConvertWarps != cw) return true;
            const int slot = t % S;
            const uint32_t ph = (uint32_t)(t / S) & 1u;
            if (!dev::mbar_wait_warp(dev::smem_u32(&xfull_bar[slot]), ph, abort_v, job.timeout_ns, job.err))
                return false;
            uint8_t *stage = smem + (size_t)slot * job.slot_bytes;
            const int nchunks = nb * NCP * 8;
            for (int ci = lane; ci < nchunks; ci += 32) {
                const int b = ci / (NCP * 8), c = (ci >> 3) % NCP, e8 = ci & 7;
                const uint4 h = *reinterpret_cast<const uint4 *>(stage + job.x16_off + b * kX16Slot + c * 128 +
                                                                ((e8 ^ (c & 7)) << 4));
                float f[8];
                widen8(f, h);
                float4 *d = reinterpret_cast<float4 *>(stage + job.x32_off + b * kX32Block + c * 256 + e8 * 32);
                d[0] = make_float4(f[0], f[1], f[2], f[3]);
                d[1] = make_float4(f[4], f[5], f[6], f[7]);
            }
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(dev::smem_u32(&xready_bar[slot]));
            return true;
        });
    } else if (warp >= kIssueWarp0) {
        // ------------------------------------------------------------ weight and X boxes
        bool waited = false;
        walk(job, glo, ghi, [&](int t, int64_t g, int ng, int kc0, int nb, bool) {
            const int slot = t % S;
            const uint32_t ph = (uint32_t)(t / S) & 1u;
            if (!dev::mbar_wait_warp(dev::smem_u32(&empty_bar[slot]), ph ^ 1u, abort_v, job.timeout_ns, job.err))
                return false;
            if (lane < kIssuersPerWarp) {
                const int me = (warp - kIssueWarp0) * kIssuersPerWarp + lane;
                const uint32_t fb = dev::smem_u32(&wfull_bar[slot]);
                const uint32_t dst = ring_u + (uint32_t)slot * job.slot_bytes;
                const int nw = ng * nb;  // <= 32 boxes: one per issuer at most
                const int mine = me < nw ? 1 : 0;
                dev::mbar_expect_tx(fb, (uint32_t)mine * kWBoxBytes);
                const int32_t row0 = (int32_t)(g * kGroupRows);
                for (int i = me; i < nw; i += kIssuers) {
                    const int q = i / nb, b = i % nb;
                    tma_load_2d(dst + (uint32_t)(q * bps + b) * kWBoxBytes, &job.wmap, kc0 + b * kBoxCols,
                                row0 + q * kGroupRows, fb);
                }
                if (me == kIssuers - 1) {
                    // the X boxes of the slot, on their own barrier, by the last issuer (it
                    // issues no more weight boxes than any other)
                    if (!waited) {
                        dev::pdl_wait();  // X is the previous kernel's output
                        waited = true;
                    }
                    const uint32_t xb = dev::smem_u32(&xfull_bar[slot]);
                    x_last[slot] = t;
                    dev::mbar_expect_tx(xb, (uint32_t)nb * kX16BoxBytes);
                    for (int b = 0; b < nb; b++)
                        tma_load_2d(dst + job.x16_off + (uint32_t)b * kX16Slot, &job.xmap, kc0 + b * kBoxCols, 0, xb);
                }
            }
            if (warp == kIssueWarp0 && lane == 0) w_issued = t + 1;
            return true;
        });
        __syncwarp();
    } else {
        // ------------------------------------------------------------ consumers
        dev::pdl_wait();  // output writes follow the kernel ahead
        const int lp = lane & 3;   // chains 2*lp and 2*lp + 1
        const int rs = lane >> 2;  // row within each of the warp's R groups
        const int c0 = (warp % CS) * CW;  // the warp's first column
        const int wg = warp / CS;         // the warp's place in its column set
        float acc[R][CW][2];
        walk(job, glo, ghi, [&](int t, int64_t g, int ng, int kc0, int nb, bool last) {
            const int slot = t % S;
            const uint32_t ph = (uint32_t)(t / S) & 1u;
            if (kc0 == 0) {
#pragma unroll
                for (int j = 0; j < R; j++)
#pragma unroll
                    for (int c = 0; c < CW; c++) acc[j][c][0] = acc[j][c][1] = 0.0f;
            }
            if (!dev::mbar_wait_warp(dev::smem_u32(&wfull_bar[slot]), ph, abort_v, job.timeout_ns, job.err) ||
                !dev::mbar_wait_warp(dev::smem_u32(&xready_bar[slot]), ph, abort_v, job.timeout_ns, job.err))
                return false;
            const uint8_t *stage = smem + (size_t)slot * job.slot_bytes;
            const int nact = min(R, ng - wg * R);  // groups of this warp in the sub-block (warp-uniform)
            if (nact > 0) {
                // row rs of group wg*R + j: box (wg*R + j)*bps + b, 128-byte row rs, word lp of a chunk
                const uint8_t *wrow = stage + (size_t)(wg * R * bps) * kWBoxBytes + rs * 128 + 4 * lp;
                const uint8_t *x32 = stage + job.x32_off + c0 * 256 + 8 * lp;
                const int nst = min(8 * bps, (job.k - kc0) >> 3);  // 8-element steps in this slice
                for (int b = 0; b * 8 < nst; b++) {
                    const uint8_t *wb = wrow + b * kWBoxBytes;
                    const uint8_t *xb = x32 + b * kX32Block;
                    // one 8-element step: R weight words, CW widened X pairs, R * CW paired FMAs
                    auto step = [&](int c8) {
                        float w[R][2];
#pragma unroll
                        for (int j = 0; j < R; j++) {
                            uint32_t h = 0;  // rows of groups past the sub-block are never stored
                            if (j < nact)
                                h = *reinterpret_cast<const uint32_t *>(wb + (size_t)(j * bps) * kWBoxBytes +
                                                                        ((c8 ^ rs) << 4));
                            widen2(w[j][0], w[j][1], h);
                        }
#pragma unroll
                        for (int c = 0; c < CW; c++) {
                            const float2 x = *reinterpret_cast<const float2 *>(xb + c * 256 + c8 * 32);
#pragma unroll
                            for (int j = 0; j < R; j++) fma_x2(acc[j][c][0], acc[j][c][1], w[j][0], w[j][1], x.x, x.y);
                        }
                    };
                    if (nst - 8 * b >= 8) {
#pragma unroll
                        for (int c8 = 0; c8 < 8; c8++) step(c8);
                    } else {
                        for (int c8 = 0; c8 < nst - 8 * b; c8++) step(c8);
                    }
                }
            }
            if (last) {
                // column c of row r: chains 2lp, 2lp+1 sit in lane pair lp of the row's four lanes.
                // xor 2 pairs lp 0<->2 and 1<->3: (l0+l4, l1+l5) and (l2+l6, l3+l7); xor 1 then
                // brings the other pair: ((l0+l4)+(l2+l6))+((l1+l5)+(l3+l7)) in every lane of the row.
#pragma unroll
                for (int j = 0; j < R; j++) {
                    const int64_t row = (g + wg * R + j) * kGroupRows + rs;
                    const bool mine = j < nact && row < job.rows;
#pragma unroll
                    for (int c = 0; c < CW; c++) {
                        const float s0 = acc[j][c][0] + __shfl_xor_sync(0xffffffffu, acc[j][c][0], 2);
                        const float s1 = acc[j][c][1] + __shfl_xor_sync(0xffffffffu, acc[j][c][1], 2);
                        const float o0 = __shfl_xor_sync(0xffffffffu, s0, 1);
                        const float o1 = __shfl_xor_sync(0xffffffffu, s1, 1);
                        const float y = (lp & 1) ? (o0 + s0) + (o1 + s1) : (s0 + o0) + (s1 + o1);
                        const int col = c0 + c;
                        if (mine && lp == (col & 3) && col < job.ncols) job.Y[(int64_t)col * job.rows + row] = y;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(dev::smem_u32(&empty_bar[slot]));
            return true;
        });
    }

    // ---------------------------------------------------------------- teardown
    __syncthreads();
    if (*abort_v && threadIdx.x == 0) {
        // every copy issued must land before this CTA's shared memory is released
        const int issued = w_issued;
        for (int s = 0; s < S && s < issued; s++) {
            const int lastw = issued - 1 - ((issued - 1 - s) % S);  // last step whose weights went to slot s
            dev::mbar_drain(dev::smem_u32(&wfull_bar[s]), (uint32_t)(lastw / S) & 1u, job.timeout_ns);
        }
        for (int s = 0; s < S; s++)
            if (x_last[s] >= 0)
                dev::mbar_drain(dev::smem_u32(&xfull_bar[s]), (uint32_t)(x_last[s] / S) & 1u, job.timeout_ns);
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

// [outer][k] 16-bit elements, boxes of 64 x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap *map, const uint16_t *base, int64_t outer, int64_t k, uint32_t box_rows)
{
    cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)k * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBoxCols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;
constexpr int kNumLayouts = sizeof(kLayouts) / sizeof(kLayouts[0]);
std::once_flag g_attr_once[kMaxDevices][5][kNumLayouts];

// The consumer layout for a CTA of `gpc` groups and NCP columns, as measured on GB300
// (Llama-3-8B and Qwen3 shapes at 2-8 columns, chains of launches over weights larger
// than L2; every layout gives the same bits):
//   - up to 4 groups (Q, down: 3-4): two column sets, one group per warp (21-31 % faster
//     than one column set at 2-4 columns), two groups per warp at 6-8 columns (39-42 %);
//   - 5 to 12 groups (Q/K/V: 5-6, gate: 12): two column sets, three groups per warp,
//     except gate-like CTAs of 9-12 groups at 2 columns, where one column set is 2 %
//     faster;
//   - 13 or more (gate/up: 24, the output product: 105): one column set, two groups
//     per warp (the others measured 1-40 % slower).
int pick_layout(int64_t gpc, int ncp)
{
    if (gpc <= 4) return ncp <= 4 ? 1 : 2;
    if (gpc <= 12) return gpc >= 9 && ncp == 2 ? 0 : 3;
    return 0;
}

template <int NCP, int LI>
int launch_layout(SgemmJob &job, int64_t grid, int64_t groups_per_cta, cudaStream_t s, const DeviceInfo &dev)
{
    constexpr int R = kLayouts[LI].R, CS = kLayouts[LI].CS;
    auto kern = k_sgemm_stream<NCP, R, CS>;
    // One CTA per SM.  The slot layout follows the groups a CTA owns: a sub-block of
    // up to 8/CS*R groups, and as many 64-element blocks per slot as keep its weight
    // boxes within 32; then as many slots as shared memory holds, so that the most
    // weight bytes are in flight.
    job.sub = (int)std::min<int64_t>(kConsumerWarps / CS * R, groups_per_cta);
    job.bps = std::max(1, std::min(kMaxBlocks, kMaxWBoxes / job.sub));
    job.x16_off = (uint32_t)(job.sub * job.bps) * kWBoxBytes;
    job.x32_off = job.x16_off + (uint32_t)job.bps * x16_slot(NCP);
    job.slot_bytes = (job.x32_off + (uint32_t)job.bps * NCP * 256u + 1023u) / 1024u * 1024u;
    const int64_t slots_per_sub = (job.k + job.bps * kBoxCols - 1) / (job.bps * kBoxCols);
    const int64_t steps = (groups_per_cta + job.sub - 1) / job.sub * slots_per_sub;
    const int64_t room = ((int64_t)dev.max_smem_optin - 2048 - 1024) / job.slot_bytes;
    if (room < 2) return fail(BM_ERR_UNSUPPORTED_DEVICE, "sgemm stream: too little shared memory");
    job.stages = (int)std::max<int64_t>(2, std::min<int64_t>({(int64_t)kMaxStages, room, steps}));
    const size_t smem = (size_t)job.stages * job.slot_bytes + 1024;

    int dev_id = 0;
    cudaGetDevice(&dev_id);
    std::call_once(g_attr_once[dev_id & (kMaxDevices - 1)][NCP / 2][LI], [&] {
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
    if (e != cudaSuccess) return fail(BM_ERR_CUDA, "sgemm stream: launch failed: %s", cudaGetErrorString(e));
    return BM_OK;
}

template <int NCP>
int launch_ncp(SgemmJob &job, cudaStream_t s, const DeviceInfo &dev)
{
    const int64_t G = job.groups;
    const int64_t grid = std::min<int64_t>((int64_t)dev.sm_count, G);
    const int64_t groups_per_cta = (G + grid - 1) / grid;
    switch (pick_layout(groups_per_cta, NCP)) {
    case 0: return launch_layout<NCP, 0>(job, grid, groups_per_cta, s, dev);
    case 1: return launch_layout<NCP, 1>(job, grid, groups_per_cta, s, dev);
    case 2: return launch_layout<NCP, 2>(job, grid, groups_per_cta, s, dev);
    default: return launch_layout<NCP, 3>(job, grid, groups_per_cta, s, dev);
    }
}

}  // namespace

int launch_sgemm_stream(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols, float *Y,
                        cudaStream_t s, const DeviceInfo &dev)
{
    if (ncols < 2 || ncols > kSgemmStreamMaxCols || rows % 4 != 0 || k % 8 != 0)
        return fail(BM_ERR_INVALID_ARG, "sgemm stream: shape outside 2..8 columns, rows %% 4 == 0, k %% 8 == 0");
    if (rows == 0) return BM_OK;
    if (rows > 0x7fffffffLL || k > 0x7fffffffLL) return fail(BM_ERR_INVALID_ARG, "sgemm stream: size too large");
    if (sgemm_ring_applies(X, ncols, k, dev)) return launch_sgemm_ring(W, rows, k, X, ncols, Y, s, dev);
    if (!encoder()) return fail(BM_ERR_CUDA, "sgemm stream: cuTensorMapEncodeTiled unavailable");
    const int ncp = (int)((ncols + 1) / 2 * 2);  // columns per thread, rounded up to even
    SgemmJob job{};
    if (!make_map(&job.wmap, W, rows, k, kGroupRows) || !make_map(&job.xmap, X, ncols, k, (uint32_t)ncp))
        return fail(BM_ERR_CUDA, "sgemm stream: tensor map encoding failed");
    job.Y = Y;
    job.rows = rows;
    job.groups = (rows + kGroupRows - 1) / kGroupRows;
    job.ncols = (int)ncols;
    job.k = (int)k;
    job.err = device_error_word();
    if (!job.err) return fail(BM_ERR_CUDA, "sgemm stream: device error word unavailable");
    job.timeout_ns = kTimeoutNs;
    switch (ncp) {
    case 2: return launch_ncp<2>(job, s, dev);
    case 4: return launch_ncp<4>(job, s, dev);
    case 6: return launch_ncp<6>(job, s, dev);
    default: return launch_ncp<8>(job, s, dev);
    }
}

}  // namespace bm
