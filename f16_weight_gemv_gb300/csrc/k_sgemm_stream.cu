// k_sgemm_stream.cu -- products of 2..16 columns on tinyBLAS's path, bit for bit,
// for the shapes bm_takes_sgemm accepts (rows % 4 == 0, k % 8 == 0).
//
// Page "docs/modules/f16.md" (Design notes, "sgemm_dot"): every output
// Y[c*rows + r] is eight f32 chains -- lane l adds W[r][8t+l] * X[c][8t+l] in
// increasing t, from +0 -- folded as ((l0+l4)+(l2+l6))+((l1+l5)+(l3+l7)).  With a
// few columns the product is bound by streaming W from HBM (2..16 flops per
// weight byte), where tensor cores buy nothing; on the CUDA cores the chains keep
// their order, so the result is tinyBLAS's bit pattern.
//
// Layout on the GPU.  One CTA per SM.  Groups of 8 weight rows are split evenly
// between the CTAs; a CTA walks its groups in sub-blocks of up to 16 groups, and
// each sub-block in k-slices of 64-element blocks (2 to 8 blocks per slice, more when
// the sub-block has fewer groups).  A ring slot holds one slice: a TMA box of 8 rows
// x 64 elements per group and block (128-byte swizzle: 16-byte chunk c of a 128-byte
// row r lands at c ^ (r % 8)), one box of NCP columns x 64 elements of X per block
// (NCP = ncols rounded up to even; columns past ncols and elements past k are
// zero-filled and never stored), and the f32 copy of those X boxes.  Warp roles:
//   - four issue warps, four lanes each, load the weight boxes of a slot (each of the
//     16 lanes arrives on the slot's barrier with its own byte count) and, on a
//     barrier of their own, its X boxes -- as far ahead as the ring allows;
//   - two convert warps, alternating slots, widen a slot's X boxes to f32 once they
//     have landed and signal the slot; the products then read f32 operands only;
//   - eight consumer warps, 16 rows each: lane 2*r + h holds row r and chains
//     l = 4h..4h+3 of every column.  Each 8-element step reads the row's 8 bytes
//     (16 rows per warp in two conflict-free wavefronts, by the swizzle), widens them
//     once, and for each column reads 16 bytes of widened X (two addresses per warp)
//     and issues two paired f32 FMAs (fma.rn.f32x2: chains l and l+1).  Every
//     operand is an exactly widened f16, so every product is exact and every FMA
//     rounds once, as tinyBLAS's does.  (The mixed-precision f16 x f16 + f32 FMA
//     would give the same bits but issues at half the f32 FMA rate, which a kernel
//     doing up to 16 FMAs per weight element cannot afford.)  At the end of a
//     sub-block the two halves of each chain set meet by one shuffle and the thread
//     with h == c % 2 folds and stores column c.
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
constexpr int kIssueWarps = 4;      // weight boxes: four lanes of each issue TMA copies
constexpr int kIssuersPerWarp = 4;
constexpr int kIssuers = kIssueWarps * kIssuersPerWarp;
constexpr int kConvertWarps = 2;    // X: load, widen to f32, signal (alternate stages)
constexpr int kIssueWarp0 = kConsumerWarps;
constexpr int kConvertWarp0 = kConsumerWarps + kIssueWarps;
constexpr int kThreads = 32 * (kConsumerWarps + kIssueWarps + kConvertWarps);
constexpr int kGroupRows = 8;
constexpr int kGroupsPerWarp = 2;                              // 16 rows per consumer warp
constexpr int kGroupsPerBlock = kConsumerWarps * kGroupsPerWarp;  // sub-block of 128 rows
constexpr int kBoxCols = 64;                                // 128 bytes: one swizzle row
constexpr uint32_t kWBoxBytes = kGroupRows * kBoxCols * 2;  // 1 KB
constexpr int kWBoxesPerStage = 32;
constexpr uint32_t kWBytes = kWBoxesPerStage * kWBoxBytes;  // 32 KB of weights per stage at most
constexpr int kMaxStages = 8;
constexpr unsigned long long kTimeoutNs = 2000000000ull;

constexpr uint32_t round_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Shared-memory geometry of one stage for NCP columns (ncols rounded up to even):
//   [W boxes: 32 KB][X boxes as loaded, f16][X widened to f32]
// X box b (NCP columns x 64 elements, 128-byte swizzle) sits at a 1 KB-aligned slot so
// that its column c is swizzle row c % 8; the widened copy holds, per block, NCP rows
// of 64 f32 (256 bytes each).
template <int NCP>
struct Geo {
    static constexpr int kMaxBlocks = NCP <= 4 ? 8 : 4;  // 64-element blocks per stage at most
    static constexpr uint32_t kX16Slot = NCP <= 8 ? 1024u : 2048u;
    static constexpr uint32_t kX16BoxBytes = NCP * 128u;
    static constexpr uint32_t kX32Block = NCP * 256u;
    static constexpr uint32_t kX16Off = kWBytes;
    static constexpr uint32_t kX32Off = kWBytes + kMaxBlocks * kX16Slot;
    static constexpr uint32_t kStageBytes = round_up(kX32Off + kMaxBlocks * kX32Block, 1024);
};

// 64-element blocks per stage for a sub-block of ng groups: up to 32 weight boxes, and
// no more blocks than the X regions of a stage hold.
template <int NCP>
__host__ __device__ __forceinline__ int blocks_per_stage(int ng)
{
    const int w = ng <= 1 ? 32 : ng <= 2 ? 16 : ng <= 4 ? 8 : ng <= 8 ? 4 : 2;
    return w < Geo<NCP>::kMaxBlocks ? w : Geo<NCP>::kMaxBlocks;
}

struct SgemmJob {
    CUtensorMap wmap;  // W as [rows][k] 16-bit elements, box 64 x 8, 128-byte swizzle
    CUtensorMap xmap;  // X as [ncols][k] 16-bit elements, box 64 x NCP, 128-byte swizzle
    float *Y;
    int64_t rows;
    int64_t groups;    // ceil(rows / 8)
    int ncols;
    int k;
    int stages;
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

// Widens the four f16 of an 8-byte chunk to f32 (exact).
__device__ __forceinline__ void widen4(float (&f)[4], const uint2 &h)
{
    asm("{\n\t.reg .b16 a, b, c, d;\n\t"
        "mov.b32 {a, b}, %4;\n\tmov.b32 {c, d}, %5;\n\t"
        "cvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\tcvt.f32.f16 %2, c;\n\tcvt.f32.f16 %3, d;\n\t}"
        : "=f"(f[0]), "=f"(f[1]), "=f"(f[2]), "=f"(f[3])
        : "r"(h.x), "r"(h.y));
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

// The walk every role takes: sub-blocks of up to 16 groups of the CTA's range, each in
// k-slices of blocks_per_stage 64-element blocks; stage t of the walk uses ring slot t % S.
template <int NCP, typename F>
__device__ __forceinline__ void walk(int64_t glo, int64_t ghi, int k, F &&f)
{
    int t = 0;
    for (int64_t g = glo; g < ghi;) {
        const int ng = (int)min((int64_t)kGroupsPerBlock, ghi - g);
        const int bps = blocks_per_stage<NCP>(ng);
        const int sw = bps * kBoxCols;
        const int nslices = (k + sw - 1) / sw;
        for (int sl = 0; sl < nslices; sl++, t++)
            if (!f(t, g, ng, bps, sl * sw, min(bps, (k - sl * sw + kBoxCols - 1) / kBoxCols), sl == nslices - 1))
                return;
        g += ng;
    }
}

template <int NCP>
__global__ void __launch_bounds__(kThreads, 1) k_sgemm_stream(const __grid_constant__ SgemmJob job)
{
    using G_ = Geo<NCP>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t wfull_bar[kMaxStages];   // weight boxes landed (16 issuer arrivals + bytes)
    __shared__ __align__(8) uint64_t xfull_bar[kMaxStages];   // X boxes landed (1 arrival + bytes)
    __shared__ __align__(8) uint64_t xready_bar[kMaxStages];  // X widened (1 arrival)
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];   // slot consumed (8 consumer warps)
    __shared__ int abort_flag;
    __shared__ int w_issued;              // stages whose weight boxes were issued
    __shared__ int x_last[kMaxStages];    // last stage whose X boxes were issued into slot s

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k = job.k;
    const int S = job.stages;
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
        walk<NCP>(glo, ghi, k, [&](int t, int64_t, int, int, int, int nb, bool) {
            if (t % kConvertWarps != cw) return true;
            const int slot = t % S;
            const uint32_t ph = (uint32_t)(t / S) & 1u;
            if (!dev::mbar_wait_warp(dev::smem_u32(&xfull_bar[slot]), ph, abort_v, job.timeout_ns, job.err))
                return false;
            uint8_t *stage = smem + (size_t)slot * G_::kStageBytes;
            const int nchunks = nb * NCP * 8;
            for (int ci = lane; ci < nchunks; ci += 32) {
                const int b = ci / (NCP * 8), c = (ci >> 3) % NCP, e8 = ci & 7;
                const uint4 h = *reinterpret_cast<const uint4 *>(stage + G_::kX16Off + b * G_::kX16Slot + c * 128 +
                                                                ((e8 ^ (c & 7)) << 4));
                float f[8];
                widen8(f, h);
                float4 *d = reinterpret_cast<float4 *>(stage + G_::kX32Off + b * G_::kX32Block + c * 256 + e8 * 32);
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
        walk<NCP>(glo, ghi, k, [&](int t, int64_t g, int ng, int bps, int kc0, int nb, bool) {
            const int slot = t % S;
            const uint32_t ph = (uint32_t)(t / S) & 1u;
            if (!dev::mbar_wait_warp(dev::smem_u32(&empty_bar[slot]), ph ^ 1u, abort_v, job.timeout_ns, job.err))
                return false;
            if (lane < kIssuersPerWarp) {
                const int me = (warp - kIssueWarp0) * kIssuersPerWarp + lane;
                const uint32_t fb = dev::smem_u32(&wfull_bar[slot]);
                const uint32_t dst = ring_u + (uint32_t)slot * G_::kStageBytes;
                const int nw = ng * nb;  // <= 32 boxes, two per issuer at most
                const int mine = (me < nw ? 1 : 0) + (me + kIssuers < nw ? 1 : 0);
                dev::mbar_expect_tx(fb, (uint32_t)mine * kWBoxBytes);
                const int32_t row0 = (int32_t)(g * kGroupRows);
                for (int i = me; i < nw; i += kIssuers) {
                    const int q = i / nb, b = i % nb;
                    tma_load_2d(dst + (uint32_t)(q * bps + b) * kWBoxBytes, &job.wmap, kc0 + b * kBoxCols,
                                row0 + q * kGroupRows, fb);
                }
                if (me == 0) {
                    // the X boxes of the slot, on their own barrier
                    if (!waited) {
                        dev::pdl_wait();  // X is the previous kernel's output
                        waited = true;
                    }
                    const uint32_t xb = dev::smem_u32(&xfull_bar[slot]);
                    x_last[slot] = t;
                    dev::mbar_expect_tx(xb, (uint32_t)nb * G_::kX16BoxBytes);
                    for (int b = 0; b < nb; b++)
                        tma_load_2d(dst + G_::kX16Off + (uint32_t)b * G_::kX16Slot, &job.xmap, kc0 + b * kBoxCols, 0,
                                    xb);
                }
            }
            if (warp == kIssueWarp0 && lane == 0) w_issued = t + 1;
            return true;
        });
        __syncwarp();
    } else {
        // ------------------------------------------------------------ consumers
        dev::pdl_wait();  // output writes follow the kernel ahead
        const int h = lane & 1;          // lanes 4h..4h+3 of the eight chains
        const int r16 = lane >> 1;       // row among the warp's 16
        const int rho = r16 & 7;         // row in its group
        const int mygrp = warp * kGroupsPerWarp + (r16 >> 3);
        float acc[NCP][4];
        walk<NCP>(glo, ghi, k, [&](int t, int64_t g, int ng, int bps, int kc0, int nb, bool last) {
            const int slot = t % S;
            const uint32_t ph = (uint32_t)(t / S) & 1u;
            if (kc0 == 0) {
#pragma unroll
                for (int c = 0; c < NCP; c++)
#pragma unroll
                    for (int e = 0; e < 4; e++) acc[c][e] = 0.0f;
            }
            if (!dev::mbar_wait_warp(dev::smem_u32(&wfull_bar[slot]), ph, abort_v, job.timeout_ns, job.err) ||
                !dev::mbar_wait_warp(dev::smem_u32(&xready_bar[slot]), ph, abort_v, job.timeout_ns, job.err))
                return false;
            const uint8_t *stage = smem + (size_t)slot * G_::kStageBytes;
            const bool active = mygrp < ng;
            if (active) {
                const uint8_t *wrow = stage + (size_t)(mygrp * bps) * kWBoxBytes + rho * 128 + 8 * h;
                const uint8_t *x32 = stage + G_::kX32Off + 16 * h;
                const int nst = min(8 * bps, (k - kc0) >> 3);  // 8-element steps in this slice
                for (int b = 0; b * 8 < nst; b++) {
                    const uint8_t *wb = wrow + b * kWBoxBytes;
                    const uint8_t *xb = x32 + b * G_::kX32Block;
                    const int n8 = min(8, nst - 8 * b);
#pragma unroll(NCP >= 12 ? 1 : 2)
                    for (int c8 = 0; c8 < n8; c8++) {
                        float w[4];
                        widen4(w, *reinterpret_cast<const uint2 *>(wb + ((c8 ^ rho) << 4)));
#pragma unroll
                        for (int c = 0; c < NCP; c++) {
                            const float4 x = *reinterpret_cast<const float4 *>(xb + c * 256 + c8 * 32);
                            fma_x2(acc[c][0], acc[c][1], w[0], w[1], x.x, x.y);
                            fma_x2(acc[c][2], acc[c][3], w[2], w[3], x.z, x.w);
                        }
                    }
                }
            }
            if (last) {
                // lanes 0..7 of column c are split over this thread and its partner (lane ^ 1):
                // ((l0+l4)+(l2+l6))+((l1+l5)+(l3+l7)); the thread with h == c % 2 stores it
                const int64_t row = (g + mygrp) * kGroupRows + rho;
#pragma unroll
                for (int c = 0; c < NCP; c++) {
                    float p[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) p[e] = __shfl_xor_sync(0xffffffffu, acc[c][e], 1);
                    float lo[4], hi[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        lo[e] = h ? p[e] : acc[c][e];
                        hi[e] = h ? acc[c][e] : p[e];
                    }
                    const float y = ((lo[0] + hi[0]) + (lo[2] + hi[2])) + ((lo[1] + hi[1]) + (lo[3] + hi[3]));
                    if (active && (c & 1) == h && c < job.ncols && row < job.rows) job.Y[(int64_t)c * job.rows + row] = y;
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
            const int lastw = issued - 1 - ((issued - 1 - s) % S);  // last stage whose weights went to slot s
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
std::once_flag g_attr_once[kMaxDevices][9];

template <int NCP>
int launch_ncp(SgemmJob &job, cudaStream_t s, const DeviceInfo &dev)
{
    using G_ = Geo<NCP>;
    auto kern = k_sgemm_stream<NCP>;
    // One CTA per SM, with a ring as deep as its share of the work needs.
    const int64_t G = job.groups;
    const int64_t grid = std::min<int64_t>((int64_t)dev.sm_count, G);
    const int64_t groups_per_cta = (G + grid - 1) / grid;
    const int64_t boxes_per_cta = groups_per_cta * ((job.k + kBoxCols - 1) / kBoxCols);
    const int64_t stages_needed = (boxes_per_cta + kWBoxesPerStage - 1) / kWBoxesPerStage + 1;
    const int64_t want = std::max<int64_t>(2, std::min<int64_t>(kMaxStages, stages_needed));
    const int64_t room = ((int64_t)dev.max_smem_optin - 2048 - 1024) / G_::kStageBytes;
    if (room < 2) return fail(BM_ERR_UNSUPPORTED_DEVICE, "sgemm stream: too little shared memory");
    job.stages = (int)std::min<int64_t>(want, room);
    const size_t smem = (size_t)job.stages * G_::kStageBytes + 1024;

    int dev_id = 0;
    cudaGetDevice(&dev_id);
    std::call_once(g_attr_once[dev_id & (kMaxDevices - 1)][NCP / 2], [&] {
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

}  // namespace

int launch_sgemm_stream(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols, float *Y,
                        cudaStream_t s, const DeviceInfo &dev)
{
    if (ncols < 2 || ncols > kSgemmStreamMaxCols || rows % 4 != 0 || k % 8 != 0)
        return fail(BM_ERR_INVALID_ARG, "sgemm stream: shape outside 2..16 columns, rows %% 4 == 0, k %% 8 == 0");
    if (rows == 0) return BM_OK;
    if (rows > 0x7fffffffLL || k > 0x7fffffffLL) return fail(BM_ERR_INVALID_ARG, "sgemm stream: size too large");
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
    case 8: return launch_ncp<8>(job, s, dev);
    case 10: return launch_ncp<10>(job, s, dev);
    case 12: return launch_ncp<12>(job, s, dev);
    case 14: return launch_ncp<14>(job, s, dev);
    default: return launch_ncp<16>(job, s, dev);
    }
}

}  // namespace bm
