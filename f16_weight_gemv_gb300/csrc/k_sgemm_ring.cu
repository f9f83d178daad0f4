// k_sgemm_ring.cu -- products of 2..8 columns on tinyBLAS's path, bit for bit, streamed
// the way the one-column kernel streams (k_gemv_stream.cu): rows % 4 == 0, k % 8 == 0,
// the activation 16-byte aligned and small enough to stage whole in shared memory.
//
// Page "docs/modules/f16.md" (Design notes, "sgemm_dot"): every output
// Y[c*rows + r] is eight f32 chains -- lane l adds W[r][8t+l] * X[c][8t+l] in
// increasing t, from +0 -- folded as ((l0+l4)+(l2+l6))+((l1+l5)+(l3+l7)).  The FMA
// here is the mixed-precision one (fma.rn.f32.f16: f16 operands taken at their exact
// values, one rounding to f32), which is tinyBLAS's step since the product of two
// f16 values is exact in f32.
//
// A few columns (the tokens of a small decode batch) are, like one column, bound by
// streaming W from HBM.  So this kernel keeps the one-column kernel's machinery and
// changes only the arithmetic: the 8-row groups of W are split evenly between the
// CTAs (two per SM, one when that gives each SM four groups or fewer); a CTA walks its
// groups in sub-blocks and k-slices whose stage holds up to 32 TMA boxes of 8 rows x
// 64 elements (128-byte swizzle: 16-byte chunk c of row r at chunk c ^ (r % 8)),
// floor(32 / groups) boxes per group; sixteen lanes of four producer warps issue a
// stage's boxes, each arriving on the stage's barrier with its own byte count, the
// weight copies starting before griddepcontrol.wait.  The NC activation columns (ncols
// rounded up to even; a padding column is zero and never stored; f16, 2 NC k bytes) are
// staged once per CTA after the wait.
//
// Consumers (eight warps, one group each): thread p of a row holds lanes 2p and 2p+1
// of every column's chains and reads, per 8-element step, the 4 bytes at element
// 8t + 2p of its row (the row's 16-byte chunk t % 8; the eight rows of a warp read
// eight distinct swizzled chunks, one conflict-free wavefront) and the matching 4
// bytes of each column (broadcast), then issues one FMA pair per column.  The fold:
// two xor-shuffles over the row's four threads in the order of the page's sum (lane
// pairs l, l+4, then the other pairs); thread c % 4 stores column c.
// Eight threads per row (one lane each, 2-byte reads, two warps per group) kept more
// warps busy in CTAs of one or two groups but measured no faster there (Llama Q
// 11.44 us with four threads per row, 11.61 with eight) and sixteen (one column per
// thread) 30 % slower: 4-byte reads feeding two FMAs each are what this kernel needs.
//
// Every mbarrier wait is bounded; on a give-up the CTA records BM_ERR_TIMEOUT, drains
// the copies it issued (bounded) and exits.
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
constexpr int kProducerWarps = 4;
constexpr int kIssuersPerWarp = 4;
constexpr int kIssuers = kProducerWarps * kIssuersPerWarp;
constexpr int kThreads = 32 * (kConsumerWarps + kProducerWarps);
constexpr int kGroupRows = 8;
constexpr int kBoxCols = 64;  // 128 bytes: one swizzle row
constexpr uint32_t kBoxBytes = kGroupRows * kBoxCols * 2;  // 1 KB
constexpr int kBoxesPerStage = 32;
constexpr uint32_t kStageBytes = kBoxesPerStage * kBoxBytes;  // 32 KB
constexpr int kMaxStages = 8;
constexpr unsigned long long kTimeoutNs = 2000000000ull;
constexpr unsigned kFull = 0xffffffffu;

constexpr int kGroupsPerBlock = kConsumerWarps;  // sub-block: one group per consumer warp

// floor(32 / ng) boxes per group for ng = 1..8, as a byte table.
__host__ __device__ __forceinline__ int boxes_per_group(int ng)
{
    return (int)((0x04040506080A1020ull >> (8 * (ng - 1))) & 0xffu);
}

struct RingJob {
    CUtensorMap map;  // W as [rows][k] 16-bit elements, box 64 x 8, 128-byte swizzle
    const uint16_t *X;  // [ncols][k] f16, 16-byte aligned
    float *Y;           // [ncols][rows]
    int ncols;
    int rows;
    int groups;  // ceil(rows / 8)
    int k;
    int stages;
    unsigned int *err;
    unsigned long long timeout_ns;
};

// a0 += w.lo * x.lo, a1 += w.hi * x.hi, each rounded once to f32 (exact f16 products).
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

// 4 bytes of shared memory at a shared-window address.  (volatile: never moved across
// the barrier waits, which are volatile too.)
__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
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

__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps)); }

// Shared memory of the staged activation: NC columns of k f16, whole KB.
__host__ __device__ constexpr uint32_t x_bytes(int nc, int64_t k) { return (uint32_t)((2 * nc * k + 1023) / 1024 * 1024); }

// The barriers and flags behind the ring: full and empty barriers of kMaxStages stages,
// the abort flag and the issued-stage count.
constexpr uint32_t kTailBytes = 256;
static_assert(2 * kMaxStages * 8 + 2 * 4 <= kTailBytes, "barrier area");

template <int NC>
__global__ void __launch_bounds__(kThreads, 2) k_sgemm_ring(const __grid_constant__ RingJob job)
{
    // Dynamic shared memory only: with no static variables its base is the start of the
    // block's window, 1024-byte aligned as the swizzled boxes need, so no bytes go to
    // padding (at two CTAs per SM that is what makes room for a third stage at 2 x 4096
    // activation elements).  Layout: the activation, the ring, the barriers and flags.
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k = job.k;
    const int S = job.stages;
    const uint32_t xbytes = x_bytes(NC, k);
    if (dev::smem_u32(smem) & 1023u) {  // not the layout above: refuse without touching anything
        if (threadIdx.x == 0) atomicExch(job.err, (unsigned)BM_ERR_UNSUPPORTED_DEVICE);
        return;
    }
    // the activation step-major: the 8 elements of step t of column c at 16 (t NC + c) bytes
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem);
    const uint32_t ring_u = dev::smem_u32(smem) + xbytes;
    uint64_t *const full_bar = reinterpret_cast<uint64_t *>(smem + xbytes + (size_t)S * kStageBytes);
    uint64_t *const empty_bar = full_bar + kMaxStages;
    int &abort_flag = *reinterpret_cast<int *>(empty_bar + kMaxStages);
    int &issued_slot = (&abort_flag)[1];
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
    dev::pdl_trigger();

    const int G = job.groups;
    const int glo = (int)((int64_t)G * blockIdx.x / gridDim.x), ghi = (int)((int64_t)G * (blockIdx.x + 1) / gridDim.x);
    const int nsteps = k >> 3;  // 8-element steps of a row

    if (warp >= kConsumerWarps) {
        // ------------------------------------------------------------ producers
        int t = 0;
        bool ok = true;
        for (int g = glo; g < ghi && ok;) {
            const int ng = min(kGroupsPerBlock, ghi - g);
            const int bpg = boxes_per_group(ng);
            const int sw = bpg * kBoxCols;
            const int nslices = (k + sw - 1) / sw;
            const int32_t row0 = (int32_t)(g * kGroupRows);
            for (int sl = 0; sl < nslices; sl++, t++) {
                const int slot = t % S;
                const uint32_t ph = (uint32_t)(t / S) & 1u;
                if (!dev::mbar_wait_warp(dev::smem_u32(&empty_bar[slot]), ph ^ 1u, abort_v, job.timeout_ns, job.err)) {
                    ok = false;
                    break;
                }
                const int kc0 = sl * sw;
                const int nb = min(bpg, (k - kc0 + kBoxCols - 1) / kBoxCols);
                if (lane < kIssuersPerWarp) {
                    const int me = (warp - kConsumerWarps) * kIssuersPerWarp + lane;
                    const uint32_t fb = dev::smem_u32(&full_bar[slot]);
                    const uint32_t dst = ring_u + (uint32_t)slot * kStageBytes;
                    const int nbox = ng * nb;  // <= 32: two per issuer at most
                    const int mine = (me < nbox ? 1 : 0) + (me + kIssuers < nbox ? 1 : 0);
                    dev::mbar_expect_tx(fb, (uint32_t)mine * kBoxBytes);
                    for (int i = me; i < nbox; i += kIssuers) {
                        const int q = i / nb, b = i % nb;
                        tma_load_2d(dst + (uint32_t)(q * bpg + b) * kBoxBytes, &job.map, kc0 + b * kBoxCols,
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
        dev::pdl_wait();  // X is the previous kernel's output; Y follows it too
        {
            const uint4 *xg = reinterpret_cast<const uint4 *>(job.X);
            uint4 *xo = reinterpret_cast<uint4 *>(xs);
            const int k8 = k >> 3;  // 16-byte chunks per column
            // in batches of eight loads, all in flight before the first store (one L2 round trip
            // per batch instead of per chunk)
            constexpr int kBatch = 8, kT = 32 * kConsumerWarps;
            for (int i0 = threadIdx.x; i0 < NC * k8; i0 += kBatch * kT) {
                uint4 h[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; u++) {
                    const int i = i0 + u * kT, ts = i / NC, c = i % NC;  // destination: step ts of column c
                    h[u] = i < NC * k8 && c < job.ncols ? __ldg(xg + (size_t)c * k8 + ts) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int u = 0; u < kBatch; u++)
                    if (i0 + u * kT < NC * k8) xo[i0 + u * kT] = h[u];
            }
        }
        consumers_sync();

        // lanes 4r..4r+3 serve row r of the warp's group, thread p lanes 2p, 2p+1
        const int tq = lane & 3;
        const int rho = lane >> 2;                // row in the group
        const int gw = warp;                      // the warp's group in the sub-block
        // Shared-window addresses.  The word of step c of a box (chunk c of the row, swizzled to
        // chunk c ^ rho) is at w ^ (c << 4) for w = the row's 128-byte base | rho << 4 | 4 tq:
        // the base's low 7 bits are zero, so the XOR swaps exactly the chunk bits.  Column q of
        // step t is at x + 16 (t NC + q), an immediate offset once t is the box's first step.
        const uint32_t xthr = dev::smem_u32(xs) + 4 * tq;
        bool ok = true;
        int t = 0;
        for (int g = glo; g < ghi && ok;) {
            const int ng = min(kGroupsPerBlock, ghi - g);
            const int bpg = boxes_per_group(ng);
            const int sw = bpg * kBoxCols;
            const int nslices = (k + sw - 1) / sw;
            const int row = (g + gw) * kGroupRows + rho;
            const bool active = gw < ng;  // warp-uniform
            float acc[NC][2];  // [column][lane]
#pragma unroll
            for (int c = 0; c < NC; c++) acc[c][0] = acc[c][1] = 0.0f;
            for (int sl = 0; sl < nslices; sl++, t++) {
                const int slot = t % S;
                const uint32_t ph = (uint32_t)(t / S) & 1u;
                if (!dev::mbar_wait_warp(dev::smem_u32(&full_bar[slot]), ph, abort_v, job.timeout_ns, job.err)) {
                    ok = false;
                    break;
                }
                const int kc0 = sl * sw;
                const uint32_t wrow = ring_u + (uint32_t)slot * kStageBytes +
                                      (uint32_t)(gw * bpg) * kBoxBytes + (uint32_t)rho * 128;
                const uint32_t wthr = wrow | ((uint32_t)rho << 4) | (uint32_t)(4 * tq);
                if (active) {
                    const int t0 = kc0 >> 3;                      // the slice's first step
                    const int nst = min(8 * bpg, nsteps - t0);    // steps in this slice
                    for (int b = 0; b * 8 < nst; b++) {
                        const uint32_t wb = wthr + (uint32_t)b * kBoxBytes;
                        const uint32_t xb = xthr + (uint32_t)(t0 + 8 * b) * (NC * 16);
                        const int n = min(8, nst - 8 * b);
                        // one 8-element step: the thread's two lanes of the row against every column
                        auto step = [&](int c) {
                            const uint32_t w = lds32(wb ^ ((uint32_t)c << 4));
#pragma unroll
                            for (int q = 0; q < NC; q++)
                                fma2(acc[q][0], acc[q][1], w, lds32(xb + (uint32_t)(16 * (c * NC + q))));
                        };
                        if (n == 8) {
#pragma unroll
                            for (int c = 0; c < 8; c++) step(c);
                        } else {
                            for (int c = 0; c < n; c++) step(c);
                        }
                    }
                }
                if (sl == nslices - 1) {
                    // ((l0+l4)+(l2+l6))+((l1+l5)+(l3+l7)) per column: xor 2 gives (l0+l4, l1+l5) in thread 0, (l2+l6, l3+l7) in thread 1
                    // (and the same sums in threads 2, 3); xor 1 then brings the other pair
#pragma unroll
                    for (int c = 0; c < NC; c++) {
                        const float s0 = acc[c][0] + __shfl_xor_sync(kFull, acc[c][0], 2);
                        const float s1 = acc[c][1] + __shfl_xor_sync(kFull, acc[c][1], 2);
                        const float o0 = __shfl_xor_sync(kFull, s0, 1), o1 = __shfl_xor_sync(kFull, s1, 1);
                        const float y = (s0 + o0) + (s1 + o1);
                        if (active && row < job.rows && tq == (c & 3) && c < job.ncols)
                            job.Y[(size_t)c * job.rows + row] = y;
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
        const int issued = issued_slot;
        for (int s = 0; s < S && s < issued; s++) {
            const int last = issued - 1 - ((issued - 1 - s) % S);
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

constexpr int kMaxDevices = 64;
std::once_flag g_attr_once[kMaxDevices][4];

}  // namespace

bool sgemm_ring_applies(const uint16_t *X, int64_t ncols, int64_t k, const DeviceInfo &dev)
{
    if (ncols < 2 || ncols > kSgemmStreamMaxCols || k % 8 != 0 || (reinterpret_cast<uintptr_t>(X) & 15) != 0)
        return false;
    const int64_t nc = (ncols + 1) / 2 * 2;
    // the staged activation and two stages must fit one CTA per SM, with 3 KB to spare
    return (int64_t)x_bytes((int)nc, k) + 2 * (int64_t)kStageBytes + 3072 <= (int64_t)dev.max_smem_optin;
}

namespace {

template <int NC>
int launch_nc(RingJob &job, cudaStream_t s, const DeviceInfo &dev)
{
    auto kern = k_sgemm_ring<NC>;
    // Two CTAs per SM, each with a ring as deep as its share of the work needs (2..8
    // stages), or one CTA per SM:
    //  - when the rows give each SM four groups or fewer: at two CTAs per SM most CTAs
    //    would hold one or two groups, so one or two consumer warps, each with a long
    //    slice per stage (same-GPU A/B at 2 columns: Llama-3-8B Q 7 %, Qwen3-0.6B Q/K/V
    //    30 %, SmolLM2 gate/up 40 % faster).  Its ring is capped at three stages: every
    //    CTA requests its ring at once and the whole matrix is only a few rings, so a
    //    deeper ring delays each CTA's first slice (Q 10.46 -> 9.82 us, 2048 x 4096
    //    9.15 -> 8.36 with three stages instead of six; 4 columns unchanged);
    //  - when the staged activation leaves no room for two stages at two CTAs per SM.
    // At two CTAs per SM a CTA of four or more groups takes the stages its half of the
    // SM holds (three at 2 x 4096 activation elements: gate 12 %, gate/up 6 %, the output
    // product 5 % faster than two); one of fewer groups keeps two, since a third stage
    // requested by every CTA at once only delays each CTA's first slice (Q/K/V 6144 x 4096
    // 4 % slower with three).
    const int64_t G = job.groups, k = job.k, sms = dev.sm_count;
    const uint32_t xbytes = x_bytes(NC, k);
    int64_t grid = std::min<int64_t>(G <= 4 * sms ? sms : 2 * sms, G);
    const int64_t groups_per_cta = (G + grid - 1) / grid;
    const int64_t boxes_per_cta = groups_per_cta * ((k + kBoxCols - 1) / kBoxCols);
    const int64_t stages_needed = (boxes_per_cta + kBoxesPerStage - 1) / kBoxesPerStage + 1;
    const int64_t want = std::max<int64_t>(2, std::min<int64_t>(kMaxStages, stages_needed));
    int64_t room = 0;
    if (grid > sms) {
        const int64_t share = ((int64_t)dev.smem_per_sm - 2 * (int64_t)dev.smem_reserved) / 2;  // one CTA's
        room = (share - (int64_t)kTailBytes - (int64_t)xbytes) / kStageBytes;
        if (groups_per_cta < 4) room = std::min<int64_t>(room, 2);
    }
    if (room < 2) {
        grid = std::min<int64_t>(grid, sms);
        room = ((int64_t)dev.max_smem_optin - 1024 - (int64_t)kTailBytes - (int64_t)xbytes) / kStageBytes;
        if (room < 2) return fail(BM_ERR_UNSUPPORTED_DEVICE, "sgemm ring: too little shared memory");
    }
    if (G <= 4 * sms) room = std::min<int64_t>(room, 3);
    job.stages = (int)std::min<int64_t>(want, room);
    const size_t smem = xbytes + (size_t)job.stages * kStageBytes + kTailBytes;

    int dev_id = 0;
    cudaGetDevice(&dev_id);
    std::call_once(g_attr_once[dev_id & (kMaxDevices - 1)][NC / 2 - 1], [&] {
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
    if (e != cudaSuccess) return fail(BM_ERR_CUDA, "sgemm ring: launch failed: %s", cudaGetErrorString(e));
    return BM_OK;
}

}  // namespace

int launch_sgemm_ring(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols, float *Y,
                      cudaStream_t s, const DeviceInfo &dev)
{
    if (rows % 4 != 0 || k % 8 != 0 || rows > 0x7fffffffLL - 8 || k > 0x7fffffffLL / 16 || ncols < 2 ||
        ncols > kSgemmStreamMaxCols)
        return fail(BM_ERR_INVALID_ARG, "sgemm ring: 2..8 columns, rows %% 4 == 0 and k %% 8 == 0 required");
    if (rows == 0) return BM_OK;
    if (!encoder()) return fail(BM_ERR_CUDA, "sgemm ring: cuTensorMapEncodeTiled unavailable");
    RingJob job{};
    {
        cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
        cuuint64_t strides[1] = {(cuuint64_t)k * 2};
        cuuint32_t box[2] = {(cuuint32_t)kBoxCols, (cuuint32_t)kGroupRows};
        cuuint32_t estr[2] = {1, 1};
        if (g_encode(&job.map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t *>(W), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return fail(BM_ERR_CUDA, "sgemm ring: tensor map encoding failed");
    }
    job.X = X;
    job.Y = Y;
    job.ncols = (int)ncols;
    job.rows = (int)rows;
    job.groups = (int)((rows + kGroupRows - 1) / kGroupRows);
    job.k = (int)k;
    job.err = device_error_word();
    if (!job.err) return fail(BM_ERR_CUDA, "sgemm ring: device error word unavailable");
    job.timeout_ns = kTimeoutNs;
    switch ((ncols + 1) / 2 * 2) {
    case 2: return launch_nc<2>(job, s, dev);
    case 4: return launch_nc<4>(job, s, dev);
    case 6: return launch_nc<6>(job, s, dev);
    default: return launch_nc<8>(job, s, dev);
    }
}

}  // namespace bm
