// k_gemv_step.cu -- a decode step's one-column products in one launch.
//
// Each call of the step is bm_f16_matvec_act's: an f32 activation rounded to f16,
// nearest-even (page "docs/modules/f16.md", Design notes, "Activation"), then
// multiplied by up to four matrices, ggml_vec_dot_f16 per row, bit for bit
// (Design notes, "vec_dot": 32 chains, (a0+a2)+(a1+a3), low + high, two
// horizontal adds, the k%32 tail in double).  The chains, TMA boxes and reduction
// order are those of k_gemv_stream.cu, so every output has the bits the separate
// calls give; the consumers here keep four threads per row (thread j holding
// accumulator j, 16-byte reads, one warp per group).
//
// What differs is the schedule.  One persistent grid (two CTAs per SM, launched
// cooperatively so that all of them are resident) walks the calls in order.  The
// producer warps of a CTA stream the weight boxes of its share of every call
// through one ring without stopping between calls -- weights are constants -- so
// while the consumers finish call c, or wait, the ring already fills with call
// c+1's weights.  Before the consumers read call c+1's activation they wait until
// every CTA has finished call c (a grid-wide counter: each CTA adds one after its
// outputs of a call are written, behind a device-scope fence), because in a
// decode step an activation is made from earlier outputs; a call may read what any
// earlier call of the step wrote.  The counter is reset by the CTA that finishes
// the step last, so the next run (stream-ordered) starts from zero.
//
// Every wait -- the ring's mbarriers and the grid counter -- is bounded by the
// global timer; a give-up records BM_ERR_TIMEOUT, stops the CTA's work, drains the
// copies it issued (bounded) and exits.
#include "../../include/bm.h"
#include "bm_device.cuh"
#include "bm_internal.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>

namespace bm {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kProducerWarps = 4;
constexpr int kIssuersPerWarp = 4;
constexpr int kIssuers = kProducerWarps * kIssuersPerWarp;
constexpr int kThreads = 32 * (kConsumerWarps + kProducerWarps);
constexpr int kGroupRows = 8;
constexpr int kGroupsPerBlock = kConsumerWarps;
constexpr int kBoxCols = 64;
constexpr uint32_t kBoxBytes = kGroupRows * kBoxCols * 2;  // 1 KB
constexpr int kBoxesPerStage = 32;
constexpr uint32_t kStageBytes = kBoxesPerStage * kBoxBytes;  // 32 KB
constexpr int kMaxStages = 8;
constexpr unsigned long long kTimeoutNs = 2000000000ull;
constexpr unsigned kFull = 0xffffffffu;

__host__ __device__ __forceinline__ int boxes_per_group(int ng)
{
    return ng <= 1 ? 32 : ng <= 2 ? 16 : ng <= 4 ? 8 : 4;
}

// One call, in device memory (the tensor maps must be 64-byte aligned there).
struct alignas(128) StepCall {
    CUtensorMap map[4];  // W[m] as [rows[m]][k] 16-bit elements, box 64 x 8, 128-byte swizzle
    float *y[4];
    const float *x;      // f32 activation, 16-byte aligned
    int rows[4];
    int gbeg[5];         // first 8-row group of matrix m; gbeg[nmat] = total groups
    int k;
    int nmat;
};

struct StepParams {
    const StepCall *calls;
    int ncalls;
    int kmax;
    int stages;
    unsigned int *counter;  // CTAs that finished a call, summed over the step's calls
    unsigned int *err;
    unsigned long long timeout_ns;
};

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

__device__ __forceinline__ void fma8(float (&acc)[8], const uint4 &w, const uint4 &x)
{
    fma2(acc[0], acc[1], w.x, x.x);
    fma2(acc[2], acc[3], w.y, x.y);
    fma2(acc[4], acc[5], w.z, x.z);
    fma2(acc[6], acc[7], w.w, x.w);
}

__device__ __forceinline__ float widen(uint16_t h) { return __half2float(__ushort_as_half(h)); }

__device__ __forceinline__ uint32_t pack_rn(float lo, float hi)
{
    __half2 p = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

__device__ __forceinline__ int matrix_of(const StepCall &c, int g)
{
    int m = 0;
#pragma unroll
    for (int q = 1; q < 4; q++)
        if (q < c.nmat && g >= c.gbeg[q]) m = q;
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

__device__ __forceinline__ void consumers_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps) : "memory");
}

__device__ __forceinline__ unsigned int ld_acquire(const unsigned int *p)
{
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ float4 ld_cg4(const float4 *p)
{
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

// The ranges of call c's groups that CTA b owns.
__device__ __forceinline__ void my_groups(const StepCall &c, int &glo, int &ghi)
{
    const int G = c.gbeg[c.nmat];
    glo = (int)((int64_t)G * blockIdx.x / gridDim.x);
    ghi = (int)((int64_t)G * (blockIdx.x + 1) / gridDim.x);
}

__global__ void __launch_bounds__(kThreads, 2) k_gemv_step(const __grid_constant__ StepParams p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ int abort_flag;
    __shared__ int issued_slot;
    __shared__ int cons_stop;  // written by consumer threads only, read between two consumer barriers

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.stages;
    const uint32_t xbytes = (uint32_t)((2 * p.kmax + 1023) / 1024 * 1024);
    uint8_t *smem = smem_raw + ((1024u - (dev::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem);
    const uint32_t ring_u = dev::smem_u32(smem) + xbytes;
    volatile int *abort_v = &abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            dev::mbar_init(dev::smem_u32(&full_bar[s]), kIssuers);
            dev::mbar_init(dev::smem_u32(&empty_bar[s]), kConsumerWarps);
        }
        abort_flag = 0;
        issued_slot = 0;
        cons_stop = 0;
        dev::fence_barrier_init();
    }
    __syncthreads();

    // One answer for every consumer warp: whether to stop (a failed wait of any of them, or
    // the CTA's abort flag).  The flag is read by all between two barriers, so no warp can
    // leave the loop while another goes on to the next barrier.
    volatile int *stop_v = &cons_stop;
    auto consumers_agree_stop = [&](bool failed) -> bool {
        if (failed || (threadIdx.x == 0 && *abort_v)) *stop_v = 1;
        consumers_sync();
        const bool stop = *stop_v != 0;
        consumers_sync();
        return stop;
    };

    if (warp >= kConsumerWarps) {
        // ------------------------------------------------------------ producers
        int t = 0;
        bool ok = true;
        for (int ci = 0; ci < p.ncalls && ok; ci++) {
            const StepCall &c = p.calls[ci];
            const int k = c.k;
            int glo, ghi;
            my_groups(c, glo, ghi);
            for (int g = glo; g < ghi && ok;) {
                const int m = matrix_of(c, g);
                const int ng = min(kGroupsPerBlock, min(ghi, c.gbeg[m + 1]) - g);
                const int bpg = boxes_per_group(ng);
                const int sw = bpg * kBoxCols;
                const int nslices = (k + sw - 1) / sw;
                const int32_t row0 = (int32_t)((g - c.gbeg[m]) * kGroupRows);
                for (int sl = 0; sl < nslices; sl++, t++) {
                    const int slot = t % S;
                    const uint32_t ph = (uint32_t)(t / S) & 1u;
                    if (!dev::mbar_wait_warp(dev::smem_u32(&empty_bar[slot]), ph ^ 1u, abort_v, p.timeout_ns, p.err)) {
                        ok = false;
                        break;
                    }
                    const int kc0 = sl * sw;
                    const int nb = min(bpg, (k - kc0 + kBoxCols - 1) / kBoxCols);
                    if (lane < kIssuersPerWarp) {
                        const int me = (warp - kConsumerWarps) * kIssuersPerWarp + lane;
                        const uint32_t fb = dev::smem_u32(&full_bar[slot]);
                        const uint32_t dst = ring_u + (uint32_t)slot * kStageBytes;
                        const int nbox = ng * nb;
                        const int mine = (me < nbox ? 1 : 0) + (me + kIssuers < nbox ? 1 : 0);
                        dev::mbar_expect_tx(fb, (uint32_t)mine * kBoxBytes);
                        for (int i = me; i < nbox; i += kIssuers) {
                            const int q = i / nb, b = i % nb;
                            tma_load_2d(dst + (uint32_t)(q * bpg + b) * kBoxBytes, &c.map[m], kc0 + b * kBoxCols,
                                        row0 + q * kGroupRows, fb);
                        }
                    }
                    if (warp == kConsumerWarps && lane == 0) issued_slot = t + 1;
                }
                g += ng;
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ consumers
        const int j = lane & 3;
        const int t4 = lane >> 2;
        const int rho = (t4 >> 1) | ((t4 & 1) << 2);
        const uint4 *x4 = reinterpret_cast<const uint4 *>(xs) + j;
        bool ok = true;
        int t = 0;
        for (int ci = 0; ci < p.ncalls && ok; ci++) {
            const StepCall &c = p.calls[ci];
            const int k = c.k;
            if (ci > 0) {
                // every CTA's outputs of the calls before this one are written
                // (warp 0 waits as a whole: lane 0 reads, every decision is the warp's)
                bool failed = false;
                if (warp == 0) {
                    const unsigned int want = (unsigned int)ci * gridDim.x;
                    const unsigned long long t0 = dev::now_ns();
                    while (true) {
                        const unsigned int v = __shfl_sync(kFull, lane == 0 ? ld_acquire(p.counter) : 0u, 0);
                        if (v >= want) break;
                        const int why = __shfl_sync(
                            kFull, lane == 0 ? (*abort_v ? 1 : (dev::now_ns() - t0 > p.timeout_ns ? 2 : 0)) : 0, 0);
                        if (why != 0) {
                            if (why == 2 && lane == 0) {
                                *abort_v = 1;
                                atomicExch(p.err, dev::kTimeoutStatus);
                            }
                            failed = true;
                            break;
                        }
                        __nanosleep(32);
                    }
                }
                if (consumers_agree_stop(failed)) break;
            }
            // the activation, rounded to f16 (bm_to_f16's bits), read through L2: it may have
            // been written during this launch by another SM
            {
                const float4 *xf = reinterpret_cast<const float4 *>(c.x);
                uint2 *xo = reinterpret_cast<uint2 *>(xs);
                for (int i = threadIdx.x; i < (k >> 2); i += 32 * kConsumerWarps) {
                    const float4 v = ld_cg4(xf + i);
                    xo[i] = make_uint2(pack_rn(v.x, v.y), pack_rn(v.z, v.w));
                }
            }
            consumers_sync();
            const int nsteps = k >> 5;
            int glo, ghi;
            my_groups(c, glo, ghi);
            for (int g = glo; g < ghi && ok;) {
                const int m = matrix_of(c, g);
                const int ng = min(kGroupsPerBlock, min(ghi, c.gbeg[m + 1]) - g);
                const int bpg = boxes_per_group(ng);
                const int sw = bpg * kBoxCols;
                const int nslices = (k + sw - 1) / sw;
                const int row = (g - c.gbeg[m] + warp) * kGroupRows + rho;
                const bool active = warp < ng;
                const int rows = c.rows[m];
                float acc[8];
#pragma unroll
                for (int e = 0; e < 8; e++) acc[e] = 0.0f;
                for (int sl = 0; sl < nslices; sl++, t++) {
                    const int slot = t % S;
                    const uint32_t ph = (uint32_t)(t / S) & 1u;
                    if (!dev::mbar_wait_warp(dev::smem_u32(&full_bar[slot]), ph, abort_v, p.timeout_ns, p.err)) {
                        ok = false;
                        break;
                    }
                    const int kc0 = sl * sw;
                    const uint8_t *rbase = smem + xbytes + (size_t)slot * kStageBytes + (size_t)(warp * bpg) * kBoxBytes +
                                           rho * 128;
                    if (active) {
                        const int nst = min(2 * bpg, nsteps - kc0 / 32);
                        int s = 0;
                        for (; s + 2 <= nst; s += 2) {
                            const uint8_t *bx = rbase + (s >> 1) * kBoxBytes;
                            const uint4 w0 = *reinterpret_cast<const uint4 *>(bx + ((j) ^ rho) * 16);
                            const uint4 w1 = *reinterpret_cast<const uint4 *>(bx + ((4 + j) ^ rho) * 16);
                            const int S0 = kc0 / 32 + s;
                            fma8(acc, w0, x4[4 * S0]);
                            fma8(acc, w1, x4[4 * S0 + 4]);
                        }
                        if (s < nst) {
                            const uint8_t *bx = rbase + (s >> 1) * kBoxBytes;
                            const uint4 w0 = *reinterpret_cast<const uint4 *>(bx + ((j) ^ rho) * 16);
                            fma8(acc, w0, x4[4 * (kc0 / 32 + s)]);
                        }
                    }
                    if (sl == nslices - 1) {
#pragma unroll
                        for (int e = 0; e < 8; e++) acc[e] += __shfl_xor_sync(kFull, acc[e], 2);
#pragma unroll
                        for (int e = 0; e < 8; e++) acc[e] += __shfl_xor_sync(kFull, acc[e], 1);
                        const float t0 = acc[0] + acc[4], t1 = acc[1] + acc[5], t2 = acc[2] + acc[6], t3 = acc[3] + acc[7];
                        const float red = (t0 + t1) + (t2 + t3);
                        if (active && j == 0 && row < rows) {
                            float out = red;
                            if (32 * nsteps < k) {
                                double sum = (double)red;
                                for (int e = 32 * nsteps; e < k; e++) {
                                    const int cc = e - kc0;
                                    const int b = cc >> 6, col = ((cc & 63) >> 3) ^ rho;
                                    const uint16_t w =
                                        *reinterpret_cast<const uint16_t *>(rbase + b * kBoxBytes + col * 16 + (cc & 7) * 2);
                                    sum += (double)__fmul_rn(widen(w), widen(xs[e]));
                                }
                                out = (float)sum;
                            }
                            c.y[m][row] = out;
                        }
                    }
                    __syncwarp();
                    if (lane == 0) dev::mbar_arrive(dev::smem_u32(&empty_bar[slot]));
                }
                g += ng;
            }
            // this CTA's outputs of the call are written (and its reads of the activation done)
            if (consumers_agree_stop(!ok)) break;
            if (threadIdx.x == 0) {
                if (ci + 1 < p.ncalls) {
                    // release: this CTA's outputs (ordered before by the consumer barrier) are
                    // visible to whoever reads the count with acquire
                    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.counter) : "memory");
                } else {
                    unsigned int done;
                    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(done) : "l"(p.counter) : "memory");
                    if (done + 1u == (unsigned int)p.ncalls * gridDim.x) atomicExch(p.counter, 0u);  // the step's last CTA
                }
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncthreads();
    if (*abort_v && threadIdx.x == 0) {
        const int issued = issued_slot;
        for (int s = 0; s < S && s < issued; s++) {
            const int last = issued - 1 - ((issued - 1 - s) % S);
            dev::mbar_drain(dev::smem_u32(&full_bar[s]), (uint32_t)(last / S) & 1u, p.timeout_ns);
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

constexpr int kMaxDevices = 64;
std::once_flag g_attr_once[kMaxDevices];

}  // namespace

// A recorded step: the calls in device memory, the grid counter, the launch shape.
struct StepPlan {
    int device;
    StepCall *calls;         // device
    unsigned int *counter;   // device, zero between runs
    int ncalls, kmax, stages, grid;
    size_t smem;
};

int step_create(const bm_matvec_call *calls, int ncalls, const DeviceInfo &dev, void **out)
{
    if (!encoder()) return fail(BM_ERR_CUDA, "bm_step_create: cuTensorMapEncodeTiled unavailable");
    StepCall *host = static_cast<StepCall *>(::operator new[](sizeof(StepCall) * (size_t)ncalls, std::align_val_t(128)));
    memset(static_cast<void *>(host), 0, sizeof(StepCall) * (size_t)ncalls);
    int kmax = 8;
    int64_t max_groups = 1;
    for (int i = 0; i < ncalls; i++) {
        const bm_matvec_call &c = calls[i];
        StepCall &h = host[i];
        h.k = (int)c.k;
        h.x = c.x;
        h.gbeg[0] = 0;
        int n = 0;
        for (int m = 0; m < c.nmat; m++) {
            if (c.rows[m] == 0) continue;
            if (!make_row_map(&h.map[n], c.W[m], c.rows[m], c.k)) {
                ::operator delete[](host, std::align_val_t(128));
                return fail(BM_ERR_CUDA, "bm_step_create: tensor map encoding failed (call %d)", i);
            }
            h.y[n] = c.y[m];
            h.rows[n] = (int)c.rows[m];
            h.gbeg[n + 1] = h.gbeg[n] + (int)((c.rows[m] + kGroupRows - 1) / kGroupRows);
            n++;
        }
        h.nmat = n;
        for (int m = n; m < 4; m++) h.gbeg[m + 1] = h.gbeg[n];
        kmax = std::max(kmax, h.k);
        max_groups = std::max<int64_t>(max_groups, h.gbeg[n]);
    }
    const uint32_t xbytes = (uint32_t)((2 * (int64_t)kmax + 1023) / 1024 * 1024);
    const int64_t room = ((int64_t)dev.max_smem_optin / 2 - 2048 - 1024 - (int64_t)xbytes) / kStageBytes;
    if (room < 2) {
        ::operator delete[](host, std::align_val_t(128));
        return fail(BM_ERR_INVALID_ARG, "bm_step_create: k = %d leaves no room for two stages at two CTAs per SM", kmax);
    }
    StepPlan *plan = new (std::nothrow) StepPlan{};
    if (!plan) {
        ::operator delete[](host, std::align_val_t(128));
        return fail(BM_ERR_CUDA, "bm_step_create: out of host memory");
    }
    cudaGetDevice(&plan->device);
    plan->ncalls = ncalls;
    plan->kmax = kmax;
    plan->stages = (int)std::min<int64_t>(kMaxStages, room);
    plan->smem = xbytes + (size_t)plan->stages * kStageBytes + 1024;
    std::call_once(g_attr_once[plan->device & (kMaxDevices - 1)], [&] {
        cudaFuncSetAttribute(k_gemv_step, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.max_smem_optin - 1024);
    });
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_gemv_step, kThreads, plan->smem) != cudaSuccess ||
        per_sm < 1) {
        cudaGetLastError();
        ::operator delete[](host, std::align_val_t(128));
        delete plan;
        return fail(BM_ERR_CUDA, "bm_step_create: the step kernel does not fit on an SM");
    }
    // every CTA waits for all others between calls: all must be resident (cooperative launch)
    plan->grid = (int)std::min<int64_t>((int64_t)dev.sm_count * std::min(per_sm, 2), std::max<int64_t>(max_groups, 1));
    cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&plan->calls), sizeof(StepCall) * (size_t)ncalls);
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void **>(&plan->counter), 256);
    if (e == cudaSuccess)
        e = cudaMemcpy(plan->calls, host, sizeof(StepCall) * (size_t)ncalls, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(plan->counter, 0, 256);
    ::operator delete[](host, std::align_val_t(128));
    if (e != cudaSuccess) {
        cudaFree(plan->calls);
        cudaFree(plan->counter);
        delete plan;
        return fail(BM_ERR_CUDA, "bm_step_create: device set-up failed: %s", cudaGetErrorString(e));
    }
    *out = plan;
    return BM_OK;
}

int step_run(void *handle, cudaStream_t s)
{
    StepPlan *plan = static_cast<StepPlan *>(handle);
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess || d != plan->device)
        return fail(BM_ERR_INVALID_ARG, "bm_step_run: the step was recorded on device %d", plan->device);
    StepParams prm{};
    prm.calls = plan->calls;
    prm.ncalls = plan->ncalls;
    prm.kmax = plan->kmax;
    prm.stages = plan->stages;
    prm.counter = plan->counter;
    prm.err = device_error_word();
    if (!prm.err) return fail(BM_ERR_CUDA, "bm_step_run: device error word unavailable");
    prm.timeout_ns = kTimeoutNs;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)plan->grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = plan->smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_gemv_step, prm);
    if (e != cudaSuccess) return fail(BM_ERR_CUDA, "bm_step_run: launch failed: %s", cudaGetErrorString(e));
    return BM_OK;
}

void step_destroy(void *handle)
{
    StepPlan *plan = static_cast<StepPlan *>(handle);
    if (!plan) return;
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != plan->device) cudaSetDevice(plan->device);
    cudaFree(plan->calls);
    cudaFree(plan->counter);
    if (cur >= 0 && cur != plan->device) cudaSetDevice(cur);
    delete plan;
}

}  // namespace bm
