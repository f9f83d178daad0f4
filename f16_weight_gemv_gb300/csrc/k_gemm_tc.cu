// k_gemm_tc.cu -- the multi-column product on tcgen05 tensor cores.
//
// Page "docs/modules/f16.md" (Summary; Design notes, "sgemm_dot"): a product
// of two or more columns takes tinyBLAS's path when the weight has a multiple
// of 4 rows and the row a multiple of 8 elements.  That path is a dense
// contraction, so here it runs on the 5th-generation tensor cores with f32
// accumulation: Y[c*rows + r] = sum_i W[r][i] * X[c][i].  The result is not
// tinyBLAS's bit pattern; it is within 4e-6 * sum_i |W[r][i] * X[c][i]| of it.
//
// Structure (one 128 x BN output tile per CTA, cta_group::1):
//   warp 0, one lane : TMA producer.  W tile 128 rows x 64 k and X tile BN
//                      columns x 64 k, both K-major with the 128-byte swizzle,
//                      into a ring of shared-memory stages (mbarrier complete_tx).
//   warp 1, one lane : MMA issuer.  Four tcgen05.mma (K = 16 each) per stage,
//                      accumulating in TMEM; tcgen05.commit frees the stage.
//   warps 0..3       : epilogue.  tcgen05.ld 32 lanes x 16 columns per trip and
//                      masked, coalesced f32 stores (a column of the tile is a
//                      contiguous run of rows in Y).
// Out-of-range rows, columns and the k % 64 end are zero-filled by TMA and add
// +0 exactly.  Every mbarrier wait is bounded by the global timer; on a
// give-up the CTA records BM_ERR_TIMEOUT in a device word, stops issuing
// work, waits (bounded) for the copies and MMAs it has in flight, frees its
// TMEM and exits.
#include "../../include/bm.h"
#include "bm_device.cuh"
#include "bm_internal.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>

namespace bm {

namespace {

constexpr int kBM = 128;          // tile rows (MMA M)
constexpr int kBK = 64;           // k per stage: one 128-byte swizzle row of f16
constexpr int kUmmaK = 16;        // k per tcgen05.mma of kind::f16
constexpr int kThreads = 128;
constexpr int kTileABytes = kBM * kBK * 2;  // 16 KB
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s

struct GemmParams {
    float *Y;
    int64_t rows, ncols, k;
    int num_kb;          // ceil(k / 64)
    int bn;              // tile columns (MMA N), multiple of 16, <= 256
    int stages;
    uint32_t tmem_cols;  // power of two >= 32, >= bn
    unsigned long long timeout_ns;
    unsigned int *err;        // device error word
    int withhold_first_load;  // self-test only: the producer never fills stage 0
};

// ----------------------------------------------------------------------------- PTX wrappers

using dev::mbar_expect_tx;
using dev::mbar_init;
using dev::mbar_try_wait;
using dev::now_ns;
using dev::smem_u32;

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                                  unsigned long long timeout_ns, unsigned int *err)
{
    return dev::mbar_wait(bar, parity, abort_flag, timeout_ns, err);
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

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand tile stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row core groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr)
{
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);   // start address
    d |= (uint64_t)(16u >> 4) << 16;            // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024u >> 4) << 32;          // stride byte offset: next 8-row group
    d |= (uint64_t)1 << 46;                     // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                     // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: f32 accumulator, f16 A and B, both K-major.
__host__ __device__ constexpr uint32_t instr_desc_f16(int m, int n)
{
    return (1u << 4)                         // D format: f32
           | (0u << 7) | (0u << 10)          // A, B format: f16
           | (0u << 15) | (0u << 16)         // A, B K-major
           | ((uint32_t)(n >> 3) << 17)      // N / 8
           | ((uint32_t)(m >> 4) << 24);     // M / 16
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ----------------------------------------------------------------------------- kernel

constexpr int kMaxStages = 8;

__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
              const GemmParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ __align__(8) uint64_t done_bar;
    __shared__ uint32_t tmem_base_slot;
    __shared__ int abort_flag;
    __shared__ int issued_slot, consumed_slot;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // 1024-byte alignment of the stage ring (the swizzle pattern repeats every 1024 bytes)
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t ring_u32 = smem_u32(ring);
    const uint32_t tile_b_bytes = (uint32_t)p.bn * kBK * 2;
    const uint32_t stage_bytes = kTileABytes + tile_b_bytes;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; s++) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        mbar_init(smem_u32(&done_bar), 1);
        abort_flag = 0;
        issued_slot = 0;
        consumed_slot = 0;
        dev::fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_base_slot)),
                     "r"(p.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = tmem_base_slot;

    const int64_t m0 = (int64_t)blockIdx.y * kBM;
    const int64_t n0 = (int64_t)blockIdx.x * p.bn;
    volatile int *abort_v = &abort_flag;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer
        int issued = 0;
        for (int kb = 0; kb < p.num_kb; kb++) {
            const int s = kb % p.stages;
            const uint32_t ph = (uint32_t)(kb / p.stages) & 1u;
            if (!mbar_wait_bounded(smem_u32(&empty_bar[s]), ph ^ 1u, abort_v, p.timeout_ns, p.err)) break;
            if (p.withhold_first_load && kb == 0) continue;  // self-test: stage 0 is never filled
            const uint32_t a_dst = ring_u32 + (uint32_t)s * stage_bytes;
            const uint32_t b_dst = a_dst + kTileABytes;
            const uint32_t fb = smem_u32(&full_bar[s]);
            mbar_expect_tx(fb, stage_bytes);
            tma_load_2d(a_dst, &map_w, kb * kBK, (int32_t)m0, fb);
            tma_load_2d(b_dst, &map_x, kb * kBK, (int32_t)n0, fb);
            issued = kb + 1;
        }
        issued_slot = issued;
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        const uint32_t idesc = instr_desc_f16(kBM, p.bn);
        int consumed = 0;
        for (int kb = 0; kb < p.num_kb; kb++) {
            const int s = kb % p.stages;
            const uint32_t ph = (uint32_t)(kb / p.stages) & 1u;
            if (!mbar_wait_bounded(smem_u32(&full_bar[s]), ph, abort_v, p.timeout_ns, p.err)) break;
            tc_fence_after();
            const uint32_t a_addr = ring_u32 + (uint32_t)s * stage_bytes;
            const uint32_t b_addr = a_addr + kTileABytes;
#pragma unroll
            for (int kk = 0; kk < kBK / kUmmaK; kk++) {
                const uint64_t ad = smem_desc_sw128(a_addr + kk * kUmmaK * 2);
                const uint64_t bd = smem_desc_sw128(b_addr + kk * kUmmaK * 2);
                mma_f16(tmem_d, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(smem_u32(&empty_bar[s]));  // the stage is free once these MMAs have read it
            consumed = kb + 1;
        }
        consumed_slot = consumed;
        mma_commit(smem_u32(&done_bar));  // always: signals when every issued MMA has finished
    }
    __syncwarp();

    // ---------------- epilogue: TMEM -> registers -> Y
    const bool done_ok = mbar_wait_bounded(smem_u32(&done_bar), 0, abort_v, p.timeout_ns, p.err);
    tc_fence_after();
    // tcgen05.ld is warp-collective: the decision must be the same for all 32 lanes.
    const bool go = __all_sync(0xffffffffu, done_ok && !*abort_v);
    if (go) {
        const int64_t row = m0 + warp * 32 + lane;
        const uint32_t t_row = tmem_d + ((uint32_t)(warp * 32) << 16);
        for (int c = 0; c < p.bn; c += 16) {
            uint32_t v[16];
            tmem_ld16(t_row + (uint32_t)c, v);
            if (row < p.rows) {
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    const int64_t col = n0 + c + i;
                    if (col < p.ncols) p.Y[col * p.rows + row] = __uint_as_float(v[i]);
                }
            }
        }
    }

    // ---------------- teardown
    tc_fence_before();
    __syncthreads();
    if (*abort_v && threadIdx.x == 0) {
        // Copies issued but never consumed must land before the CTA's shared memory goes away.
        for (int kb = consumed_slot; kb < issued_slot; kb++) {
            const int s = kb % p.stages;
            const uint32_t ph = (uint32_t)(kb / p.stages) & 1u;
            const unsigned long long t0 = now_ns();
            while (!mbar_try_wait(smem_u32(&full_bar[s]), ph) && now_ns() - t0 < p.timeout_ns) {
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_d), "r"(p.tmem_cols)
                     : "memory");
    }
}

// ----------------------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder()
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

// 2-D map over a row-major f16 matrix [outer][k], box = 64 k x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap *map, const uint16_t *base, int64_t outer, int64_t k, int box_rows)
{
    cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)k * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t *>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

uint32_t pow2_at_least(uint32_t v)
{
    uint32_t p = 32;
    while (p < v) p <<= 1;
    return p;
}

constexpr int kMaxDevices = 64;
std::once_flag g_attr_once[kMaxDevices];

int launch_impl(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols, float *Y,
                cudaStream_t s, const DeviceInfo &dev, unsigned long long timeout_ns, int withhold)
{
    if (!get_encoder()) return fail(BM_ERR_CUDA, "tensor-core product: cuTensorMapEncodeTiled unavailable");
    if (rows > 0x7fffffffLL || ncols > 0x7fffffffLL)
        return fail(BM_ERR_INVALID_ARG, "tensor-core product: rows and ncols must be below 2^31");
    GemmParams p{};
    p.Y = Y;
    p.rows = rows;
    p.ncols = ncols;
    p.k = k;
    p.num_kb = (int)((k + kBK - 1) / kBK);
    const int64_t n16 = (ncols + 15) / 16 * 16;
    p.bn = (int)(n16 < 256 ? n16 : 256);
    p.tmem_cols = pow2_at_least((uint32_t)p.bn);
    const int stage_bytes = kTileABytes + p.bn * kBK * 2;
    const int budget = dev.max_smem_optin - 1024 - 1024;  // alignment slack and static shared memory
    p.stages = budget / stage_bytes;
    if (p.stages > kMaxStages) p.stages = kMaxStages;
    if (p.stages < 2) return fail(BM_ERR_CUDA, "tensor-core product: not enough shared memory");
    p.timeout_ns = timeout_ns;
    p.err = device_error_word();
    if (!p.err) return fail(BM_ERR_CUDA, "tensor-core product: device error word unavailable");
    p.withhold_first_load = withhold;

    CUtensorMap mw, mx;
    if (!make_map(&mw, W, rows, k, kBM) || !make_map(&mx, X, ncols, k, p.bn))
        return fail(BM_ERR_CUDA, "tensor-core product: tensor map encoding failed");

    int dev_id = 0;
    cudaGetDevice(&dev_id);
    std::call_once(g_attr_once[dev_id & (kMaxDevices - 1)], [&] {
        cudaFuncSetAttribute(k_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.max_smem_optin - 1024);
    });
    // One CTA per SM at most (the launch bounds and this shared-memory request),
    // so the TMEM allocations of co-resident CTAs never exceed 512 columns.
    const size_t smem = (size_t)p.stages * stage_bytes + 1024;
    const size_t one_per_sm = 120 * 1024;
    const size_t smem_req = smem < one_per_sm ? one_per_sm : smem;
    dim3 grid((unsigned)((ncols + p.bn - 1) / p.bn), (unsigned)((rows + kBM - 1) / kBM));
    if (grid.y > 65535u) return fail(BM_ERR_INVALID_ARG, "tensor-core product: too many row tiles");
    k_gemm_tc<<<grid, kThreads, smem_req, s>>>(mw, mx, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(BM_ERR_CUDA, "tensor-core product: launch failed: %s", cudaGetErrorString(e));
    return BM_OK;
}

}  // namespace

int launch_gemm_tc(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols, float *Y,
                   cudaStream_t s, const DeviceInfo &dev)
{
    return launch_impl(W, rows, k, X, ncols, Y, s, dev, kDefaultTimeoutNs, 0);
}

int launch_gemm_tc_withheld(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols, float *Y,
                            cudaStream_t s, const DeviceInfo &dev, unsigned long long timeout_ns)
{
    return launch_impl(W, rows, k, X, ncols, Y, s, dev, timeout_ns, 1);
}

}  // namespace bm
