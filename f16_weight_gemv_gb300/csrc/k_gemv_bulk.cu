// k_gemv_bulk.cu -- the one-column product (ggml_vec_dot_f16 per row, bit for
// bit) for rows that are not 16-byte aligned (k % 8 != 0), streamed through
// shared memory by 1-D bulk copies.
//
// The order is that of the page "docs/modules/f16.md" (Design notes, "vec_dot"),
// as in k_gemv_stream.cu: 32 f32 chains per row (element 32s + 8j + l feeds
// accumulator j, lane l), each adding its products in increasing s from +0; then
// (a0+a2)+(a1+a3), low four lanes + high four lanes, two horizontal adds, and the
// k%32 tail added in double in order.
//
// A row of k % 8 != 0 elements starts 2 * (r * k mod 8) bytes past a 16-byte
// boundary, so it cannot be described by a tiled tensor map.  Each row's share of
// a k-slice is brought in instead by one bulk copy of its 16-byte-aligned window:
// from the boundary at or below the slice's first element to the boundary at or
// above its last, into a slot of its own in the stage.  Consumer thread j of a
// row's four reads, for each 32-element step, the two aligned 16-byte chunks that
// hold elements 32s + 8j .. +7 and cuts those eight out (a word shift by selects
// and a 2-byte shift by byte permutes, both fixed per row), so the chains see
// exactly the elements, in exactly the order, of the page's steps.  Slots are
// 2 * slice + 64 bytes apart (an odd multiple of 64 bytes), so the two rows of
// every 8-lane phase read disjoint banks.
//
// Work split, ring and waits as in k_gemv_stream.cu: 8-row groups of all
// matrices split evenly between the CTAs, sub-blocks of up to eight groups, 16
// issuing lanes in four producer warps each arriving on the stage's barrier with
// its own byte count; the weight copies start before griddepcontrol.wait, the
// activation (16-byte aligned) is staged after it.  The copy of the matrix's very
// last window stops at the last whole 16 bytes inside the matrix; the few
// elements past that are read directly.  Every mbarrier wait is bounded; on a
// give-up the CTA records BM_ERR_TIMEOUT, drains its copies (bounded) and exits.
#include "../../include/bm.h"
#include "bm_device.cuh"
#include "bm_internal.h"

#include <cuda_fp16.h>

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
constexpr int kGroupsPerBlock = kConsumerWarps;
constexpr int kMaxStages = 8;
constexpr unsigned long long kTimeoutNs = 2000000000ull;
constexpr unsigned kFull = 0xffffffffu;

// Slice width (elements) of a sub-block of ng groups: 256 for 5..8 groups, doubling as
// the groups halve, so a stage holds about the same bytes at any sub-block size and each
// row's copy is at least 528 bytes.
__host__ __device__ __forceinline__ int slice_width(int ng) { return ng <= 1 ? 2048 : ng <= 2 ? 1024 : ng <= 4 ? 512 : 256; }
// A row's slot: the slice, up to 7 leading elements of its window, padding.
__host__ __device__ __forceinline__ int slot_pitch(int sw) { return 2 * sw + 64; }
constexpr uint32_t kStageBytes = kGroupsPerBlock * kGroupRows * (2 * 256 + 64);  // 36 KB, the largest stage
constexpr int kUnroll = 4;  // chain steps whose shared-memory reads are issued together

struct BulkJob {
    const uint16_t *W[4];
    float *y[4];
    int64_t rows[4];
    int64_t gbeg[5];  // first 8-row group of matrix m; gbeg[nmat] = total groups
    const uint16_t *x;  // f16 activation, 16-byte aligned
    int64_t k;
    int nmat;
    int stages;
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

// Elements 2q + odd .. +7 of the 16 elements in lo:hi as four words: a shift by q words
// (selects) and by `odd` halves (byte permute `sel`: 0x5432 odd, 0x3210 even).
__device__ __forceinline__ uint4 cut(const uint4 &lo, const uint4 &hi, int q, uint32_t sel)
{
    const bool s2 = (q & 2) != 0, s1 = (q & 1) != 0;
    const uint32_t t0 = s2 ? lo.z : lo.x, t1 = s2 ? lo.w : lo.y, t2 = s2 ? hi.x : lo.z, t3 = s2 ? hi.y : lo.w,
                   t4 = s2 ? hi.z : hi.x, t5 = s2 ? hi.w : hi.y;
    const uint32_t u0 = s1 ? t1 : t0, u1 = s1 ? t2 : t1, u2 = s1 ? t3 : t2, u3 = s1 ? t4 : t3, u4 = s1 ? t5 : t4;
    return make_uint4(__byte_perm(u0, u1, sel), __byte_perm(u1, u2, sel), __byte_perm(u2, u3, sel),
                      __byte_perm(u3, u4, sel));
}

// Eight elements of the matrix from element e0 on, those at or past `total` as zero.
__device__ __forceinline__ uint4 ld_direct(const uint16_t *W, int64_t e0, int64_t total)
{
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const uint32_t lo = e0 + 2 * i < total ? W[e0 + 2 * i] : 0u;
        const uint32_t hi = e0 + 2 * i + 1 < total ? W[e0 + 2 * i + 1] : 0u;
        w[i] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ int matrix_of(const BulkJob &job, int64_t g)
{
    int m = 0;
#pragma unroll
    for (int q = 1; q < 4; q++)
        if (q < job.nmat && g >= job.gbeg[q]) m = q;
    return m;
}

// Elements of row r's window for the slice at column c0 that its bulk copy brings:
// from the 16-byte boundary below the slice's first element up to the boundary above
// min(c0 + sw, k), stopping at the last whole 16 bytes inside the matrix.
__device__ __forceinline__ int64_t window_elems(int64_t r, int64_t k, int64_t c0, int sw, int64_t total)
{
    const int64_t start = r * k;
    const int64_t d = start & 7;
    const int64_t src = start - d + c0;
    const int64_t want = (d + min((int64_t)sw, k - c0) + 7) & ~(int64_t)7;
    const int64_t room = (total - src) & ~(int64_t)7;
    return min(want, room);
}

__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps)); }

__global__ void __launch_bounds__(kThreads, 2) k_gemv_bulk(const __grid_constant__ BulkJob job)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ int abort_flag;
    __shared__ int issued_slot;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t k = job.k;
    const int S = job.stages;
    const int64_t nchunk = (k + 7) >> 3;  // 16-byte chunks of the activation
    const uint32_t xbytes = (uint32_t)((nchunk * 16 + 127) & ~127);
    uint8_t *smem = smem_raw + ((128u - (dev::smem_u32(smem_raw) & 127u)) & 127u);
    uint4 *xs4 = reinterpret_cast<uint4 *>(smem);
    uint8_t *ring = smem + xbytes;
    const uint32_t ring_u = dev::smem_u32(ring);
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

    const int64_t G = job.gbeg[job.nmat];
    const int64_t glo = G * blockIdx.x / gridDim.x, ghi = G * (blockIdx.x + 1) / gridDim.x;
    const int64_t nsteps = k >> 5;

    if (warp >= kConsumerWarps) {
        // ------------------------------------------------------------ producers
        int t = 0;
        bool ok = true;
        const int me = (warp - kConsumerWarps) * kIssuersPerWarp + lane;
        for (int64_t g = glo; g < ghi && ok;) {
            const int m = matrix_of(job, g);
            const int ng = (int)min((int64_t)kGroupsPerBlock, min(ghi, job.gbeg[m + 1]) - g);
            const int sw = slice_width(ng), pitch = slot_pitch(sw);
            const int64_t nslices = (k + sw - 1) / sw;
            const int64_t rows = job.rows[m], total = rows * k;
            const int64_t row0 = (g - job.gbeg[m]) * kGroupRows;
            const uint16_t *W = job.W[m];
            for (int64_t sl = 0; sl < nslices; sl++, t++) {
                const int slot = t % S;
                const uint32_t ph = (uint32_t)(t / S) & 1u;
                if (!dev::mbar_wait_warp(dev::smem_u32(&empty_bar[slot]), ph ^ 1u, abort_v, job.timeout_ns, job.err)) {
                    ok = false;
                    break;
                }
                const int64_t c0 = sl * sw;
                if (lane < kIssuersPerWarp) {
                    const uint32_t fb = dev::smem_u32(&full_bar[slot]);
                    const uint32_t dst0 = ring_u + (uint32_t)slot * kStageBytes;
                    uint32_t bytes = 0;
                    for (int i = me; i < kGroupRows * ng; i += kIssuers) {
                        const int64_t r = row0 + i;
                        if (r < rows) bytes += 2u * (uint32_t)window_elems(r, k, c0, sw, total);
                    }
                    dev::mbar_expect_tx(fb, bytes);
                    for (int i = me; i < kGroupRows * ng; i += kIssuers) {
                        const int64_t r = row0 + i;
                        if (r >= rows) continue;
                        const int64_t n = window_elems(r, k, c0, sw, total);
                        if (n > 0)
                            dev::bulk_g2s(dst0 + (uint32_t)(i * pitch), W + (r * k - ((r * k) & 7) + c0),
                                          2u * (uint32_t)n, fb);
                    }
                }
                if (warp == kConsumerWarps && lane == 0) issued_slot = t + 1;
            }
            g += ng;
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ consumers
        dev::pdl_wait();  // the activation is the previous kernel's output; outputs follow too
        const uint4 *xg = reinterpret_cast<const uint4 *>(job.x);
        {
            // in batches of eight loads, all in flight before the first store
            constexpr int kBatch = 8, kT = 32 * kConsumerWarps;
            for (int64_t i0 = threadIdx.x; i0 < nchunk; i0 += kBatch * kT) {
                uint4 h[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; u++) {
                    const int64_t i = i0 + u * kT;
                    h[u] = i >= nchunk ? make_uint4(0u, 0u, 0u, 0u)
                                       : 8 * i + 8 <= k ? __ldg(xg + i) : ld_direct(job.x, 8 * i, k);
                }
#pragma unroll
                for (int u = 0; u < kBatch; u++)
                    if (i0 + u * kT < nchunk) xs4[i0 + u * kT] = h[u];
            }
        }
        consumers_sync();

        const int j = lane & 3, tr = lane >> 2;  // accumulator j; row tr of the group
        const uint4 *x4 = xs4 + j;                 // x[32s + 8j] at x4[4s]
        const uint16_t *xs = reinterpret_cast<const uint16_t *>(xs4);
        bool ok = true;
        int t = 0;
        for (int64_t g = glo; g < ghi && ok;) {
            const int m = matrix_of(job, g);
            const int ng = (int)min((int64_t)kGroupsPerBlock, min(ghi, job.gbeg[m + 1]) - g);
            const int sw = slice_width(ng), pitch = slot_pitch(sw);
            const int64_t nslices = (k + sw - 1) / sw;
            const int64_t rows = job.rows[m], total = rows * k;
            const int64_t row = (g - job.gbeg[m]) * kGroupRows + warp * kGroupRows + tr;
            const bool active = warp < ng;  // warp-uniform
            const bool valid = active && row < rows;
            const int64_t start = row * k;
            const int d = (int)(start & 7);
            const int q = d >> 1;
            const uint32_t sel = (d & 1) ? 0x5432u : 0x3210u;
            const uint16_t *W = job.W[m];
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; e++) acc[e] = 0.0f;
            for (int64_t sl = 0; sl < nslices; sl++, t++) {
                const int slot = t % S;
                const uint32_t ph = (uint32_t)(t / S) & 1u;
                if (!dev::mbar_wait_warp(dev::smem_u32(&full_bar[slot]), ph, abort_v, job.timeout_ns, job.err)) {
                    ok = false;
                    break;
                }
                const int64_t c0 = sl * sw;
                const uint8_t *rslot = ring + (size_t)slot * kStageBytes + (size_t)(warp * kGroupRows + tr) * pitch;
                const uint4 *rs4 = reinterpret_cast<const uint4 *>(rslot) + j;
                if (valid) {
                    // chunks of this row's window that its copy brought (all but at the matrix's end)
                    const int64_t have = window_elems(row, k, c0, sw, total) >> 3;
                    const int nst = (int)min((int64_t)(sw >> 5), nsteps - (c0 >> 5));  // chain steps in this slice
                    const int64_t wbase = start - d + c0;  // the window's first element
                    const int need = d != 0 ? 2 : 1;  // chunks that hold a step's eight elements
                    // steps whose chunks all came with the copy (every step but the matrix's last
                    // few): 4s + j + need <= have
                    const int64_t slack = have - need - j;  // step s is safe while 4s <= slack
                    const int sfast = slack < 0 ? 0 : (int)min((int64_t)nst, slack / 4 + 1);
                    const uint4 *xq = x4 + 4 * (c0 >> 5);
                    int s = 0;
                    for (; s + kUnroll <= sfast; s += kUnroll) {
                        uint4 lo[kUnroll], hi[kUnroll], xv[kUnroll];
#pragma unroll
                        for (int u = 0; u < kUnroll; u++) {
                            lo[u] = rs4[4 * (s + u)];
                            hi[u] = rs4[4 * (s + u) + 1];  // unused when d == 0
                            xv[u] = xq[4 * (s + u)];
                        }
#pragma unroll
                        for (int u = 0; u < kUnroll; u++) fma8(acc, cut(lo[u], hi[u], q, sel), xv[u]);
                    }
                    for (; s < sfast; s++) fma8(acc, cut(rs4[4 * s], rs4[4 * s + 1], q, sel), xq[4 * s]);
                    for (; s < nst; s++) {
                        const int c = 4 * s + j;
                        const uint4 lo = c < have ? rs4[4 * s] : ld_direct(W, wbase + 8 * c, total);
                        const uint4 hi = need == 2 ? ld_direct(W, wbase + 8 * (c + 1), total) : lo;
                        fma8(acc, cut(lo, hi, q, sel), xq[4 * s]);
                    }
                }
                if (sl == nslices - 1) {
#pragma unroll
                    for (int e = 0; e < 8; e++) acc[e] += __shfl_xor_sync(kFull, acc[e], 2);
#pragma unroll
                    for (int e = 0; e < 8; e++) acc[e] += __shfl_xor_sync(kFull, acc[e], 1);
                    const float t0 = acc[0] + acc[4], t1 = acc[1] + acc[5], t2 = acc[2] + acc[6], t3 = acc[3] + acc[7];
                    const float red = (t0 + t1) + (t2 + t3);
                    if (valid && j == 0) {
                        float out = red;
                        if (32 * nsteps < k) {
                            // the tail lies in this last slice's window (c0 <= 32 * nsteps)
                            const int64_t have_e = window_elems(row, k, c0, sw, total);
                            const uint16_t *rsl = reinterpret_cast<const uint16_t *>(rslot);
                            double sum = (double)red;
                            for (int64_t e = 32 * nsteps; e < k; e++) {
                                const int64_t we = d + (e - c0);  // element of the window
                                const uint16_t w = we < have_e ? rsl[we] : W[start + e];
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
        const int issued = issued_slot;
        for (int s = 0; s < S && s < issued; s++) {
            const int last = issued - 1 - ((issued - 1 - s) % S);
            dev::mbar_drain(dev::smem_u32(&full_bar[s]), (uint32_t)(last / S) & 1u, job.timeout_ns);
        }
    }
    __syncthreads();
}

constexpr int kMaxDevices = 64;
std::once_flag g_attr_once[kMaxDevices];

}  // namespace

int launch_gemv_bulk(const VecdotJob &vj, cudaStream_t s, const DeviceInfo &dev)
{
    BulkJob job{};
    job.nmat = vj.nmat;
    job.k = vj.k;
    job.x = vj.X;
    job.gbeg[0] = 0;
    for (int m = 0; m < vj.nmat; m++) {
        job.W[m] = vj.W[m];
        job.y[m] = vj.y[m];
        job.rows[m] = vj.rows[m];
        job.gbeg[m + 1] = job.gbeg[m] + (vj.rows[m] + kGroupRows - 1) / kGroupRows;
    }
    for (int m = vj.nmat; m < 4; m++) job.gbeg[m + 1] = job.gbeg[vj.nmat];
    const int64_t G = job.gbeg[vj.nmat];
    if (G == 0) return BM_OK;
    job.err = device_error_word();
    if (!job.err) return fail(BM_ERR_CUDA, "vec_dot (bulk): device error word unavailable");
    job.timeout_ns = kTimeoutNs;

    const int64_t xbytes = (((vj.k + 7) / 8) * 16 + 127) & ~(int64_t)127;
    // two CTAs per SM with 2..8 stages; when the activation leaves no room for two stages
    // at two CTAs per SM (very long rows), one CTA per SM
    int64_t grid = std::min<int64_t>((int64_t)dev.sm_count * 2, G);
    int64_t room = ((int64_t)dev.max_smem_optin / 2 - 2048 - 1024 - xbytes) / kStageBytes;
    if (room < 2) {
        grid = std::min<int64_t>(grid, dev.sm_count);
        room = ((int64_t)dev.max_smem_optin - 2048 - 1024 - xbytes) / kStageBytes;  // >= 4 for k <= BM_MAX_K
    }
    if (room < 2) return fail(BM_ERR_INVALID_ARG, "vec_dot (bulk): k too large");
    job.stages = (int)std::min<int64_t>(kMaxStages, room);
    const size_t smem = (size_t)xbytes + (size_t)job.stages * kStageBytes + 128;

    int dev_id = 0;
    cudaGetDevice(&dev_id);
    std::call_once(g_attr_once[dev_id & (kMaxDevices - 1)], [&] {
        cudaFuncSetAttribute(k_gemv_bulk, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.max_smem_optin - 1024);
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
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_gemv_bulk, job);
    if (e != cudaSuccess) return fail(BM_ERR_CUDA, "vec_dot (bulk): launch failed: %s", cudaGetErrorString(e));
    return BM_OK;
}

}  // namespace bm
