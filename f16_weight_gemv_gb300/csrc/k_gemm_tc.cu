// k_gemm_tc.cu -- the multi-column product on tcgen05 tensor cores.
//
// Page "docs/modules/f16.md" (Summary; Design notes, "sgemm_dot"): a product
// of two or more columns takes tinyBLAS's path when the weight has a multiple
// of 4 rows and the row a multiple of 8 elements.  That path is a dense
// contraction, so here it runs on the 5th-generation tensor cores with f32
// accumulation: Y[c*rows + r] = sum_i W[r][i] * X[c][i].  The result is not
// tinyBLAS's bit pattern; it is within 4e-6 * sum_i |W[r][i] * X[c][i]| of it.
//
// Persistent, warp-specialised kernel (cta_group::1, one CTA per SM):
//   warp 0, one lane : TMA producer.  For each k-block a W tile (128 * MT rows x
//                      64) and an X tile (BN columns x 64), K-major with the
//                      128-byte swizzle, into a ring of shared-memory stages.
//   warp 1, one lane : MMA issuer.  4 * MT tcgen05.mma (M = 128, K = 16) per
//                      k-block into the unit's MT accumulators; tcgen05.commit
//                      frees the stage, and after a unit's last k-block signals
//                      the epilogue.  Warp 1 also owns the TMEM allocation.
//   warps 2..9       : epilogue, two warps per TMEM lane quarter (warp % 4),
//                      each taking every other 32-column chunk.  tcgen05.ld of
//                      the next chunk is in flight while the current chunk's
//                      coalesced f32 stores go out (a column of a tile is a
//                      contiguous run of rows in Y).  A 256 x 256 unit's
//                      epilogue takes about 6 us either way: when every CTA
//                      writes its tiles at once the stores run at HBM write
//                      speed.  The accumulators are handed back to the MMA warp
//                      once they have been read; when TMEM holds two sets
//                      (MT * BN <= 256) the epilogue of one unit overlaps the
//                      MMAs of the next.
// Work units are (row unit of MT tiles of 128 rows, column tile, k-split).  MT = 2
// lets two MMAs share each X tile, so a k-block moves 64 KB of operands for the
// work that takes 96 KB with MT = 1 -- the operand feed, not the tensor pipe, is
// what limits this kernel (the MMA sequence alone runs at full rate).  With S > 1
// splits each unit writes its partial tiles to a workspace (small enough to stay in
// L2 on the shapes that split), and k_splitk_reduce, launched right behind with
// programmatic dependent launch, sums the S partials of every element in split
// order 0..S-1 across the whole GPU -- so the result does not depend on which unit
// finished last, and the reduction runs with every SM's memory parallelism instead
// of in the tail of a few units.
//
// Balanced k ranges (stream-K, Osama et al., PPoPP 2023): when whole units leave
// part of the last wave idle, the CTAs are dealt to the column tiles in turn (CTA c
// serves column tile c % nt, so neighbouring CTAs read the same W rows at the same
// time and share them through L2, as in the unit order above), and each column's
// k-blocks, laid end to end (row unit after row unit, k fastest), are cut into one
// contiguous range per CTA of equal length.  A CTA walks its range from the top
// down, so the piece it shares with
// the CTA above (the start of a tile that continues there) comes first and is
// written to the CTA's own partial slot early; the piece it shares with the CTAs
// below (the end of a tile that started there) comes last, and the CTA that holds
// a tile's last k-block owns the tile: it adds the lower pieces in k order to its
// own accumulators and stores Y.  Each epilogue warp publishes its part of a piece
// with its own flag (a 64-bit token unique to the launch; the owner resets the
// flag to zero after reading), so no barrier spans warps and every wait is bounded.
// A CTA only ever waits for CTAs of lower index, which the GPU starts first.
// MT, the tile width, S and the mode come from a model of the predicted time (waves
// x per-unit time, plus the reduction or the owners' reads, calibrated by
// measurements).
//
// Out-of-range rows, columns and the k % 64 end are zero-filled by TMA and add
// +0 exactly.  Every mbarrier wait is bounded by the global timer; on a
// give-up the CTA records BM_ERR_TIMEOUT in the device error word, stops
// issuing work, waits (bounded) for the copies and MMAs it has in flight,
// frees its TMEM and exits.
#include "../../include/bm.h"
#include "bm_device.cuh"
#include "bm_internal.h"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstring>
#include <mutex>

namespace bm {

namespace {

constexpr int kBM = 128;          // tile rows (MMA M)
constexpr int kBK = 64;           // k per stage: one 128-byte swizzle row of f16
constexpr int kUmmaK = 16;        // k per tcgen05.mma of kind::f16
constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, splitting the columns
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kTileABytes = kBM * kBK * 2;  // 16 KB
constexpr int kMaxStages = 8;
constexpr int kPreWaitStages = 2;  // stages whose W copy is requested before griddepcontrol.wait
constexpr int kMaxSplits = 8;
constexpr int kMaxMats = 4;       // matrices sharing one activation in one launch
constexpr int kWarpChunks = 4;    // 32-column chunks per epilogue warp and row tile (bn <= 256)
constexpr int kOwnerDepth = 4;    // 4 KB blocks in flight per epilogue warp while an owner reads pieces
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s

// Up to kMaxMats matrices W[m] (rows[m] x k) times one activation X (ncols x k), each
// into its own Y[m] (ncols x rows[m]).  The matrices' row units are laid end to end:
// matrix m owns row units ubeg[m] .. ubeg[m+1]-1 and the split-k workspace's 128-row
// tiles tbeg[m] .. (its row units x MT).
struct GemmParams {
    float *Y[kMaxMats];
    int rows[kMaxMats];
    int ubeg[kMaxMats + 1];
    int tbeg[kMaxMats + 1];
    int nmat;
    float *ws;                // partial tiles, [tile][split][BN][128] (split count > 1 only)
    int ncols, k;
    int num_kb;               // ceil(k / 64)
    int bn;                   // tile columns (MMA N), multiple of 16, <= 256
    int bn_alloc;             // TMEM columns per accumulator: power of two >= max(32, bn)
    int nt;                   // column tiles
    int mtu;                  // row units of all matrices (MT row tiles each): ubeg[nmat]
    int nbuf;                 // TMEM accumulator sets: 2 (double-buffered) or 1
    int splits;
    int stages;
    // balanced k ranges (sk != 0; splits == 1): CTA c serves column tile c % nt and
    // takes iterations [iters * g / G, iters * (g + 1) / G) of that column's
    // iters = mtu x num_kb (row unit after row unit, k fastest), g = c / nt, G = grid / nt
    int sk;
    int64_t iters;
    float *skws;                 // one partial slot per CTA: 4 KB blocks [m][epilogue warp][chunk][col][lane]
    int64_t slot_floats;         // MT * kEpiWarps * kWarpChunks * 1024
    unsigned long long *flags;   // [CTA][epilogue warp]: token once the slot's part is written
    unsigned long long token;
    unsigned long long timeout_ns;
    unsigned int *err;        // device error word
    int withhold_first_load;  // self-test only: the producer never fills its first stage
};

using dev::mbar_expect_tx;
using dev::mbar_init;
using dev::mbar_try_wait;
using dev::now_ns;
using dev::smem_u32;

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

// 32 consecutive accumulator columns of this thread's TMEM lane.
// 32 lanes x 32 columns of TMEM into v; the values may be used only after tmem_wait_ld.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
}

// Waits for this thread's TMEM loads; the empty asm makes every later use of v depend
// on the wait, so no read of v is scheduled before the data has arrived.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&v)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    asm volatile(""
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                   "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]),
                   "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]),
                   "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]),
                   "+r"(v[29]), "+r"(v[30]), "+r"(v[31]));
}

// The tensor maps: one per weight matrix (box 64 x 128 * MT rows) and the activation's.
struct TmaMaps {
    CUtensorMap w[kMaxMats];
    CUtensorMap x;
};

// a[m] for a small parameter array, by compile-time indices only (a run-time index
// would copy the kernel's parameters to local memory)
template <class T, int N>
__device__ __forceinline__ T pick(const T (&a)[N], int m)
{
    T v = a[0];
#pragma unroll
    for (int q = 1; q < N; q++)
        if (m == q) v = a[q];
    return v;
}

struct Unit {
    int mat;    // the matrix
    int m0;     // first row of the unit in its matrix: MT row tiles of 128 rows
    int n0, s, kb0, kb1;
    int tile0;  // workspace index of the unit's first row tile (row tile t: tile0 + t * nt)
};

// Units are (row unit, column tile, k-split), ordered column tile fastest, then split,
// then row unit: CTAs that run side by side share a W block (the column tiles)
// through L2.
template <int MT>
__device__ __forceinline__ Unit unit_of(const GemmParams &p, int u)
{
    Unit x;
    const int nt = u % p.nt;
    const int rest = u / p.nt;
    x.s = rest % p.splits;
    const int mu = rest / p.splits;
    int m = 0;
#pragma unroll
    for (int q = 1; q < kMaxMats; q++)
        if (q < p.nmat && mu >= p.ubeg[q]) m = q;
    const int local = mu - pick(p.ubeg, m);
    x.mat = m;
    x.m0 = local * MT * kBM;
    x.n0 = nt * p.bn;
    x.tile0 = (pick(p.tbeg, m) + local * MT) * p.nt + nt;
    x.kb0 = p.num_kb * x.s / p.splits;  // num_kb < 2^25 (k < 2^31), s < splits <= 8: below 2^31
    x.kb1 = p.num_kb * (x.s + 1) / p.splits;
    return x;
}

// What the epilogue does with a segment's accumulators.
enum SegRole {
    kWhole = 0,  // all k-blocks of the tile: store Y
    kSplit = 1,  // one k-split: store the partial tile for k_splitk_reduce
    kPiece = 2,  // balanced ranges, not the tile's last k-block: this CTA's partial slot
    kOwner = 3,  // balanced ranges, the tile's last k-block after lower CTAs' pieces
};

// One stretch of k-blocks of one unit: what the producer, the MMA warp and the
// epilogue walk, in the same order.
struct Seg {
    Unit x;
    int kb0, kb1;
    int role;
    int cfirst, ncon;  // kOwner: CTAs cfirst + i * nt (i < ncon) hold the tile's earlier k-blocks
};

struct SegIter {
    int64_t beg, end;  // balanced ranges: this CTA's iterations
    int64_t t;         // the next tile (balanced ranges, walked downwards) or unit
    int64_t lo;        // balanced ranges: the lowest row unit of the range
};

__device__ __forceinline__ void seg_begin(const GemmParams &p, SegIter &it)
{
    if (p.sk) {
        const int64_t G = gridDim.x / p.nt, g = blockIdx.x / p.nt;
        it.beg = p.iters * g / G;
        it.end = p.iters * (g + 1) / G;
        it.t = it.end > it.beg ? (it.end - 1) / p.num_kb : -1;
        it.lo = it.beg / p.num_kb;
    } else {
        it.beg = it.end = it.lo = 0;
        it.t = blockIdx.x;
    }
}

// The range (of G per column tile) that holds iteration i: the largest g with
// floor(iters * g / G) <= i.
__device__ __forceinline__ int range_of(const GemmParams &p, int64_t i)
{
    const int64_t G = gridDim.x / p.nt;
    return (int)(((i + 1) * G + p.iters - 1) / p.iters) - 1;
}

template <int MT>
__device__ __forceinline__ bool seg_next(const GemmParams &p, SegIter &it, Seg &sg)
{
    if (p.sk) {
        // row unit it.t of column tile blockIdx.x % nt, walked downwards
        if (it.t < it.lo) return false;
        const int64_t t0 = it.t * p.num_kb;
        const int n = (int)(blockIdx.x % p.nt);
        sg.x = unit_of<MT>(p, (int)it.t * p.nt + n);
        sg.kb0 = (int)(max(it.beg, t0) - t0);
        sg.kb1 = (int)(min(it.end, t0 + p.num_kb) - t0);
        sg.cfirst = 0;
        sg.ncon = 0;
        if (sg.kb0 == 0 && sg.kb1 == p.num_kb) {
            sg.role = kWhole;
        } else if (sg.kb1 < p.num_kb) {
            sg.role = kPiece;  // the top of this CTA's range; at most one per CTA
        } else {
            sg.role = kOwner;
            const int g0 = range_of(p, t0);
            sg.cfirst = g0 * p.nt + n;
            sg.ncon = (int)(blockIdx.x / p.nt) - g0;
        }
        it.t--;
        return true;
    }
    const int units = p.mtu * p.nt * p.splits;
    if (it.t >= units) return false;
    sg.x = unit_of<MT>(p, (int)it.t);
    sg.kb0 = sg.x.kb0;
    sg.kb1 = sg.x.kb1;
    sg.role = p.splits > 1 ? kSplit : kWhole;
    sg.cfirst = 0;
    sg.ncon = 0;
    it.t += gridDim.x;
    return true;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *f)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(f) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long *f, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(f), "l"(v) : "memory");
}

// 16-byte asynchronous global -> shared copy (through L2 only) and its groups.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Waits until *f holds `token`; gives up on the CTA's abort flag or after timeout_ns
// (raising the flag and recording BM_ERR_TIMEOUT).
__device__ __forceinline__ bool flag_wait(const unsigned long long *f, unsigned long long token,
                                          volatile int *abort_flag, unsigned long long timeout_ns,
                                          unsigned int *err_word)
{
    if (ld_acquire_u64(f) == token) return true;
    const unsigned long long t0 = now_ns();
    while (true) {
        __nanosleep(100);
        if (ld_acquire_u64(f) == token) return true;
        if (*abort_flag) return false;
        if (now_ns() - t0 > timeout_ns) {
            *abort_flag = 1;
            atomicExch(err_word, dev::kTimeoutStatus);
            return false;
        }
    }
}

// Float offset of the 4 KB block (32 columns x 32 rows, column-major) that epilogue
// warp ew writes for its chunk j of row tile m in a partial slot.
__device__ __forceinline__ size_t slot_block(int m, int ew, int j)
{
    return ((size_t)(m * kEpiWarps + ew) * kWarpChunks + j) * 1024;
}

// The owner's epilogue of a tile whose earlier k-blocks lie in CTAs cfirst + i * nt:
// for each (row tile m, chunk j) of this warp, the accumulators plus every lower piece's
// block in CTA order, stored to Y.  The blocks come through the operand ring, idle by
// now (this is the CTA's last segment and its MMAs have completed): each warp owns
// kOwnerDepth 4 KB buffers there and keeps that many blocks in flight with cp.async.
template <int MT>
__device__ __forceinline__ void owner_epilogue(const GemmParams &p, const Seg &sg, uint32_t tacc, uint32_t ring_u32,
                                               uint8_t *smem_raw, int ew, int half, int quarter, int lane, int nch)
{
    // the ring's last readers were the tensor cores (async proxy); these are generic writes
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const int ncon = sg.ncon;
    const int jobs = MT * nch * ncon;  // (m, j, piece), piece fastest
    const uint32_t buf_u32 = ring_u32 + (uint32_t)ew * (kOwnerDepth * 4096u);
    const float *buf = reinterpret_cast<const float *>(smem_raw + (buf_u32 - smem_u32(smem_raw)));
    auto issue = [&](int n) {
        if (n < jobs) {
            const int cc = sg.cfirst + (n % ncon) * p.nt, mj = n / ncon;
            const float *src = p.skws + (size_t)cc * p.slot_floats + slot_block(mj / nch, ew, mj % nch);
            const uint32_t dst = buf_u32 + (uint32_t)(n % kOwnerDepth) * 4096u;
#pragma unroll
            for (int r = 0; r < 8; r++) cp_async16(dst + (uint32_t)(r * 32 + lane) * 16u, src + (r * 32 + lane) * 4);
        }
        cp_async_commit();  // one group per job slot, empty past the end: the wait count stays fixed
    };
#pragma unroll
    for (int n = 0; n < kOwnerDepth; n++) issue(n);
    const int rows = pick(p.rows, sg.x.mat);
    float *const Y = pick(p.Y, sg.x.mat);
    float acc[32];
    for (int n = 0; n < jobs; n++) {
        const int mj = n / ncon, m = mj / nch, j = mj % nch, c0 = 32 * (2 * j + half);
        if (n % ncon == 0) {
            uint32_t v[32];
            tmem_ld32(tacc + (uint32_t)(m * p.bn_alloc) + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c0, v);
            tmem_wait_ld(v);
#pragma unroll
            for (int q = 0; q < 32; q++) acc[q] = __uint_as_float(v[q]);
        }
        cp_async_wait<kOwnerDepth - 1>();  // this lane's copies of job n have landed
        __syncwarp();                      // and every other lane's
        const float *bk = buf + (n % kOwnerDepth) * 1024;
#pragma unroll
        for (int q = 0; q < 32; q++) acc[q] += bk[q * 32 + lane];
        __syncwarp();  // the buffer is read before it is refilled
        issue(n + kOwnerDepth);
        if (n % ncon == ncon - 1) {
            const int row = sg.x.m0 + m * kBM + quarter * 32 + lane;
            if (row < rows) {
#pragma unroll
                for (int q = 0; q < 32; q++) {
                    const int col = sg.x.n0 + c0 + q;
                    if (c0 + q < p.bn && col < p.ncols) Y[(size_t)col * rows + row] = acc[q];
                }
            }
        }
    }
    cp_async_wait<0>();
}

// MT = 1: a unit is 128 rows x BN columns.  MT = 2: 256 rows x BN columns, two
// M = 128 MMAs per k-step sharing the X tile, so each k-block moves 64 KB of operands
// for twice the work (32 KB per 128 x 256 x 64 block instead of 48 KB).  The
// accumulators of a unit take MT * BN TMEM columns; with room for two sets
// (p.nbuf == 2) the epilogue of one unit overlaps the MMAs of the next.
template <int MT>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_tc(const __grid_constant__ TmaMaps maps, const __grid_constant__ GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ __align__(8) uint64_t acc_full[2];
    __shared__ __align__(8) uint64_t acc_empty[2];
    __shared__ __align__(8) uint64_t done_bar;
    __shared__ uint32_t tmem_base_slot;
    __shared__ int abort_flag;
    __shared__ int issued_slot;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // 1024-byte alignment of the stage ring (the swizzle pattern repeats every 1024 bytes)
    const uint32_t ring_u32 = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t stage_bytes = MT * kTileABytes + (uint32_t)p.bn * kBK * 2;
    const uint32_t tmem_cols = (uint32_t)(p.nbuf * MT * p.bn_alloc);
    volatile int *abort_v = &abort_flag;

    if (threadIdx.x == 0) {
        // the TMA unit reads the tensor maps on first use: fetch them while the set-up runs
        for (int m = 0; m < p.nmat; m++)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.w[m])) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.x)) : "memory");
        for (int s = 0; s < p.stages; s++) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < p.nbuf; b++) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            mbar_init(smem_u32(&acc_empty[b]), kEpiWarps);
        }
        mbar_init(smem_u32(&done_bar), 1);
        abort_flag = 0;
        issued_slot = 0;
        dev::fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_base_slot)),
                     "r"(tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_slot;
    dev::pdl_trigger();  // the next kernel may start its own set-up and weight loads

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            // Under programmatic dependent launch the weights (constants) of the first
            // stages are requested before griddepcontrol.wait; the activation tiles (the
            // previous kernel's output) only after it.
            // Everything the loop needs is hoisted into registers and the stage and its
            // phase advance by increments: this one thread's per-k-block instruction chain
            // (divisions, parameter loads) otherwise took longer than the copies it issues.
            const int stages = p.stages;
            // W copies requested before griddepcontrol.wait: the engine serves copies in
            // order, so every W box queued ahead delays the first X tile (and the first
            // MMA) when the kernel ahead has already finished; two stages keep that
            // delay short and still start the weights early when it has not.
            const int pre_wait = stages < kPreWaitStages ? stages : kPreWaitStages;
            const int withhold = p.withhold_first_load;
            const unsigned long long tmo = p.timeout_ns;
            unsigned int *const errw = p.err;
            const uint32_t full0 = smem_u32(&full_bar[0]), empty0 = smem_u32(&empty_bar[0]);
            int t = 0;        // k-blocks walked
            int st = 0;       // the stage of k-block t
            uint32_t ph = 0;  // and the parity of its phase
            bool ok = true, waited = false;
            int pend = 0;  // stages that hold their W copy, X still to come: k-blocks 0 .. pend-1
            // (walked again rather than remembered: stores to a local array before each
            // barrier arrive cost a memory round trip per k-block)
            auto issue_pending_x = [&]() {
                dev::pdl_wait();
                waited = true;
                SegIter it2;
                seg_begin(p, it2);
                Seg s2;
                int q = 0;
                while (q < pend && seg_next<MT>(p, it2, s2))
                    for (int kb = s2.kb0; kb < s2.kb1 && q < pend; kb++, q++)
                        if (!(withhold && q == 0))
                            tma_load_2d(ring_u32 + (uint32_t)q * stage_bytes + MT * kTileABytes, &maps.x, kb * kBK,
                                        s2.x.n0, full0 + 8u * (uint32_t)q);
                pend = 0;
            };
            SegIter it;
            seg_begin(p, it);
            Seg sg;
            while (ok && seg_next<MT>(p, it, sg)) {
                const CUtensorMap *wmap = &maps.w[sg.x.mat];
                const int32_t m0 = sg.x.m0, n0 = sg.x.n0;
                for (int kb = sg.kb0; kb < sg.kb1; kb++) {
                    if (!dev::mbar_wait(empty0 + 8u * (uint32_t)st, ph ^ 1u, abort_v, tmo, errw)) {
                        ok = false;
                        break;
                    }
                    if (withhold && t == 0) {  // self-test: stage 0 is never filled
                        pend++;
                        if (t + 1 == pre_wait) issue_pending_x();
                    } else {
                        const uint32_t a_dst = ring_u32 + (uint32_t)st * stage_bytes;
                        const uint32_t fb = full0 + 8u * (uint32_t)st;
                        mbar_expect_tx(fb, stage_bytes);
                        tma_load_2d(a_dst, wmap, kb * kBK, m0, fb);  // MT * 128 rows in one box
                        if (waited) {
                            tma_load_2d(a_dst + MT * kTileABytes, &maps.x, kb * kBK, n0, fb);
                        } else {  // t < stages here: k-block t fills stage t
                            pend++;
                            if (t + 1 == pre_wait) issue_pending_x();
                        }
                    }
                    t++;
                    if (++st == stages) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            }
            issued_slot = t;
            if (!waited) issue_pending_x();  // fewer k-blocks than stages, or a give-up: complete every stage
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            // Hoisted and incremental as in the producer.  The operand descriptors of a
            // stage differ from the ring's first one only in the start address field
            // (address / 16, below 2^14 for any shared-memory address), so each is that
            // descriptor plus an offset.
            const uint32_t idesc = instr_desc_f16(kBM, p.bn);
            const int stages = p.stages, nbuf = p.nbuf;
            const uint32_t bn_alloc = (uint32_t)p.bn_alloc;
            const unsigned long long tmo = p.timeout_ns;
            unsigned int *const errw = p.err;
            const uint32_t full0 = smem_u32(&full_bar[0]), empty0 = smem_u32(&empty_bar[0]);
            const uint32_t accf0 = smem_u32(&acc_full[0]), acce0 = smem_u32(&acc_empty[0]);
            const uint64_t desc0 = smem_desc_sw128(ring_u32);
            const uint32_t stage16 = stage_bytes >> 4;
            int st = 0, b = 0;
            uint32_t ph = 0, uph = 0;  // phase parities: the stage's, and accumulator set b's uses
            bool ok = true;
            SegIter it;
            seg_begin(p, it);
            Seg sg;
            while (ok && seg_next<MT>(p, it, sg)) {
                if (!dev::mbar_wait(acce0 + 8u * (uint32_t)b, uph ^ 1u, abort_v, tmo, errw)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(b * MT) * bn_alloc;
                for (int kb = sg.kb0; kb < sg.kb1; kb++) {
                    if (!dev::mbar_wait(full0 + 8u * (uint32_t)st, ph, abort_v, tmo, errw)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = desc0 + (uint64_t)((uint32_t)st * stage16);
                    const uint64_t bd = ad + (uint64_t)(MT * kTileABytes >> 4);
#pragma unroll
                    for (int kk = 0; kk < kBK / kUmmaK; kk++)
#pragma unroll
                        for (int m = 0; m < MT; m++)
                            mma_f16(d + (uint32_t)m * bn_alloc, ad + (uint64_t)(m * (kTileABytes >> 4) + kk * (kUmmaK * 2 >> 4)),
                                    bd + (uint64_t)(kk * (kUmmaK * 2 >> 4)), idesc, (kb > sg.kb0 || kk > 0) ? 1u : 0u);
                    mma_commit(empty0 + 8u * (uint32_t)st);  // the stage is free once these MMAs have read it
                    if (++st == stages) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(accf0 + 8u * (uint32_t)b);  // the accumulators are complete
                if (++b == nbuf) {
                    b = 0;
                    uph ^= 1u;
                }
            }
            mma_commit(smem_u32(&done_bar));  // always: completes when every issued MMA has finished
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- epilogue
        const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. +31 (warp % 4 rule)
        const int half = (warp - 2) >> 2;             // this warp's 32-column chunks: 32 * (2j + half)
        const int rloc = quarter * 32 + lane;         // row inside a 128-row tile
        const int ew = warp - 2;                      // epilogue warp: its flag in a CTA's row of flags
        int i = 0;
        SegIter it;
        seg_begin(p, it);
        Seg sg;
        for (; seg_next<MT>(p, it, sg); i++) {
            const Unit &x = sg.x;
            const int b = i % p.nbuf;
            const uint32_t use = (uint32_t)(i / p.nbuf);
            if (!dev::mbar_wait_warp(smem_u32(&acc_full[b]), use & 1u, abort_v, p.timeout_ns, p.err)) break;
            tc_fence_after();
            // this warp's 32-column chunks of a row tile: columns 32 * (2j + half), j < nch
            const int nch = (p.bn / 32 - half + 1) / 2 + ((p.bn % 32) && (p.bn / 32) % 2 == half ? 1 : 0);
            if (sg.role == kOwner) {
                // The tile's last k-blocks: wait, warp by warp, for the same warp's part of
                // every lower CTA's piece (bounded; a give-up leaves Y unwritten and raised),
                // then add the pieces in k order to the accumulators and store Y.
                bool have = true;
                for (int i = 0; i < sg.ncon && have; i++)
                    have = flag_wait(p.flags + (size_t)(sg.cfirst + i * p.nt) * kEpiWarps + ew, p.token, abort_v,
                                     p.timeout_ns, p.err);
                have = __all_sync(0xffffffffu, have);
                if (have) {
                    owner_epilogue<MT>(p, sg, tmem_base + (uint32_t)(b * MT * p.bn_alloc), ring_u32, smem_raw, ew, half,
                                       quarter, lane, nch);
                    // the lower pieces are read: their flags go back to zero for the next launch
                    __syncwarp();
                    if (lane == 0)
                        for (int i = 0; i < sg.ncon; i++) p.flags[(size_t)(sg.cfirst + i * p.nt) * kEpiWarps + ew] = 0ull;
                }
            } else {
                for (int m = 0; m < MT; m++) {
                    const uint32_t taddr =
                        tmem_base + (uint32_t)((b * MT + m) * p.bn_alloc) + ((uint32_t)(quarter * 32) << 16);
                    const int row = x.m0 + m * kBM + rloc;
                    const int rows = pick(p.rows, x.mat);
                    float *const Y = pick(p.Y, x.mat);
                    const int tile = x.tile0 + m * p.nt;
                    float *ws_unit =
                        sg.role == kSplit ? p.ws + ((size_t)tile * p.splits + x.s) * (size_t)p.bn * kBM : nullptr;
                    // one chunk's 32 values of this row: to the split's partial tile, to this
                    // CTA's partial slot, or to Y
                    auto store = [&](const uint32_t(&v)[32], int c) {
                        if (sg.role == kSplit) {
#pragma unroll
                            for (int q = 0; q < 32; q++)
                                if (c + q < p.bn) ws_unit[(size_t)(c + q) * kBM + rloc] = __uint_as_float(v[q]);
                        } else if (sg.role == kPiece) {
                            float *blk = p.skws + (size_t)blockIdx.x * p.slot_floats + slot_block(m, ew, (c / 32 - half) / 2);
#pragma unroll
                            for (int q = 0; q < 32; q++) blk[q * 32 + lane] = __uint_as_float(v[q]);
                        } else if (row < rows) {
#pragma unroll
                            for (int q = 0; q < 32; q++) {
                                const int col = x.n0 + c + q;
                                if (c + q < p.bn && col < p.ncols) Y[(size_t)col * rows + row] = __uint_as_float(v[q]);
                            }
                        }
                    };
                    // two chunks in flight: the next chunk's TMEM load overlaps this chunk's stores
                    uint32_t va[32], vb[32];
                    if (nch > 0) {
                        tmem_ld32(taddr + (uint32_t)(32 * half), va);
                        tmem_wait_ld(va);
                    }
                    for (int j = 0; j < nch; j += 2) {
                        const int ca = 32 * (2 * j + half), cb = ca + 64;
                        if (j + 1 < nch) tmem_ld32(taddr + (uint32_t)cb, vb);
                        store(va, ca);
                        if (j + 1 < nch) {
                            tmem_wait_ld(vb);
                            if (j + 2 < nch) tmem_ld32(taddr + (uint32_t)(cb + 64), va);
                            store(vb, cb);
                            if (j + 2 < nch) tmem_wait_ld(va);
                        }
                    }
                }
                if (sg.role == kPiece) {
                    // this warp's part of the slot is written: publish it for the owner
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) st_release_u64(p.flags + (size_t)blockIdx.x * kEpiWarps + ew, p.token);
                }
            }
            // hand the accumulators back to the MMA warp
            tc_fence_before();
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(smem_u32(&acc_empty[b]));
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
        // no MMA may still be writing TMEM, and on a give-up no copy may still be
        // landing in shared memory, when the CTA releases them
        dev::mbar_drain(smem_u32(&done_bar), 0, p.timeout_ns);
        if (*abort_v) {
            const int issued = issued_slot;
            for (int s = 0; s < p.stages && s < issued; s++) {
                const int last = issued - 1 - ((issued - 1 - s) % p.stages);  // last stage issued into slot s
                dev::mbar_drain(smem_u32(&full_bar[s]), (uint32_t)(last / p.stages) & 1u, p.timeout_ns);
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(tmem_cols)
                     : "memory");
    }
}

// Split-k reduction: Y[m][col * rows[m] + row] = sum of the S partials in order 0..S-1,
// where the partial of split s for (matrix m, row, col) lies at
// ws[((tile * S + s) * bn + col % bn) * 128 + row % 128],
// tile = (tbeg[m] + row / 128) * nt + col / bn.  The elements of all matrices form one
// index space (matrix m's four-row groups start at ebeg[m]).  Each thread takes four
// consecutive rows of one column (rows % 4 == 0 on this path) and issues the 16-byte
// loads of every split before the first add (a loop bounded only at run time left one
// round trip per split: 8 us for eight splits); vec4 says every Y is 16-byte aligned,
// else the four results are stored one by one.
constexpr int kReduceThreads = 256;

struct ReduceJob {
    float *Y[kMaxMats];
    int rows[kMaxMats];
    int tbeg[kMaxMats];
    int64_t ebeg[kMaxMats + 1];
    int nmat, ncols, bn, nt, S, vec4;
};

__global__ void __launch_bounds__(kReduceThreads) k_splitk_reduce(const float *__restrict__ ws,
                                                                  const __grid_constant__ ReduceJob j)
{
    dev::pdl_wait();  // the partials are the previous kernel's output
    const int64_t total = j.ebeg[j.nmat];
    for (int64_t e = (int64_t)blockIdx.x * kReduceThreads + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * kReduceThreads) {
        int m = 0;
#pragma unroll
        for (int q = 1; q < kMaxMats; q++)
            if (q < j.nmat && e >= j.ebeg[q]) m = q;
        const int rows = pick(j.rows, m), rows4 = rows >> 2;
        const int64_t le = e - pick(j.ebeg, m);
        const int col = (int)(le / rows4), row = (int)(le - (int64_t)col * rows4) * 4;
        const int tile = (pick(j.tbeg, m) + (row >> 7)) * j.nt + col / j.bn;
        const float4 *src = reinterpret_cast<const float4 *>(
            ws + (((size_t)tile * j.S) * j.bn + col % j.bn) * kBM + (row & (kBM - 1)));
        const size_t split_stride = (size_t)j.bn * kBM / 4;  // in float4
        float4 v[kMaxSplits];
#pragma unroll
        for (int sp = 0; sp < kMaxSplits; sp++)  // every split's load in flight before the first add
            if (sp < j.S) v[sp] = __ldcg(src + sp * split_stride);
        float4 acc = v[0];
#pragma unroll
        for (int sp = 1; sp < kMaxSplits; sp++) {
            if (sp < j.S) {
                acc.x += v[sp].x;
                acc.y += v[sp].y;
                acc.z += v[sp].z;
                acc.w += v[sp].w;
            }
        }
        float *dst = pick(j.Y, m) + (size_t)col * rows + row;
        if (j.vec4) {
            *reinterpret_cast<float4 *>(dst) = acc;
        } else {
            dst[0] = acc.x;
            dst[1] = acc.y;
            dst[2] = acc.z;
            dst[3] = acc.w;
        }
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

int pow2_at_least(int v)
{
    int p = 32;
    while (p < v) p <<= 1;
    return p;
}

// Measured time of one k-block with 256-column tiles: 0.45 us for a 128-row unit,
// 0.80 us for a 256-row unit (twice the work, two thirds of the operand bytes per
// unit of work).
constexpr double kKblockUs[3] = {0.0, 0.45, 0.80};
// The split-k reduction: a dependent launch, then one pass over the partials and Y.
constexpr double kReduceFixedUs = 2.0;
constexpr double kReduceBytesPerUs = 6.0e6;

// Tiles of 64 columns or fewer: a k-block's time depends on how many SMs stream at
// once.  One SM takes at least kNarrowKblockUs per k-block; all the busy SMs together
// draw their weight tiles from HBM at about kNarrowHbmBytesPerUs.  Measured on GB300
// at 8 to 64 columns over 32 to 224 row tiles and 1 to 8 splits: 0.32-0.35 us with
// up to 112 SMs streaming, 0.40 us with 128, 0.47 us with all 152.  (A partial wave
// of 112 row tiles unsplit then beats four splits of three waves and the reduction.)
constexpr double kNarrowKblockUs = 0.33;
constexpr double kNarrowHbmBytesPerUs = 5.3e6;

// Predicted time of a plan in microseconds: waves x (k-blocks per unit x the time of
// a k-block), plus, with S > 1, the reduction kernel.
double plan_us(int64_t units_per_split, int64_t tiles128, int num_kb, int bn, int mt, int s, int ctas, int64_t rows,
               int64_t ncols)
{
    double us;
    if (bn <= 64) {
        const int64_t units = units_per_split * s, full = units / ctas, rest = units % ctas;
        auto kblock_us = [&](int64_t busy) {
            return std::max(kNarrowKblockUs, (double)busy * mt * kTileABytes / kNarrowHbmBytesPerUs);
        };
        us = std::ceil((double)num_kb / s) * ((double)full * kblock_us(ctas) + (rest ? kblock_us(rest) : 0.0));
    } else {
        const double waves = std::ceil((double)units_per_split * s / ctas);
        us = waves * std::ceil((double)num_kb / s) * kKblockUs[mt];
    }
    if (s > 1)
        us += kReduceFixedUs + ((double)tiles128 * s * bn * kBM * 4.0 + (double)rows * ncols * 4.0) / kReduceBytesPerUs;
    return us;
}

// Balanced k ranges, calibrated on GB300 with an L2 flush before each product: with
// every SM busy a k-block takes longer than in the whole-tile plans (0.55 / 0.85 us
// for 128- / 256-row units); a CTA writes its piece while every other CTA writes
// theirs (about 5.5 MB/us in all), and with one TMEM set its next MMAs wait for
// that; an owner reads each lower piece at about 0.15 MB/us.  Where the time
// model is free to choose (bm_set_stream_k(-1)) the balanced plan must be predicted
// 10 % faster than the best other plan: measured gains were small (at most 3 % on the
// Llama-3-8B shapes at 512 columns, 10 % on gate at 64), losses on others up to 8 %,
// and the model is coarse.  The exception is a product of three or more full waves
// of whole 256-column tiles (the output product at 512 columns): there every SM streams
// in both plans, so a k-block costs the same, the balanced plan only removes the idle
// part of the last wave, and it measured 2-4 % faster in chains of launches; a 2 %
// margin.  (At 16 and 64 columns the same rule measured no gain.)
constexpr double kSkKblockUs[3] = {0.0, 0.55, 0.85};
constexpr double kSkFixedUs = 1.0;
constexpr double kSkStoreBytesPerUs = 5.5e6;  // all CTAs' partial-tile stores at once
constexpr double kSkOverlap = 0.3;            // share of that hidden behind MMAs with two TMEM sets
constexpr double kSkReadBytesPerUs = 1.5e5;   // one SM's piece loads
constexpr double kSkMargin = 0.90;
constexpr double kSkMarginManyWaves = 0.98;

// Predicted time of balanced ranges over `units` row units of MT * 128 rows of each of
// nt column tiles, `ctas` CTAs per column tile; nbuf TMEM accumulator sets.
double plan_sk_us(int64_t units, int num_kb, int bn, int mt, int ctas, int64_t nt, int nbuf, bool many_waves)
{
    const int64_t iters = units * num_kb;
    const int64_t per = (iters + ctas - 1) / ctas;
    double us = (double)per * (many_waves ? kKblockUs[mt] : kSkKblockUs[mt]);
    const bool aligned = iters % ctas == 0 && per % num_kb == 0;  // every range whole tiles
    if (!aligned) {
        const double slot = (double)mt * kBM * bn * 4.0;
        const double lower = std::ceil((double)num_kb / (double)per);  // pieces an owner adds, at most
        const double write = (double)ctas * nt * slot / kSkStoreBytesPerUs;
        us += kSkFixedUs + (nbuf == 1 ? write : kSkOverlap * write) + lower * slot / kSkReadBytesPerUs;
    }
    return us;
}

constexpr int kMaxDevices = 64;
std::once_flag g_attr_once[kMaxDevices][2];
std::once_flag g_pool_once[kMaxDevices];
cudaMemPool_t g_pool[kMaxDevices];

// This library's own stream-ordered memory pool for split-k workspaces (one per
// device), keeping freed blocks for reuse instead of returning them at every
// synchronisation.
cudaMemPool_t workspace_pool(int dev_id)
{
    std::call_once(g_pool_once[dev_id], [dev_id] {
        cudaMemPoolProps props{};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev_id;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) == cudaSuccess) {
            uint64_t keep = UINT64_MAX;
            cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
            g_pool[dev_id] = pool;
        }
    });
    return g_pool[dev_id];
}

// Balanced ranges' workspace: the CTAs' partial slots, then their flags.
size_t sk_flags_offset(int grid, int64_t slot_floats)
{
    return ((size_t)grid * (size_t)slot_floats * sizeof(float) + 255) / 256 * 256;
}

// A 64-bit value for the flags of one launch: never zero, and unique within the
// process (a counter through the splitmix64 finaliser, seeded per process), so no
// value left in reused workspace memory by another launch can stand for it.
unsigned long long next_token()
{
    static std::atomic<unsigned long long> seq{0};
    static const unsigned long long seed =
        (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count() ^
        (unsigned long long)reinterpret_cast<uintptr_t>(&seq);
    unsigned long long z = seed + 0x9E3779B97F4A7C15ull * (seq.fetch_add(1) + 1);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    return z | 1ull;
}

struct Plan {
    GemmParams p;
    int mt_per_unit;  // MT: 128-row tiles per work unit (1 or 2)
    int grid;
    size_t smem;
    size_t ws_bytes;
};

template <int MT>
void set_smem_attr(const DeviceInfo &dev)
{
    int dev_id = 0;
    cudaGetDevice(&dev_id);
    std::call_once(g_attr_once[dev_id & (kMaxDevices - 1)][MT - 1], [&] {
        cudaFuncSetAttribute(k_gemm_tc<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.max_smem_optin - 1024);
    });
}

// CTAs of k_gemm_tc<mt> with `smem` bytes of dynamic shared memory that one SM can
// hold at once, by the occupancy calculator (0 when the query fails).
int resident_ctas_per_sm(int mt, size_t smem, const DeviceInfo &dev)
{
    int n = 0;
    cudaError_t e;
    if (mt == 2) {
        set_smem_attr<2>(dev);
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemm_tc<2>, kThreads, smem);
    } else {
        set_smem_attr<1>(dev);
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemm_tc<1>, kThreads, smem);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();  // a failed query leaves no sticky error behind
        return 0;
    }
    return n;
}

// Plans one launch over nmat matrices of rows[m] x k sharing ncols activation columns.
// sk_mode: balanced k ranges never (0), always (1) or where predicted faster (-1);
// max_splits: the most k-splits a plan may take (1: none).
int plan_gemm(Plan *pl, int nmat, const int64_t *rows, int64_t k, int64_t ncols, const DeviceInfo &dev,
              int max_splits, bool allow_mt2, int sk_mode)
{
    if (nmat < 1 || nmat > kMaxMats) return fail(BM_ERR_INVALID_ARG, "tensor-core product: 1..4 matrices");
    GemmParams &p = pl->p;
    p = GemmParams{};
    int64_t mts[kMaxMats], total_mt = 0, total_rows = 0;
    for (int m = 0; m < nmat; m++) {
        if (rows[m] < 1 || rows[m] > 0x7fffffffLL)
            return fail(BM_ERR_INVALID_ARG, "tensor-core product: rows must lie in 1 .. 2^31-1");
        p.rows[m] = (int)rows[m];
        mts[m] = (rows[m] + kBM - 1) / kBM;
        total_mt += mts[m];
        total_rows += rows[m];
    }
    if (ncols > 0x7fffffffLL || k > 0x7fffffffLL)
        return fail(BM_ERR_INVALID_ARG, "tensor-core product: k and ncols must be below 2^31");
    p.nmat = nmat;
    p.ncols = (int)ncols;
    p.k = (int)k;
    p.num_kb = (int)((k + kBK - 1) / kBK);
    const int64_t n16 = (ncols + 15) / 16 * 16;
    if ((total_mt + nmat) * ((ncols + 15) / 16) * kMaxSplits > 0x7fffffffLL)
        return fail(BM_ERR_INVALID_ARG, "tensor-core product: too many tiles");
    // Tile width, row tiles per unit (MT) and k-splits with the least predicted time.
    // 256-column tiles move the fewest operand bytes per unit of work; 128-column tiles
    // (a k-block takes about as long) double the units of a product with few row tiles,
    // which can beat splitting k and reducing.  256-row units (two MMAs sharing the X
    // tile) are taken only with full 256-column tiles, where they were measured.
    int mt_unit = 1, splits = 1, bn = (int)(n16 < 256 ? n16 : 256), sk = 0;
    double best_us = 1e300;
    const int widths[2] = {(int)(n16 < 256 ? n16 : 256), n16 > 128 ? 128 : 0};
    for (int wi = 0; wi < 2; wi++) {
        const int bw = widths[wi];
        if (bw == 0) continue;
        const int64_t nt = (ncols + bw - 1) / bw;
        const int64_t tiles128 = total_mt * nt;
        for (int mt = 1; mt <= (allow_mt2 && total_mt >= 2 && bw == 256 ? 2 : 1); mt++) {
            int64_t units_rows = 0;
            for (int m = 0; m < nmat; m++) units_rows += (mts[m] + mt - 1) / mt;
            const int64_t tiles = units_rows * nt;
            auto consider = [&](double us, int sp, int with_sk) {
                if (us < best_us - 1e-9) {
                    best_us = us;
                    mt_unit = mt;
                    splits = sp;
                    bn = bw;
                    sk = with_sk;
                }
            };
            if (sk_mode != 1)
                for (int sp = 1; sp <= std::max(1, std::min(std::min(kMaxSplits, max_splits), p.num_kb)); sp++)
                    consider(plan_us(tiles, tiles128, p.num_kb, bw, mt, sp, dev.sm_count, total_rows, ncols), sp, 0);
            // balanced ranges need the operand ring to hold the owners' read buffers
            const int stage_b = mt * kTileABytes + bw * kBK * 2;
            const int ring_b = std::min(kMaxStages, (dev.max_smem_optin - 2048) / stage_b) * stage_b;
            const int64_t per_col = std::min<int64_t>(dev.sm_count / nt, units_rows * p.num_kb);  // CTAs per column
            // Where the planner is free to choose, tiles of 64 columns or fewer never take
            // balanced ranges: measured 10-30 % slower than whole tiles on the Llama-3-8B
            // shapes at 8-64 columns, and up to twice as slow on products of a few MB
            // (2048 x 1024, 3072 x 576 and 576 x 576 at 8-16 columns: 12-14 us against
            // 6.8-7.5 us for whole tiles with k-splits).
            const bool sk_ok = sk_mode == 1 || (sk_mode == -1 && bw > 64);
            if (sk_ok && ring_b >= kEpiWarps * kOwnerDepth * 4096 && per_col >= 1) {
                const int nbuf = 2 * mt * pow2_at_least(bw) <= 512 ? 2 : 1;
                const bool many_waves = tiles >= 3 * (int64_t)dev.sm_count && bw == 256;  // measured there only
                const double us = plan_sk_us(units_rows, p.num_kb, bw, mt, (int)per_col, nt, nbuf, many_waves);
                consider(sk_mode == 1 ? us : us / (many_waves ? kSkMarginManyWaves : kSkMargin), 1, 1);
            }
        }
    }
    p.bn = bn;
    p.bn_alloc = pow2_at_least(p.bn);
    p.nt = (int)((ncols + p.bn - 1) / p.bn);
    pl->mt_per_unit = mt_unit;
    p.ubeg[0] = 0;
    p.tbeg[0] = 0;
    for (int m = 0; m < nmat; m++) {
        const int units_m = (int)((mts[m] + mt_unit - 1) / mt_unit);
        p.ubeg[m + 1] = p.ubeg[m] + units_m;
        p.tbeg[m + 1] = p.tbeg[m] + units_m * mt_unit;  // a unit's second tile past the matrix end included
    }
    for (int m = nmat; m < kMaxMats; m++) {
        p.ubeg[m + 1] = p.ubeg[nmat];
        p.tbeg[m + 1] = p.tbeg[nmat];
    }
    p.mtu = p.ubeg[nmat];
    p.nbuf = 2 * mt_unit * p.bn_alloc <= 512 ? 2 : 1;  // TMEM holds 512 columns
    const int64_t tiles = (int64_t)p.mtu * p.nt;       // work tiles of 128 * MT rows
    p.splits = splits;
    const int stage_bytes = mt_unit * kTileABytes + p.bn * kBK * 2;
    const int budget = dev.max_smem_optin - 1024 - 1024;  // alignment slack and static shared memory
    p.stages = std::min(kMaxStages, budget / stage_bytes);
    if (p.stages < 2) return fail(BM_ERR_CUDA, "tensor-core product: not enough shared memory");
    const int64_t units = tiles * p.splits;
    pl->grid = (int)std::min<int64_t>(units, dev.sm_count);
    p.sk = sk;
    if (sk) {
        p.iters = (int64_t)p.mtu * p.num_kb;
        if (p.iters > ((int64_t)1 << 40))
            return fail(BM_ERR_INVALID_ARG, "tensor-core product: too many k-blocks");
        pl->grid = (int)(std::min<int64_t>(dev.sm_count / p.nt, p.iters) * p.nt);
        p.slot_floats = (int64_t)mt_unit * kEpiWarps * kWarpChunks * 1024;
    }
    // One CTA per SM (this request is more than half of the SM's shared memory), so the
    // accumulators (up to 512 columns) never exceed the SM's TMEM.
    const size_t smem = (size_t)p.stages * stage_bytes + 1024;
    const size_t one_per_sm = (size_t)dev.max_smem_optin / 2 + 4096;
    pl->smem = std::max(smem, one_per_sm);
    pl->ws_bytes = p.splits > 1 ? (size_t)p.tbeg[nmat] * p.nt * p.splits * p.bn * kBM * sizeof(float) : 0;
    if (sk) {
        // An owner waits for the CTAs below it, so every CTA of the grid must be resident
        // at once: one per SM by design, confirmed by the occupancy calculator (a plan the
        // SMs could not hold whole falls back to the whole-tile plans).
        if (resident_ctas_per_sm(mt_unit, pl->smem, dev) < 1 || pl->grid > dev.sm_count)
            return plan_gemm(pl, nmat, rows, k, ncols, dev, max_splits, allow_mt2, 0);
        pl->ws_bytes = sk_flags_offset(pl->grid, p.slot_floats) + (size_t)pl->grid * kEpiWarps * 8;
    }
    return BM_OK;
}

template <int MT>
int launch_mt(const Plan &pl, const TmaMaps &maps, cudaStream_t s, const DeviceInfo &dev)
{
    set_smem_attr<MT>(dev);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)pl.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_gemm_tc<MT>, maps, pl.p);
    if (e != cudaSuccess) return fail(BM_ERR_CUDA, "tensor-core product: launch failed: %s", cudaGetErrorString(e));
    return BM_OK;
}

// The split-k reduction right behind the product on the same stream, with
// programmatic dependent launch so its launch overlaps the product's tail; it waits
// (griddepcontrol.wait) for the product before it reads the partials.
int launch_reduce(const Plan &pl, cudaStream_t s, const DeviceInfo &dev)
{
    ReduceJob j{};
    j.nmat = pl.p.nmat;
    j.ncols = pl.p.ncols;
    j.bn = pl.p.bn;
    j.nt = pl.p.nt;
    j.S = pl.p.splits;
    j.vec4 = 1;
    j.ebeg[0] = 0;
    for (int m = 0; m < pl.p.nmat; m++) {
        j.Y[m] = pl.p.Y[m];
        j.rows[m] = pl.p.rows[m];
        j.tbeg[m] = pl.p.tbeg[m];
        j.ebeg[m + 1] = j.ebeg[m] + (int64_t)(pl.p.rows[m] / 4) * pl.p.ncols;
        if (reinterpret_cast<uintptr_t>(pl.p.Y[m]) & 15) j.vec4 = 0;
    }
    for (int m = pl.p.nmat; m < kMaxMats; m++) j.ebeg[m + 1] = j.ebeg[pl.p.nmat];
    const int64_t total = j.ebeg[pl.p.nmat];
    int64_t blocks = (total + kReduceThreads - 1) / kReduceThreads;
    blocks = std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)dev.sm_count * 8));
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kReduceThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_splitk_reduce, (const float *)pl.p.ws, j);
    if (e != cudaSuccess)
        return fail(BM_ERR_CUDA, "tensor-core product: reduction launch failed: %s", cudaGetErrorString(e));
    return BM_OK;
}

int launch_plan(const Plan &pl, const uint16_t *const *W, const uint16_t *X, cudaStream_t s, const DeviceInfo &dev)
{
    if (!get_encoder()) return fail(BM_ERR_CUDA, "tensor-core product: cuTensorMapEncodeTiled unavailable");
    TmaMaps maps;
    memset(&maps, 0, sizeof(maps));
    for (int m = 0; m < pl.p.nmat; m++)
        if (!make_map(&maps.w[m], W[m], pl.p.rows[m], pl.p.k, kBM * pl.mt_per_unit))
            return fail(BM_ERR_CUDA, "tensor-core product: tensor map encoding failed");
    if (!make_map(&maps.x, X, pl.p.ncols, pl.p.k, pl.p.bn))
        return fail(BM_ERR_CUDA, "tensor-core product: tensor map encoding failed");
    const int st = pl.mt_per_unit == 2 ? launch_mt<2>(pl, maps, s, dev) : launch_mt<1>(pl, maps, s, dev);
    if (st != BM_OK || pl.p.splits == 1) return st;
    return launch_reduce(pl, s, dev);
}

}  // namespace

int launch_gemm_tc_multi(int nmat, const uint16_t *const *W, const int64_t *rows, int64_t k, const uint16_t *X,
                         int64_t ncols, float *const *Y, cudaStream_t s, const DeviceInfo &dev)
{
    unsigned int *err = device_error_word();
    if (!err) return fail(BM_ERR_CUDA, "tensor-core product: device error word unavailable");
    Plan pl;
    int st = plan_gemm(&pl, nmat, rows, k, ncols, dev, kMaxSplits, true, stream_k_mode());
    if (st != BM_OK) return st;
    for (int m = 0; m < nmat; m++) pl.p.Y[m] = Y[m];
    pl.p.err = err;
    pl.p.timeout_ns = kDefaultTimeoutNs;
    if (pl.ws_bytes == 0) return launch_plan(pl, W, X, s, dev);

    // Workspace for the partial tiles (split-k, or balanced ranges' slots and flags),
    // stream-ordered (so concurrent products on other streams never share it, and
    // graph capture records it as an allocation node).
    int dev_id = 0;
    cudaGetDevice(&dev_id);
    cudaMemPool_t pool = workspace_pool(dev_id & (kMaxDevices - 1));
    if (!pool) return fail(BM_ERR_CUDA, "tensor-core product: workspace pool unavailable");
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, pl.ws_bytes, pool, s);
    if (e != cudaSuccess)
        return fail(BM_ERR_CUDA, "tensor-core product: workspace allocation failed: %s", cudaGetErrorString(e));
    if (pl.p.sk) {
        pl.p.skws = static_cast<float *>(ws);
        pl.p.flags = reinterpret_cast<unsigned long long *>(static_cast<unsigned char *>(ws) +
                                                            sk_flags_offset(pl.grid, pl.p.slot_floats));
        pl.p.token = next_token();
    } else {
        pl.p.ws = static_cast<float *>(ws);
    }
    st = launch_plan(pl, W, X, s, dev);
    cudaError_t e2 = cudaFreeAsync(ws, s);
    if (st == BM_OK && e2 != cudaSuccess)
        return fail(BM_ERR_CUDA, "tensor-core product: workspace release failed: %s", cudaGetErrorString(e2));
    return st;
}

int launch_gemm_tc(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols, float *Y,
                   cudaStream_t s, const DeviceInfo &dev)
{
    return launch_gemm_tc_multi(1, &W, &rows, k, X, ncols, &Y, s, dev);
}

// ----------------------------------------------------------------------------- no-allocation variant
//
// The same tensor-core product for callers that cannot allocate device memory:
// its split-k workspace is this file-scope array instead of a stream-ordered
// allocation.  The array is part of the library's module, so every GPU that
// loads the library holds it until the process exits.

constexpr size_t kNoAllocScratchBytes = BM_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
std::once_flag g_scratch_once[kMaxDevices];
unsigned char *g_scratch_ptr[kMaxDevices];
cudaError_t g_scratch_status[kMaxDevices];
}  // namespace

// The plan of the no-allocation product: whole tiles (no balanced ranges), and, when
// the fastest plan's partial tiles would not fit the scratch, the fastest plan with
// fewer k-splits whose partials do -- at worst no split, which needs no scratch.
int plan_noalloc(Plan *pl, int64_t rows, int64_t k, int64_t ncols, const DeviceInfo &dev)
{
    int max_splits = kMaxSplits;
    while (true) {
        int st = plan_gemm(pl, 1, &rows, k, ncols, dev, max_splits, true, 0);
        if (st != BM_OK) return st;
        if (pl->ws_bytes <= kNoAllocScratchBytes || pl->p.splits <= 1) return BM_OK;
        max_splits = pl->p.splits - 1;
    }
}

int launch_gemm_tc_noalloc(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols, float *Y,
                           cudaStream_t s, const DeviceInfo &dev)
{
    unsigned int *err = device_error_word();
    if (!err) return fail(BM_ERR_CUDA, "no-allocation product: device error word unavailable");
    Plan pl;
    int st = plan_noalloc(&pl, rows, k, ncols, dev);
    if (st != BM_OK) return st;
    const size_t need = pl.ws_bytes;
    if (need > kNoAllocScratchBytes)  // cannot happen: an unsplit plan needs no scratch
        return fail(BM_ERR_INVALID_ARG,
                    "bm_f16_matmul_noalloc: this product needs %zu bytes of split-k scratch; the static scratch "
                    "holds %zu (use bm_f16_matmul)",
                    need, kNoAllocScratchBytes);
    pl.p.Y[0] = Y;
    pl.p.err = err;
    pl.p.timeout_ns = kDefaultTimeoutNs;
    if (pl.p.splits > 1) {
        // In host code g_noalloc_scratch names a host-side stand-in, not device memory:
        // the kernel gets the device address, looked up once per device with that
        // device current.
        int d = -1;
        if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices)
            return fail(BM_ERR_CUDA, "bm_f16_matmul_noalloc: cannot query the current device");
        std::call_once(g_scratch_once[d], [d] {
            void *ptr = nullptr;
            g_scratch_status[d] = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
            g_scratch_ptr[d] = static_cast<unsigned char *>(ptr);
        });
        if (g_scratch_status[d] != cudaSuccess || !g_scratch_ptr[d])
            return fail(BM_ERR_CUDA, "bm_f16_matmul_noalloc: scratch address lookup failed: %s",
                        cudaGetErrorString(g_scratch_status[d]));
        pl.p.ws = reinterpret_cast<float *>(g_scratch_ptr[d]);
    }
    return launch_plan(pl, &W, X, s, dev);
}

int launch_gemm_tc_withheld(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols, float *Y,
                            cudaStream_t s, const DeviceInfo &dev, unsigned long long timeout_ns)
{
    unsigned int *err = device_error_word();
    if (!err) return fail(BM_ERR_CUDA, "tensor-core product: device error word unavailable");
    Plan pl;
    int st = plan_gemm(&pl, 1, &rows, k, ncols, dev, 1, false, 0);
    if (st != BM_OK) return st;
    pl.p.Y[0] = Y;
    pl.p.err = err;
    pl.p.timeout_ns = timeout_ns;
    pl.p.withhold_first_load = 1;
    return launch_plan(pl, &W, X, s, dev);
}

int plan_info_gemm_tc(int64_t rows, int64_t k, int64_t ncols, bool noalloc, const DeviceInfo &dev, int64_t *info)
{
    Plan pl;
    int st = noalloc ? plan_noalloc(&pl, rows, k, ncols, dev)
                     : plan_gemm(&pl, 1, &rows, k, ncols, dev, kMaxSplits, true, stream_k_mode());
    if (st != BM_OK) return st;
    info[0] = pl.mt_per_unit;
    info[1] = pl.p.bn;
    info[2] = pl.p.splits;
    info[3] = pl.p.sk;
    info[4] = (int64_t)pl.ws_bytes;
    info[5] = pl.grid;
    return BM_OK;
}

}  // namespace bm
