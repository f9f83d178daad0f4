/*
 * bm.h -- C ABI of the F16-weight product library for NVIDIA GB300 (sm_103a).
 *
 * The operations are those of the page "docs/modules/f16.md" (bankML, the
 * F16 weights multiplied as ggml b11192 multiplies them):
 *   - the activation is first rounded to f16, round to nearest even
 *     (section "Design notes", bullet "Activation");
 *   - a one-column product is ggml_vec_dot_f16 per row, bit for bit
 *     (section "Design notes", bullet "vec_dot");
 *   - a product of two or more columns takes tinyBLAS's 8-lane chain when the
 *     weight has a multiple of 4 rows and the row a multiple of 8 elements, and
 *     falls back to vec_dot otherwise (sections "Summary", "Technical usage",
 *     "Design notes", bullet "sgemm_dot").  Here that tinyBLAS path runs on
 *     tcgen05 tensor cores accurate to 4e-6 * sum|w_i * a_i| of tinyBLAS's
 *     result, or -- for products of up to bm_set_exact_sgemm_cols columns
 *     (default 2) -- on a CUDA-core kernel that gives tinyBLAS's bits; the
 *     fallback is bit-exact.
 *
 * Conventions shared by every call:
 *   - f16 values are passed as their IEEE binary16 bit patterns (uint16_t),
 *     little-endian.  A weight matrix W is row-major [rows][k] (a row is
 *     contiguous); a column X[c] of a multi-column activation is contiguous, so
 *     X is [ncols][k] row-major.  The product output is Y[c * rows + r], f32
 *     (page f16.md, section "Matrix products", "mat_mul_par").
 *   - Every pointer argument named as device memory must point to memory the
 *     GPU can read (or write) -- e.g. from cudaMalloc or torch.  The caller
 *     owns all of it; the library allocates nothing the caller frees and keeps
 *     no state across calls besides per-device caches of device properties.
 *   - Input pointers must be 16-byte aligned; output pointers 16-byte aligned
 *     for bm_to_f16, 4-byte aligned elsewhere.  Outputs are overwritten, never
 *     accumulated into, and must not overlap any input.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and never synchronise.  A non-zero return means nothing
 *     was launched, except BM_ERR_CUDA, which reports a launch error.  Device
 *     side give-ups of bounded waits are reported by bm_device_status().
 *   - Empty products (n, rows or ncols equal to 0) are valid and launch nothing.
 *   - All calls are thread-safe; bm_last_error() is per host thread.
 */
#ifndef BM_H
#define BM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *bm_stream_t;

typedef enum {
    BM_OK = 0,
    BM_ERR_INVALID_ARG = 1,        /* null pointer, bad size, overlapping output */
    BM_ERR_ALIGNMENT = 2,          /* a pointer breaks the alignment rule above */
    BM_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not compute capability 10.3 */
    BM_ERR_CUDA = 4,               /* a CUDA runtime or driver call failed */
    BM_ERR_TIMEOUT = 5             /* a kernel gave up a bounded wait (bm_device_status) */
} bm_status;

/* Largest row length k accepted by the products (the f16 activation of one
 * column is staged whole in shared memory by the one-column kernels). */
#define BM_MAX_K 65536

/*
 * h[i] = f16(x[i]) rounded to nearest, ties to even, for 0 <= i < n
 * (f16.md, "Design notes", "Activation"; ggml_cpu_fp32_to_fp16).
 *   x : device, f32[n], 16-byte aligned.     h : device, uint16[n], 16-byte aligned.
 *   n >= 0.  |x| >= 65520 gives +-inf, f16 subnormals are produced, f32
 *   subnormals give +-0.  NaN inputs give a NaN (payload unspecified).
 */
int bm_to_f16(const float *x, uint16_t *h, int64_t n, bm_stream_t stream);

/*
 * y[r] = vec_dot(W[r], x) for 0 <= r < rows, bit-exact with ggml_vec_dot_f16
 * (f16.md, "Matrix products", mat_vec_par; "Design notes", "vec_dot"):
 * 32 f32 chains (element i of a 32-element step feeds accumulator (i%32)/8,
 * lane i%8, in increasing i from +0), reduced (a0+a2)+(a1+a3), low half plus
 * high half, two horizontal adds, then the k%32 tail added in double in order.
 *   W : device, f16[rows][k].   x : device, f16[k].   y : device, f32[rows].
 *   rows >= 0, 1 <= k <= BM_MAX_K.
 */
int bm_f16_matvec(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *x, float *y,
                  bm_stream_t stream);

/*
 * bm_f16_matvec for up to four matrices that share one activation x, in one
 * launch (f16.md, "Matrix products", mat_vec_multi_par: Q, K and V; gate and up).
 * Every output row is still one vec_dot, so y[m] equals bm_f16_matvec(W[m], ...)
 * bit for bit.
 *   nmat in 1..4.  W, rows and y are HOST arrays of nmat entries; W[m] and y[m]
 *   are device pointers (f16[rows[m]][k] and f32[rows[m]]); rows[m] >= 0.
 */
int bm_f16_matvec_multi(int nmat, const uint16_t *const *W, const int64_t *rows, int64_t k,
                        const uint16_t *x, float *const *y, bm_stream_t stream);

/*
 * The activation rounding and the fused one-column products in one launch:
 * h = bm_to_f16(x), then y[m] = vec_dot(W[m][r], h) for up to four matrices
 * (f16.md, "Design notes", "Activation" and "vec_dot"; forward.md, Advantages,
 * "Shared activations": one rounded activation feeds Q, K and V, or gate and
 * up).  Every bit equals bm_to_f16 followed by bm_f16_matvec_multi.
 *   x : device, f32[k], 16-byte aligned.  h : device, uint16[k], 16-byte aligned,
 *   or NULL to skip storing the rounded activation (it is needed, and must be
 *   given, when k % 8 != 0).  W, rows, y as for bm_f16_matvec_multi (nmat 1..4).
 */
int bm_f16_matvec_act(int nmat, const uint16_t *const *W, const int64_t *rows, int64_t k,
                      const float *x, uint16_t *h, float *const *y, bm_stream_t stream);

/*
 * A decode step's one-column products, recorded once and run as one launch (no
 * counterpart on the pages, which run each product as its own pool pass: a
 * schedule of this library for f16.md's one-column products).  Each call is
 * bm_f16_matvec_act's -- the f32 activation x rounded to f16, then multiplied
 * by up to four matrices sharing it, every output row ggml_vec_dot_f16 bit for
 * bit -- and bm_step_run gives exactly the bits that making the calls in order
 * with bm_f16_matvec_act gives.  A call may read what an earlier call of the
 * step wrote: its activation is read only once every earlier call's outputs
 * are written (the kernel waits, on the device, between calls).  What one
 * launch buys: the weights of the next calls stream while a call finishes or
 * waits, and no launch gaps.
 *   calls[i].nmat 1..4; W[m] device f16[rows[m]][k], 16-byte aligned, rows[m] in
 *   0 .. 2^31-1 (0: skipped); 8 <= k <= BM_MAX_K and k % 8 == 0 (rows are streamed
 *   as 16-byte-aligned boxes; other k: bm_f16_matvec_act); x device f32[k],
 *   16-byte aligned; y[m] device f32[rows[m]], 4-byte aligned.  Within a call no
 *   output overlaps an input or another output; across calls outputs may be
 *   later calls' activations (or be overwritten by later calls), never weights.
 *   1 <= ncalls <= 65535.
 * bm_step_create validates every call, encodes the weights' tensor maps and
 * copies the call table to the current device (the step's only allocation, freed
 * by bm_step_destroy), and synchronises the device once.  The pointers are kept:
 * the same memory is read and written by every run, with whatever it holds then.
 * bm_step_run launches the step on `stream` (asynchronous; one cooperative launch
 * of two CTAs per SM, which must all be resident: BM_ERR_CUDA if the device
 * cannot hold them).  Runs of one step must not overlap on the GPU (they share
 * the step's device counter); runs of different steps may.  After a run whose
 * bm_device_status is BM_ERR_TIMEOUT the step must be destroyed and recorded
 * again.  bm_step_destroy frees the step (NULL is allowed); the step's device
 * must still exist.
 */
typedef struct bm_matvec_call {
    int nmat;
    const uint16_t *W[4];
    int64_t rows[4];
    int64_t k;
    const float *x;
    float *y[4];
} bm_matvec_call;
typedef struct bm_step bm_step;
int bm_step_create(const bm_matvec_call *calls, int ncalls, bm_step **step);
int bm_step_run(const bm_step *step, bm_stream_t stream);
int bm_step_destroy(bm_step *step);

/*
 * rms_norm then mul of f32 rows by an f32 norm weight (page forward.md,
 * "Technical usage", "Other public pieces": the sum of squares in double, no
 * FMA; "Design notes", step three: the first RMS norm with its weight gives
 * attn_norm-0), optionally rounded to f16 (f16.md, "Activation") for the
 * products that follow -- each row of a prefill micro-batch before bm_f16_matmul.
 *     q_i = x_i * x_i (f32);  mean = mean of the q_i rounded once to f32;
 *     scale = 1 / sqrtf(mean + eps) (f32 add, IEEE square root and divide);
 *     out_i = (x_i * scale) * g_i (two f32 multiplies);  h_i = f16(out_i).
 * The page takes the mean from a double sum of the squares, which lies within
 * (k - 1) * 2^-53 (relative) of the exact sum.  Here the squares are summed
 * exactly in 128-bit fixed point (squares more than 2^63 below the largest left
 * out: together under k * 2^-63 of the sum) and the mean is divided out to 2^-62
 * by integer steps, so it does not depend on any order and is the same in every
 * call and in bm_f16_matvec_norm.  The f32 mean, and with it every output bit,
 * equals the double-sum route's unless the exact mean lies within about
 * (k + 4) * 2^-53 (relative) of an f32 rounding boundary.  A zero row with eps
 * == 0 gives NaN, as the formula does; a NaN or infinite square makes the mean
 * NaN or +inf.
 *   x : device, f32[nrows][k].  g : device, f32[k].  out : device, f32[nrows][k],
 *   or NULL; out == x (in place) is allowed, any other overlap is not.
 *   h : device, uint16[nrows][k] (f16 bits), or NULL; at least one of out, h.
 *   nrows >= 0, 1 <= k <= BM_MAX_K.  x, g, out 4-byte aligned, h 2-byte aligned
 *   (16-byte aligned pointers and k % 4 == 0 take the vector loads).
 */
int bm_rms_norm_mul(const float *x, const float *g, int64_t nrows, int64_t k, float eps,
                    float *out, uint16_t *h, bm_stream_t stream);

/*
 * The decode front end in one launch: n = rms_norm then mul of x by g (as
 * bm_rms_norm_mul, same bits), h = f16(n), then y[m] = vec_dot(W[m][r], h) for
 * up to four matrices (forward.md, "Design notes", steps three and four: the
 * first RMS norm with its weight, then the Q, K and V projections of the normed
 * row; the same for gate and up after the second norm).  Every bit equals
 * bm_rms_norm_mul followed by bm_f16_matvec_multi.
 *   x, g : device, f32[k], 16-byte aligned.  eps : the norm's epsilon.
 *   n_out : device, f32[k], 16-byte aligned, or NULL (the normed row is then not
 *   stored).  h : device, uint16[k], 16-byte aligned, or NULL (needed, and must
 *   be given, when k % 8 != 0).  W, rows, y as for bm_f16_matvec_multi.
 */
int bm_f16_matvec_norm(int nmat, const uint16_t *const *W, const int64_t *rows, int64_t k,
                       const float *x, const float *g, float eps, float *n_out, uint16_t *h,
                       float *const *y, bm_stream_t stream);

/*
 * Y[c*rows + r] = W[r] . X[c] for every row r and column c
 * (f16.md, "Matrix products", mat_mul_par), with the path ggml takes:
 *   - bm_takes_sgemm(rows, k, ncols): tcgen05 tensor cores, f32 accumulation,
 *     |Y - sgemm_dot(W[r], X[c])| <= 4e-6 * sum_i |W[r][i] * X[c][i]|; except
 *     that a product of at most bm_set_exact_sgemm_cols columns gives tinyBLAS's
 *     sgemm_dot per element, bit for bit (eight f32 lane chains, lane l taking
 *     elements 8t + l in increasing t, folded ((l0+l4)+(l2+l6))+((l1+l5)+(l3+l7));
 *     "Design notes", "sgemm_dot");
 *   - otherwise: vec_dot per element, bit-exact (ncols == 1 is bm_f16_matvec).
 *   W : device, f16[rows][k].   X : device, f16[ncols][k].   Y : device, f32[ncols*rows].
 *   rows, ncols >= 0, 1 <= k <= BM_MAX_K.
 */
int bm_f16_matmul(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols,
                  float *Y, bm_stream_t stream);

/*
 * bm_f16_matmul for up to four matrices that share one activation X -- the
 * prefill counterpart of bm_f16_matvec_multi (Q, K and V of a micro-batch; gate
 * and up): Y[m][c*rows[m] + r] = W[m][r] . X[c].  Each matrix keeps its own
 * path by its own shape, exactly as bm_f16_matmul (forward.md, "Batched
 * prefill": each element keeps the bits of its per-pair dot): the matrices
 * that take the tensor cores share one launch (more work units, one set-up and
 * one tail), each within the same 4e-6 * sum|w*a| bound of tinyBLAS -- the
 * f32 sums may be ordered differently from a separate bm_f16_matmul of the same
 * matrix; the others (vec_dot, or tinyBLAS's bits on the CUDA-core kernel) run
 * as their own products with the same bits as bm_f16_matmul.
 *   nmat in 1..4.  W, rows and Y are HOST arrays of nmat entries; W[m] is a
 *   device f16[rows[m]][k], Y[m] a device f32[ncols][rows[m]]; rows[m] >= 0.
 *   X : device, f16[ncols][k].  1 <= k <= BM_MAX_K, ncols >= 0.
 */
int bm_f16_matmul_multi(int nmat, const uint16_t *const *W, const int64_t *rows, int64_t k,
                        const uint16_t *X, int64_t ncols, float *const *Y, bm_stream_t stream);

/* Size of the static device scratch that bm_f16_matmul_noalloc uses (8 MiB). */
#define BM_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * bm_f16_matmul for callers that cannot allocate device memory (no counterpart
 * on the pages: a property of this library).  Some callers may not call
 * cudaMalloc or any allocator at all: a serving engine that reserved the whole
 * device for its own arena at start-up, a plugin living inside a host whose
 * allocator owns every byte, or a latency-critical thread where an allocation
 * could block or synchronise.  bm_f16_matmul needs a temporary device workspace
 * when it splits a product along k; this entry point uses instead a scratch
 * array that is part of the library's device code, BM_NOALLOC_SCRATCH_BYTES
 * large, held by every GPU that loads the library until the process exits.
 * It allocates nothing: no cudaMalloc, no stream-ordered allocation, no
 * allocating library routine.  The caller still passes W, X and Y, with the
 * same layout, validation, path selection and results as bm_f16_matmul with
 * balanced k ranges off (bm_set_stream_k(0)); where bm_f16_matmul takes them the
 * two results may differ in their last bits, both within the tensor-core bound.
 *   - When the fastest plan's split-k partial tiles would not fit the scratch,
 *     the product takes the fastest plan with fewer k-splits whose partials do
 *     (at worst no split, which needs no scratch), so no valid product is
 *     refused for its size; it may then run slower than bm_f16_matmul.  Should
 *     a plan ever exceed the scratch all the same, the call fails with
 *     BM_ERR_INVALID_ARG and a reason (bm_last_error) and launches nothing.
 *   - The first call on a device looks up the scratch's device address (once per
 *     device, with that device current); make that first call before any stream
 *     capture.
 *   - Every call shares the one scratch array, which keeps the last call's
 *     contents.  Nothing in it needs to start at zero: every split writes its
 *     whole partial tile before the reduction reads it, so stale contents are
 *     never read.  Calls whose kernels overlap on the GPU (e.g. on two streams at
 *     once) race on the scratch and must be ordered by the caller.
 */
int bm_f16_matmul_noalloc(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X,
                          int64_t ncols, float *Y, bm_stream_t stream);

/*
 * Logits over a tied token embedding (page "docs/modules/forward.md", Summary:
 * with no output.weight the logits read token_embd.weight): the product of
 * E (f16[vocab][hidden]) with ncols normalised activations X (f16[ncols][hidden]),
 * Y[c*vocab + v].  It is one product over all columns, so its path follows
 * bm_takes_sgemm(vocab, hidden, ncols) exactly as bm_f16_matmul's does.
 *
 * Which rows to pass is the caller's rule (forward.md, "Why only the output rows
 * leave the last layer"): on the last layer only the rows the engine outputs (its
 * inp_out_ids: none, the last one, or all) go through the feed-forward products and
 * the logits.  Pass exactly those rows, gathered into X, and nothing else: the
 * column count picks the path, so the last row alone (one column, vec_dot) and the
 * same row inside a product over all rows (tinyBLAS) give different bits, each
 * matching the engine that makes the same choice.
 */
int bm_f16_logits(const uint16_t *E, int64_t vocab, int64_t hidden, const uint16_t *X,
                  int64_t ncols, float *Y, bm_stream_t stream);

/*
 * Rows of an f16 table widened to f32, exactly: the token-embedding lookup
 * (f16.md, "Technical usage", dequantize_row -- F16 bytes widened to f32, as
 * get_rows does; widen is exact).  out[i*hidden + j] = (float) E[ids[i]*hidden + j].
 *   E : device, f16[vocab][hidden].   ids : device, int32[n].
 *   out : device, f32[n][hidden] (16-byte aligned output takes the fast path).
 *   vocab, hidden >= 1 unless n == 0; n >= 0.  An id outside [0, vocab) leaves its
 *   output row untouched and makes bm_device_status return BM_ERR_INVALID_ARG.
 */
int bm_f16_get_rows(const uint16_t *E, int64_t vocab, int64_t hidden, const int32_t *ids, int64_t n,
                    float *out, bm_stream_t stream);

/*
 * The f16 accumulator helpers of the attention side (f16.md, "Technical usage":
 * `mad` is ggml_vec_mad_f16, flash attention's V accumulator; `scale` is
 * ggml_vec_scale_f16), in place on acc[0..n):
 *   bm_f16_mad:   acc[i] = RNE_f16(fma(widen(v[i]), w, widen(acc[i])))
 *   bm_f16_scale: acc[i] = RNE_f16(widen(acc[i]) * s)
 * mad's product and sum round once in f32 (a fused multiply-add, as ggml's F16C + FMA
 * path computes it -- the page names the function, not its rounding), then to f16
 * nearest-even; scale is one f32 multiply, then f16.  acc, v: device f16[n], 2-byte
 * aligned (16-byte aligned vectors take an 8-wide path); v may be acc itself but may
 * not otherwise overlap it.  n >= 0 (0: nothing launched).  NaN results are NaN (their
 * payload is unspecified).
 */
int bm_f16_mad(uint16_t *acc, const uint16_t *v, float w, int64_t n, bm_stream_t stream);
int bm_f16_scale(uint16_t *acc, float s, int64_t n, bm_stream_t stream);

/* ggml's path selector (f16.md, "Technical usage"): 1 when
 * ncols >= 2 && rows % 4 == 0 && k % 8 == 0, else 0.  Pure; never fails. */
int bm_takes_sgemm(int64_t rows, int64_t k, int64_t ncols);

/*
 * Programmatic dependent launch for the products (default off; process-wide).
 * When on, a product of one column with k % 8 == 0, a bm_takes_sgemm product on
 * the bit-exact kernel (bm_set_exact_sgemm_cols) or on the tensor cores, and the
 * norm and embedding kernels are launched so that they may start before the
 * kernel ahead of them on the stream has finished: a product sets up and begins
 * copying its weight matrix (and bm_f16_matvec_norm its norm weight) into the
 * chip at once, and waits for that kernel only before it reads its activation
 * and writes its output.  Precondition while on: the kernel immediately ahead of
 * a product on its stream must not write that product's weight matrix or norm
 * weight (they are constants in a forward pass).  Results are identical either
 * way.  Returns the previous setting.
 */
int bm_set_pdl(int enable);

/*
 * Bit-exact tinyBLAS products (process-wide; no counterpart on the pages: a choice
 * between two implementations of the same contract).  A bm_takes_sgemm product of
 * at most `ncols` columns runs on a CUDA-core kernel that keeps tinyBLAS's chain
 * order and returns its bits; wider ones run on the tensor cores within the bound.
 * `ncols` is clamped to 0..8 (0 or 1: always the tensor cores).  The default, 2,
 * gives tinyBLAS's bits to two-column products, where on GB300 the exact kernel is
 * also the faster one (it streams the weights like the one-column product: Llama-3-8B
 * gate 20.9 us against 26.1 on the tensor cores, Q 9.9 against 12.8).  Larger values
 * buy tinyBLAS's bits at some speed on the long products (gate at 3 columns 29.3 us
 * against 26.1), at none on short ones (Q at 3 columns 12.6 against 12.9).  Returns the
 * previous setting.
 */
int bm_set_exact_sgemm_cols(int ncols);

/*
 * Balanced k ranges for the tensor-core products (process-wide; no counterpart on
 * the pages: a work split of this library, stream-K after Osama et al., PPoPP 2023).
 * The k-blocks of all tiles of a product are cut into equal ranges, one per SM;
 * a tile shared by several SMs is finished by the SM holding its last k-block,
 * which adds the other pieces in k order.  mode -1 (default): used where the
 * library's time model predicts it clearly faster than whole tiles or k-splits,
 * never for products of 64 columns or fewer (measured slower there); 0: never; 1: wherever it applies (at least one SM per column tile of the
 * product).  Any other value counts as its sign.  The result stays within the
 * tensor-core bound in every mode and is repeatable (the same bits for the same
 * product, mode and GPU).  The workspace (one partial tile per SM and a flag word
 * per epilogue warp) comes from the library's stream-ordered pool like the k-split
 * one; bm_f16_matmul_noalloc never uses this mode.  An owner waits for the SMs
 * below it, so the mode is taken only where the occupancy calculator confirms that
 * one CTA of the product fits on every SM the grid uses; otherwise the product
 * falls back to whole tiles.  Returns the previous setting.
 */
int bm_set_stream_k(int mode);

/*
 * The plan a tensor-core product takes (introspection, no counterpart on the
 * pages): for a bm_takes_sgemm product of rows x k x ncols on the current device,
 * under the current bm_set_stream_k mode, or bm_f16_matmul_noalloc's plan when
 * noalloc != 0.  Writes info[0..5] (host array of 6): 128-row tiles per work
 * unit (1 or 2), tile columns, k-splits, balanced k ranges (0 or 1), scratch
 * bytes (split-k partial tiles, or the balanced ranges' slots and flags) and
 * CTAs.  It launches and allocates nothing.  The plan is the same whatever
 * bm_set_exact_sgemm_cols says; whether the product reaches the tensor cores at
 * all follows bm_f16_matmul's path selection.  BM_ERR_INVALID_ARG for sizes the
 * tensor-core product does not take (rows % 4, k % 8, ncols < 2, k > BM_MAX_K).
 */
int bm_tc_plan(int64_t rows, int64_t k, int64_t ncols, int noalloc, int64_t *info);

/* Waits for `stream`, then reads and clears this library's device error word
 * on the current device: BM_OK, BM_ERR_TIMEOUT (a kernel gave up a bounded
 * wait and wrote nothing trustworthy), BM_ERR_INVALID_ARG (bm_f16_get_rows met
 * an id out of range), BM_ERR_UNSUPPORTED_DEVICE (the bit-exact few-column kernel
 * found its shared memory not 1024-byte aligned and wrote nothing; not seen on
 * GB300), or BM_ERR_CUDA (the wait failed). */
int bm_device_status(bm_stream_t stream);

/* Self-test of the bounded device waits (no counterpart on the pages; it
 * checks this library's failure reporting).  Runs one 128 x 64 x 16
 * tensor-core product whose data producer deliberately never fills its only
 * pipeline stage, so the consumer's bounded wait gives up after about 20 ms;
 * the kernel then records the give-up, frees its tensor memory and exits with
 * the context intact.  Synchronises `stream`.  Returns BM_ERR_TIMEOUT when the
 * give-up was detected and reported (the expected result), any other status
 * otherwise.  W: device f16[128][64], X: device f16[16][64], Y: device
 * f32[16*128] (contents of Y are unspecified afterwards). */
int bm_selftest_wait_timeout(const uint16_t *W, const uint16_t *X, float *Y, bm_stream_t stream);

/* Static text for a status code. */
const char *bm_status_string(int status);

/* The reason for the last non-zero status returned on this host thread
 * ("" if none).  Valid until the next call on this thread. */
const char *bm_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* BM_H */
