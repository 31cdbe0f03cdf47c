/*
 * tn_gemm.h -- C ABI of the GB300 (sm_103a) dense TN GEMM library
 *              (libdense_gemm_tn.so).
 *
 * The operation, for every 0 <= m < M and 0 <= n < N:
 *
 *     C[m,n] = sum_{k=0}^{K-1} A[m,k] * B[k,n]
 *
 * is the plain matrix product of hello-gpu ch.11 "GEMM-Like", section 11.1
 * (no alpha, no beta: C is overwritten), in the "TN" storage of the AMD ROCm
 * blog "FP16 GEMM optimization on AMD RDNA 3 and RDNA 4", section "What we
 * compute":
 *
 *   A  row-major M x K:     element (m,k) at A[m*lda + k],  lda >= max(1,K)
 *   B  column-major K x N:  element (k,n) at B[k + n*ldb],  ldb >= max(1,K)
 *   C  column-major M x N:  element (m,n) at C[m + n*ldc],  ldc >= max(1,M)
 *
 * so A and B are both contiguous along K.  (A PyTorch caller holds B as an
 * (N, K) row-major tensor and C as an (N, M) row-major tensor.)  Products
 * are accumulated in FP32 on the tensor cores and rounded once to the output
 * type with round-to-nearest-even.  M, N and K need not be multiples of any
 * tile size (the same section requires non-divisible shapes to work).
 *
 * Conventions shared by every entry point below:
 *   - Pointers A, B, C are DEVICE pointers (or managed memory) on the
 *     current CUDA device.  The caller owns all of them; the library keeps
 *     no reference after the call returns.
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *     default stream.  Calls are asynchronous: they return after enqueueing
 *     work; errors found inside a kernel (a bounded wait that ran out) are
 *     reported later by gemm_poll_device_status().
 *   - M == 0 or N == 0: nothing is launched, GEMM_OK.  K == 0: C is filled
 *     with +0.
 *   - C must not overlap A or B (undefined result).
 *   - Operands whose row stride (ld * element size) or base address is not
 *     a multiple of 16 bytes are first copied into a library-owned, lazily
 *     grown device workspace with a padded stride, one per (device,
 *     stream), so calls on different streams may take this path at once.
 *   - When the tiles of a launch end in a partly filled wave, each leftover
 *     tile is computed as two halves of its k range whose FP32 partial sums
 *     meet in a library-owned buffer kept per (device, stream), allocated on
 *     first need (about 0.5 MiB per leftover tile).  The sum is taken in a
 *     fixed way, so results do not depend on timing.  cudaStreamPerThread
 *     counts as one stream per host thread.  Problems with at most 64
 *     columns n and a short K run a kernel of their own whose k ranges meet
 *     in the same buffer (at most 128 KiB per 128 rows m), also in a fixed
 *     order.
 *   - CUDA graphs: once a call has run on a stream (the first call may
 *     allocate that stream's buffers and set kernel attributes), later calls
 *     with the same sizes on that stream enqueue kernel launches only and can
 *     be captured and replayed; the kernels leave their buffers ready for the
 *     next launch.
 *   - Thread safety: every entry point may be called from several host
 *     threads, also on one stream (the legacy default stream included); the
 *     per-device state is guarded internally.  A call may enqueue several
 *     kernels (a row copy, the GEMM, a reduce pass) that share the stream's
 *     buffers; the calls on one stream hold a lock of that stream from their
 *     first buffer lookup through their last launch, so two threads' calls
 *     never interleave their kernels on it.  gemm_release_workspace() waits
 *     for calls in progress on other threads.  On a thread's first call for
 *     a device, the library makes that device's primary context current on
 *     the thread (cudaSetDevice), so a thread that has made no CUDA call of
 *     its own can call it.
 */
#ifndef DENSE_GEMM_TN_H
#define DENSE_GEMM_TN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,   /* negative size, ld too small, NULL or misaligned pointer */
    GEMM_ERR_UNSUPPORTED = 2,   /* device is not sm_103, or a size beyond 2^31 - 256 */
    GEMM_ERR_CUDA = 3,          /* a CUDA runtime / driver call failed (see gemm_last_error) */
    GEMM_ERR_TIMEOUT = 4        /* a kernel's bounded wait ran out (reported by poll) */
} gemm_status_t;

/*
 * FP16 TN GEMM.  A, B: IEEE binary16 (__half); C: binary16.
 * Errors: GEMM_ERR_INVALID_ARG for M, N or K < 0, lda/ldb < max(1,K),
 * ldc < max(1,M), a NULL pointer with work to do, or a pointer not 2-byte
 * aligned; GEMM_ERR_UNSUPPORTED off sm_103; GEMM_ERR_CUDA on a failed launch.
 */
gemm_status_t gemm_f16_tn(int64_t M, int64_t N, int64_t K,
                          const void *A, int64_t lda,
                          const void *B, int64_t ldb,
                          void *C, int64_t ldc,
                          void *stream);

/*
 * FP8 TN GEMM.  A, B: OCP E4M3 ("e4m3fn") codes, one byte each; C: bfloat16.
 * scale_a and scale_b are per-tensor DEQUANTISATION factors: the FP32
 * accumulator is multiplied by (scale_a * scale_b) in FP32 and rounded once
 * to bfloat16, i.e. C[m,n] = bf16(acc[m,n] * scale_a * scale_b).  (The FP8
 * variant with per-tensor scales and bf16 output has no printed counterpart
 * on the pages; the blog above announces the FP8 port as its part 2.)
 * Errors as for gemm_f16_tn (pointers need 1-byte alignment, C 2-byte).
 */
gemm_status_t gemm_f8e4m3_tn(int64_t M, int64_t N, int64_t K,
                             const void *A, int64_t lda,
                             const void *B, int64_t ldb,
                             void *C, int64_t ldc,
                             float scale_a, float scale_b,
                             void *stream);

/*
 * FP8 TN GEMM with device-resident per-tensor scales: gemm_f8e4m3_tn with
 * scale_a and scale_b passed as DEVICE pointers to one fp32 value each.  The
 * kernel reads them when it runs, so an earlier kernel on the same stream
 * (gemm_quantize_e4m3) may produce them without a round trip to the host.
 * C[m,n] = bf16(acc[m,n] * ((*scale_a) * (*scale_b))), the product of the two
 * scales taken in FP32 -- the same arithmetic as gemm_f8e4m3_tn, so both
 * entry points give bit-identical C for the same scale values.  The caller
 * owns the scale buffers.  Errors as for gemm_f8e4m3_tn, plus
 * GEMM_ERR_INVALID_ARG for a NULL or not 4-byte aligned scale pointer.
 */
gemm_status_t gemm_f8e4m3_tn_dscale(int64_t M, int64_t N, int64_t K,
                                    const void *A, int64_t lda,
                                    const void *B, int64_t ldb,
                                    void *C, int64_t ldc,
                                    const float *scale_a, const float *scale_b,
                                    void *stream);

/*
 * Attention scores with the softmax's row statistics, fused into the GEMM's
 * epilogue: the QK^T step of hello-gpu ch.11's closing note (the next chapter
 * joins the GEMM and the softmax so that less of the intermediate goes back to
 * memory) and of the TileLang attention article (its QK^T block, M = N = 1024,
 * K = 128, with the softmax fused into the same kernel).  A holds Q (M x K,
 * row-major), B holds K (its column n = key n, i.e. an N x K row-major array).
 * With acc = the FP32 sum over k:
 *
 *     C[m,n]     = fp16(fp32(acc[m,n] * scale))           column-major, ldc, as gemm_f16_tn
 *     row_max[m] = max over n of fp32(acc[m,n] * scale)
 *     row_sum[m] = sum over n of exp(fp32(acc[m,n] * scale) - row_max[m])
 *
 * i.e. the softmax of row m of the scores is exp(s - row_max[m]) / row_sum[m]
 * (the pages do not fix the statistics; these are the two reductions that
 * normalise a softmax, from the FP32 scores before their rounding).  The sum
 * is formed in FP32 (each exp as 2^(x log2 e) with the hardware ex2, relative
 * error about 2^-22) in a fixed order, so results repeat exactly.
 * row_max and row_sum: DEVICE arrays of M floats owned by the caller.
 * scale: any finite float (typically 1/sqrt(K)).  M or N == 0: nothing is
 * written.  K == 0: C = scale * 0, row_max = 0, row_sum = N.
 * Uses a library-owned buffer per (device, stream) for the partial
 * statistics, allocated on first use.  Tiles are never split along K here.
 * Errors as for gemm_f16_tn, plus GEMM_ERR_INVALID_ARG for NULL or misaligned
 * row_max / row_sum or a non-finite scale.
 */
gemm_status_t gemm_f16_tn_softmax_stats(int64_t M, int64_t N, int64_t K,
                                        const void *A, int64_t lda,
                                        const void *B, int64_t ldb,
                                        void *C, int64_t ldc, float scale,
                                        float *row_max, float *row_sum,
                                        void *stream);

/* Element types gemm_quantize_e4m3 reads. */
typedef enum {
    GEMM_IN_F32 = 0,    /* IEEE binary32 */
    GEMM_IN_F16 = 1,    /* IEEE binary16 */
    GEMM_IN_BF16 = 2    /* bfloat16 */
} gemm_quant_in_t;

/*
 * Per-tensor E4M3 quantisation of one operand, the amax taken on the device:
 *
 *     amax  = max |x[r,c]|                       over the whole tensor
 *     s_q   = 448 / amax                         fp32 (0 if amax = 0; FLT_MAX if it overflows)
 *     q[r,c] = E4M3(fp32(x[r,c] * s_q))          round to nearest even, saturating to +-448
 *     *scale = amax / 448                        fp32: the dequantisation factor
 *
 * so that gemm_f8e4m3_tn_dscale(..., scale_a, scale_b) on two quantised
 * operands approximates the GEMM of the originals.  (The pages print no FP8
 * rule; the ROCm blog above only announces an FP8 port.  This is the plain
 * per-tensor scaling to the E4M3 maximum, 448.)
 *
 * x: rows x cols, row-major, element (r,c) at x[r*ldx + c], x_type one of
 *    gemm_quant_in_t, aligned to its element size; ldx >= max(1, cols).
 *    For the GEMM's operands: A is M x K with ldx = lda, B (column-major
 *    K x N) is N x K with ldx = ldb.
 * q: rows x cols OCP E4M3 ("e4m3fn") codes, q[r*ldq + c], ldq >= max(1, cols).
 * scale: one fp32 in device memory.
 * All three are DEVICE pointers owned by the caller; q and scale must not
 * overlap x.  rows or cols == 0 writes *scale = 0 and nothing else.
 * Inputs must be finite (an Inf or NaN gives unspecified codes and scale).
 *
 * Two kernel launches per call on `stream`: the first finds each CTA's
 * maximum and leaves it in a small library-owned array kept per (device,
 * stream) and allocated on first use; the second reads them and quantises.
 * No CTA waits on another.  Calls on one stream may share the array; calls on
 * different streams use different arrays.
 * Errors: GEMM_ERR_INVALID_ARG for an unknown x_type, negative sizes, an ld
 * below its minimum, NULL pointers with work to do, a misaligned x or scale;
 * GEMM_ERR_UNSUPPORTED off sm_103 or above 2^40 elements; GEMM_ERR_CUDA on a
 * failed allocation or launch.
 */
gemm_status_t gemm_quantize_e4m3(const void *x, int x_type, int64_t rows, int64_t cols, int64_t ldx,
                                 void *q, int64_t ldq, float *scale, void *stream);

/*
 * gemm_f16_tn without any device allocation by the library.
 *
 * The paper has no counterpart to this entry point; it exists for callers
 * that cannot let a library call cudaMalloc: programs that hand out all
 * device memory from their own pool or fixed budget, and latency-critical
 * paths where the implicit device synchronisation of cudaMalloc / cudaFree
 * is not acceptable.  Arguments, layouts and results are those of
 * gemm_f16_tn; the caller still passes (and owns) A, B and C.
 *
 * Where gemm_f16_tn would copy an operand into its lazily grown workspace
 * (base, row stride or K not a multiple of 16 bytes), this call copies it
 * into a fixed 32 MiB array that is part of the library's device image
 * instead (every GPU that loads the library holds it until the process
 * exits).  If the padded copies need more than 32 MiB
 * (2 * roundup(K, 8) * (rows of each operand that needs the copy), each
 * operand rounded up to 256 bytes), the call returns GEMM_ERR_INVALID_ARG
 * and launches nothing.  Aligned operands need no copy and no scratch.
 *
 * The array is shared by every call on a device and keeps the last call's
 * contents (each call overwrites all of the part it reads).  Calls that
 * overlap on the GPU -- on different streams, without ordering -- race on it.
 * Calls on one stream do not, whatever host threads make them: each call
 * enqueues its copy and its GEMM with no other call's launches between.
 * The call never takes the paths that need the library's per-stream buffers
 * (split-K partial sums in memory); small grids with a long K add up their
 * k ranges inside a cluster of CTAs instead, which needs no buffer.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.
 */
gemm_status_t gemm_f16_tn_noalloc(int64_t M, int64_t N, int64_t K,
                                  const void *A, int64_t lda,
                                  const void *B, int64_t ldb,
                                  void *C, int64_t ldc,
                                  void *stream);

/* Human-readable name of a status code (static storage). */
const char *gemm_status_string(gemm_status_t status);

/* Detail of the last error returned on the calling host thread (static,
 * thread-local storage; "" when none). */
const char *gemm_last_error(void);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word.  Returns GEMM_ERR_TIMEOUT if a kernel gave up on a bounded wait since
 * the last poll (its C is then incomplete), GEMM_ERR_CUDA if the stream
 * reported an error, GEMM_OK otherwise.
 */
gemm_status_t gemm_poll_device_status(void *stream);

/* Frees the current device's workspaces, all kept per stream: the row
 * copies of unaligned operands, the split-K partial sums, the quantiser's
 * arrays and the softmax-statistics buffers, and the smaller buffers that
 * growth replaced.  It first waits for calls in progress on other host
 * threads to have enqueued their kernels, then synchronises the device
 * (cudaFree).  The next call that needs a buffer allocates it again. */
void gemm_release_workspace(void);

/*
 * Output-tile order of the persistent scheduler, exported so the host can
 * check it.  Tile `id` of a tiles_m x tiles_n grid maps to (*tile_m, *tile_n)
 * by the grouped raster of hello-gpu ch.11 section 11.3.4 (GROUP_M) and of the
 * ROCm blog's "Step 6" (blocks grouped into tall regions of `group` tile rows,
 * the last group short): consecutive ids walk down `group` rows of one tile
 * column before moving to the next column.  Returns 0, or -1 if an argument
 * is out of range (a grid of more than 2^31 - 1 tiles included).
 */
int gemm_tile_coord(int64_t tiles_m, int64_t tiles_n, int64_t group, int64_t id,
                    int64_t *tile_m, int64_t *tile_n);

/*
 * Limit, in nanoseconds, of every device-side wait of kernels launched after
 * this call on any device (default 2e9).  0 restores the default.  A wait that
 * exceeds it makes the kernel record GEMM_ERR_TIMEOUT, drain its in-flight
 * copies, free its tensor memory and return.
 */
void gemm_set_wait_limit_ns(uint64_t limit_ns);

/*
 * Test hook: while `mode` is non-zero, launched GEMM kernels make one thread
 * wait first on a barrier nothing arrives on, so its bounded wait runs out and
 * the kernel leaves through its timeout path (no fault, no hang):
 *   1  the MMA-issuing thread;
 *   2  the TMA producer of the even CTA of each pair (or of each CTA);
 *   3  the TMA producer of the odd CTA of each pair.
 * 0 turns the hook off.
 */
void gemm_debug_inject_stall(int mode);

/*
 * Test hook: 0 (default) lets the library choose the tile shape per call;
 * 1 forces one CTA per 128 x 256 tile, 2 a CTA pair per 256 x 256 tile in
 * 2-CTA clusters.  Returns 0, or -1 for other values.
 */
int gemm_debug_force_cta_group(int group);

/*
 * Test hook: whether CTA pairs compute 256 x 512 tiles (two N = 256 halves
 * sharing the n-side rows, a 512-column accumulator) instead of 256 x 256.
 * 0 (default): an estimate of the launch's length in tile times decides;
 * 1: always, wherever CTA pairs run without the softmax statistics; -1:
 * never.  Returns 0, or -1 for
 * other values.
 */
int gemm_debug_force_wide_tiles(int mode);

/*
 * Test hook: the height, in tile rows, of the scheduler's raster groups
 * (see gemm_tile_coord); 0 restores the default (8).  Even values only, so
 * that raster ids 2j and 2j + 1 stay neighbouring m tiles of one n tile.
 * Returns 0, or -1 for odd values or values outside 0 .. 64.
 */
int gemm_debug_set_raster_group(int rows);

/*
 * Test hook: the order in which whole tiles walk their k blocks.  0
 * (default): the library's choice; 1: every tile from the first k block to
 * the last; 2: tiles of odd waves (tile id / co-resident slots odd) from the
 * last to the first, so that a wave starts on the k slices that the wave
 * before it, which shares its A panels, read last.  Only the order of the
 * FP32 partial sums changes (results on integer inputs are identical).
 * Returns 0, or -1 for other values.
 */
int gemm_debug_set_k_order(int mode);

/*
 * Test hook: how a grid of at most half the co-resident slots with a long K
 * (at least 32 k blocks) is cut into k ranges.  0 (default): the library's
 * choice; 1: always the split-reduce (FP32 partials in a per-stream buffer,
 * summed by a second kernel); 2: wherever the tiles are single-CTA tiles,
 * a cluster of 2 to 4 CTAs per tile that add their partials through
 * distributed shared memory (no buffer, no second kernel).  Returns 0, or
 * -1 for other values.
 */
int gemm_debug_set_long_k_mode(int mode);

/*
 * Test hook: the configuration of launches whose units are all m-part units
 * of single CTAs (grids of at most half the co-resident slots' tiles with a
 * short K, each tile cut into four 64-row or two 128-row ranges of m).  The
 * lean configuration has a ring sized for such a unit (three stages of 24 KiB
 * for quarters, two of 32 KiB for halves), 128 or 256 TMEM columns, and runs
 * two CTAs per SM; the full one has four stages of 48 KiB, 512 columns and
 * one CTA per SM.  0 (default): the library's choice (lean for launches of
 * more units than half the co-resident slots with at most 8 k blocks, 4 for
 * halves); 1: always the full one; 2: lean wherever the units are quarters
 * or halves.  The arithmetic, and so every result, is the same.  Returns 0,
 * or -1 for other values.
 */
int gemm_debug_set_lean_mode(int mode);

/*
 * Test hook: problems with N <= 64 (no softmax statistics) may run a kernel
 * with the operands on the other sides of the MMA (128 rows m of A by the N
 * columns n), whose k ranges meet in a small per-stream workspace.  0
 * (default): the library's choice (where K holds at most 64 blocks of 128
 * bytes); 1: never; 2: always where N <= 64.
 * Returns 0, or -1 for other values.
 */
int gemm_debug_set_skinny_mode(int mode);

/*
 * Measurement hook: while `counters` (a DEVICE pointer to 3 zeroed unsigned
 * 64-bit words) is set, every launch of the general GEMM kernel (not the
 * kernel for at most 64 columns) afterwards adds, from the first thread of
 * its first CTA, the SM cycles (%clock64) and nanoseconds
 * (%globaltimer) from its start to its end to counters[0] and counters[1],
 * and 1 to counters[2] (three atomic adds per launch, nothing else).
 * counters[0] / counters[1] is then the average SM clock, in GHz, that those
 * launches ran at.  NULL turns it off (the default).  The caller owns the
 * buffer and keeps it alive while launches that use it may run.
 */
void gemm_debug_set_clock_probe(unsigned long long *counters);

/* Description of the last GEMM kernel launch on the calling host thread
 * (tile shape, grid, co-resident cluster slots), for logs and tests
 * (thread-local storage; "" before the first launch). */
const char *gemm_debug_last_launch(void);

/* Tile configuration and build string, e.g. for logs (static storage). */
const char *gemm_build_info(void);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_GEMM_TN_H */
