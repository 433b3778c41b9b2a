/*
 * mxgemm.h -- C interface of the GB300 (sm_103a) MX block-scaled FP8 GEMM.
 *
 *   C[M,N] (+)= (A * 2^(sA-127)) x (B * 2^(sB-127))
 *
 * The operation is the scaled tensor-core product documented as
 * `tlx.async_dot_scaled(A, B, acc, A_scale, "e4m3", B_scale, "e4m3", use_acc)`
 * ("TLX API Quick Reference", section "Matrix Multiply (MMA)": D = (A*scale_A)
 * @ (B*scale_B) + D with FP8 inputs; "Tensor core operations", sections
 * "2-CTA Scaled MMA" and "TMEM-backed MX Scales").  Element format E4M3 and
 * scale format E8M0 (one scale per 32 consecutive K elements) follow the OCP
 * Microscaling Formats specification v1.0.  Accumulation is FP32.
 *
 * Layouts (every pointer is caller-owned DEVICE memory on the handle's GPU,
 * dense row-major, no leading-dimension parameters; mxgemm_run_host takes
 * host memory instead):
 *   A       : M x K      uint8 element codes (E4M3 by default, see
 *                        MXGEMM_OPT_A_FORMAT), K contiguous
 *   A_scale : M x (K/32) uint8 E8M0 codes
 *   B       : K x N      uint8 element codes (MXGEMM_OPT_B_FORMAT), N contiguous
 *                        (or N x K, K contiguous: MXGEMM_OPT_B_MAJOR)
 *   B_scale : N x (K/32) uint8 E8M0 codes (row j holds column j's scales)
 *   C       : M x N      float (MXGEMM_OUT_F32) or bfloat16 (MXGEMM_OUT_BF16)
 *
 * Semantics of use_acc: 0 -> C = A.B (C's previous contents, even NaN, are
 * ignored); 1 -> C = C + A.B, C read in out_dtype, the sum formed in FP32 and
 * rounded once to out_dtype (round to nearest even).
 *
 * Error behaviour: every entry point returns an mxgemm_status_t and never
 * throws.  Arguments are validated before anything is enqueued; on an error
 * nothing is launched and C is untouched.  Launches are asynchronous on the
 * given stream: a device-side wait that exceeds its time limit does not trap,
 * it records MXGEMM_ERR_TIMEOUT in the handle's device status word, which
 * mxgemm_get_device_status reads.
 *
 * Threads and streams: a handle may be used from one host thread at a time,
 * and its internal workspace is reused in stream order, so concurrent calls
 * on different streams need different handles.
 *
 * Entry points: mxgemm_run (device operands), mxgemm_run_host (host
 * operands, copies pipelined with the GEMM), mxgemm_run_noalloc (no device
 * allocation, fixed scratch; with mxgemm_noalloc_get_status and
 * mxgemm_noalloc_set_option), mxgemm_quantize and mxgemm_quantize_sr
 * (FP32/BF16 -> E4M3 codes and E8M0 scales on the GPU, rounding to nearest
 * or stochastically), plus handle, option, status and timing helpers.
 */
#ifndef MXGEMM_H_
#define MXGEMM_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mxgemm_ctx *mxgemm_handle_t;

/* cudaStream_t without pulling in the CUDA headers. */
typedef void *mxgemm_stream_t;

typedef enum {
  MXGEMM_OUT_F32 = 0,
  MXGEMM_OUT_BF16 = 1
} mxgemm_out_dtype_t;

typedef enum {
  MXGEMM_OK = 0,
  MXGEMM_ERR_INVALID_VALUE = 1,      /* bad size, pointer, dtype or handle */
  MXGEMM_ERR_MISALIGNED = 2,         /* A, B or C not 16-byte aligned */
  MXGEMM_ERR_UNSUPPORTED_DEVICE = 3, /* device is not compute capability 10.3 */
  MXGEMM_ERR_OUT_OF_MEMORY = 4,      /* workspace allocation failed */
  MXGEMM_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed */
  MXGEMM_ERR_TIMEOUT = 6,            /* a device-side wait ran out (status word) */
  MXGEMM_ERR_TOO_LARGE = 7           /* mxgemm_run_noalloc: scratch need above its fixed size */
} mxgemm_status_t;

/* Options for mxgemm_set_option. */
typedef enum {
  /* Tile mode: 0 = automatic (the transposed kernel of mode 3 when M <= 128
   * and both element formats are 8-bit, else a CTA pair when M > 128, else
   * one CTA), 1 = one CTA per 128x256 tile, 2 = CTA pair (cta_group::2) per
   * 256x256 tile, 3 = the transposed kernel for few rows: C^T = B^T x A^T
   * with 128 columns of B on the tensor cores' 128-row side and the M rows
   * of A as the MMA's N (M rounded up to 16), K split over a cluster of up
   * to 8 CTAs whose partials are added in shared memory in a fixed order;
   * needs M <= 128 and E4M3 / E5M2 operands (else a run returns
   * MXGEMM_ERR_INVALID_VALUE); the options SCHEDULER and STREAM_K do not
   * apply to it.  Default 0. */
  MXGEMM_OPT_MODE = 1,
  /* Device-side wait limit in nanoseconds (default 2e9).  A wait that runs
   * out sets MXGEMM_ERR_TIMEOUT and the kernel drains and returns. */
  MXGEMM_OPT_WAIT_TIMEOUT_NS = 2,
  /* Test hook for the failure-detection path: when 1, the load-issuing warp
   * of the next launches issues no loads, so the consumer waits run out and
   * the kernel reports MXGEMM_ERR_TIMEOUT.  Default 0. */
  MXGEMM_OPT_TEST_STALL_PRODUCER = 3,
  /* Tile scheduler: 0 = static striding over a persistent grid of one CTA
   * (pair) per SM; 1 = cluster launch control ("TLX API Quick Reference",
   * section "CLC (Cluster Launch Control)"): the grid has one cluster per
   * work item, and running clusters cancel clusters that have not launched
   * yet and take their items (no stream-K tail under this scheduler).
   * Default 0. */
  MXGEMM_OPT_SCHEDULER = 4,
  /* Balancing of the tiles left over after the last full wave.  1
   * (default): with long K (64+ steps of 128) their K steps are split
   * evenly over all CTAs (stream-K), one CTA per tile adding the others'
   * FP32 partials (kept in the handle's workspace) before it stores C;
   * otherwise, when they fill at most half a wave, each is computed as two
   * 128-column halves.  0: every tile is computed whole. */
  MXGEMM_OPT_STREAM_K = 5,
  /* Element format of A (MXGEMM_OPT_A_FORMAT) and of B
   * (MXGEMM_OPT_B_FORMAT), an mxgemm_format_t; default MXGEMM_FMT_E4M3.
   * The formats are those of the MX family that the tensor cores' scaled
   * MMA takes ("TLX API Quick Reference", section "Matrix Multiply (MMA)":
   * the A_format / B_format strings of async_dot_scaled).  A and B may
   * differ. */
  MXGEMM_OPT_A_FORMAT = 6,
  MXGEMM_OPT_B_FORMAT = 7,
  /* Layout of A_scale and B_scale, an mxgemm_scale_layout_t; default
   * MXGEMM_SCALES_ROW_MAJOR.  With MXGEMM_SCALES_PACKED the run takes the
   * scales in the order the tensor cores read them (as mxgemm_quantize_ex
   * writes them) and runs no scale repack before the kernel. */
  MXGEMM_OPT_SCALE_LAYOUT = 8,
  /* Layout of the 6- and 4-bit element codes in A and B, an
   * mxgemm_element_layout_t; default MXGEMM_ELEMS_BYTE.  No effect on 8-bit
   * formats. */
  MXGEMM_OPT_ELEMENT_LAYOUT = 10,
  /* Layout of B, an mxgemm_b_major_t; default MXGEMM_B_K_BY_N. */
  MXGEMM_OPT_B_MAJOR = 11
} mxgemm_option_t;

/* Layouts of B (B_scale is N x (K/32) either way).
 *   MXGEMM_B_K_BY_N : B is K x N, N contiguous (row pitch N bytes), as the
 *     product C = A.B is written.
 *   MXGEMM_B_N_BY_K : B is stored transposed, N x K with K contiguous (row
 *     pitch K bytes; row j holds column j of B) -- the layout of a linear
 *     layer's weight [out features][in features].  Its rows need no
 *     re-pitch for any N, and 6- and 4-bit groups of 16 run along K. */
typedef enum { MXGEMM_B_K_BY_N = 0, MXGEMM_B_N_BY_K = 1 } mxgemm_b_major_t;

/* Element layouts of 6- and 4-bit operands (both take one byte per element
 * of address space: A is M x K bytes, B is K x N bytes).
 *   MXGEMM_ELEMS_BYTE   : one element per byte, the code in the low bits
 *     (the upper bits are ignored).  Each run repacks A and B into the form
 *     below before the GEMM (a pass over each operand).
 *   MXGEMM_ELEMS_PACKED : the form the tensor cores read: each 16-byte group
 *     of a row (16 consecutive K elements of a row of A, 16 consecutive N
 *     elements of a row of B) holds its 16 elements as one little-endian
 *     128-bit number, element i at bits [b*i, b*i + b) for b = 6 or 4, that
 *     is in the group's first 12 or 8 bytes (the other bytes are ignored).
 *     Read as it is, with no pass before the GEMM; a 6- or 4-bit B then needs
 *     N % 16 == 0 (MXGEMM_ERR_INVALID_VALUE). */
typedef enum { MXGEMM_ELEMS_BYTE = 0, MXGEMM_ELEMS_PACKED = 1 } mxgemm_element_layout_t;

/* Scale layouts.
 *   MXGEMM_SCALES_ROW_MAJOR : A_scale M x (K/32), B_scale N x (K/32), dense.
 *   MXGEMM_SCALES_PACKED    : 512-byte chunks, one per 128 rows of A (or 128
 *     columns of B) and 128-deep K step (4 scales per row).  Byte
 *     (r % 32) * 16 + (r / 32) * 4 + j of a chunk holds the scale of its row
 *     (column) r, r < 128, for K block 4 ks + j.  With S = ceil(K / 128):
 *       A_scale: chunk (b, ks) of rows 128 b .. 128 b + 127 at byte
 *                (b * S + ks) * 512;           ceil(M / 128) * S * 512 bytes
 *       B_scale: chunk (c, ks) of columns 128 c .. 128 c + 127 at byte
 *                ((c / 2 * S + ks) * 2 + c % 2) * 512;
 *                                              ceil(N / 256) * S * 1024 bytes
 *     Entries for rows (columns) past M (N) and K blocks past K/32 must hold
 *     a finite scale (mxgemm_quantize_ex writes 127 there).  Device pointers
 *     16-byte aligned (MXGEMM_ERR_MISALIGNED). */
typedef enum { MXGEMM_SCALES_ROW_MAJOR = 0, MXGEMM_SCALES_PACKED = 1 } mxgemm_scale_layout_t;

/* Element formats (OCP Microscaling Formats v1.0).  Every element occupies
 * one byte in A and B, also for the 6- and 4-bit formats, whose code sits
 * in the low bits of its byte (the upper bits are ignored). */
typedef enum {
  MXGEMM_FMT_E4M3 = 0, /* FP8, max 448, no infinities */
  MXGEMM_FMT_E5M2 = 1, /* FP8, max 57344, with infinities */
  MXGEMM_FMT_E2M3 = 2, /* FP6, max 7.5 */
  MXGEMM_FMT_E3M2 = 3, /* FP6, max 28 */
  MXGEMM_FMT_E2M1 = 4  /* FP4, max 6 */
} mxgemm_format_t;

/* Create a handle bound to CUDA device `device`.  The handle carries the
 * state that mxgemm_run needs between calls (workspace, plan cache, status
 * word); the scaled product itself is `async_dot_scaled` of "TLX API Quick
 * Reference", section "Matrix Multiply (MMA)", whose operands mxgemm_run
 * takes in the same order.  Fails with
 * MXGEMM_ERR_UNSUPPORTED_DEVICE unless the device is compute capability 10.3
 * (sm_103, GB300).  Allocates the handle's device status word and its
 * partial-sum flag slots. */
int mxgemm_create(mxgemm_handle_t *out, int device);

/* Enqueue C (+)= A.B on `stream` (NULL = the legacy default stream): the
 * scaled product D = (A*scale_A) @ (B*scale_B) (+ D) of "TLX API Quick
 * Reference", section "Matrix Multiply (MMA)" (`async_dot_scaled` with
 * A_format = B_format = "e4m3" and use_acc), over the whole of M, N, K.
 *   M, N, K   : sizes, each in [0, 2^31); K must be a multiple of 32.
 *               M == 0 or N == 0 is a no-op; K == 0 sets C to 0 (use_acc=0)
 *               or leaves it unchanged (use_acc=1).
 *   A, B, C   : device pointers, 16-byte aligned (MXGEMM_ERR_MISALIGNED).
 *   A_scale, B_scale : device pointers, any alignment (row-major layout,
 *               the default); with MXGEMM_OPT_SCALE_LAYOUT =
 *               MXGEMM_SCALES_PACKED the packed chunks of
 *               mxgemm_scale_layout_t, 16-byte aligned.
 *   use_acc   : 0 or 1 (see above).
 *   out_dtype : MXGEMM_OUT_F32 or MXGEMM_OUT_BF16.
 * C must not overlap A, B or the scales.  The call returns after enqueueing;
 * the handle keeps no reference to the caller's buffers after the work
 * completes. */
int mxgemm_run(mxgemm_handle_t h, int64_t M, int64_t N, int64_t K,
               const void *A, const void *A_scale, const void *B,
               const void *B_scale, void *C, int use_acc, int out_dtype,
               mxgemm_stream_t stream);

/* The same product with every operand and the result in HOST memory.
 * Arguments as for mxgemm_run, except that A, A_scale, B, B_scale and C
 * are host pointers (any alignment).  The call copies B and B_scale to the
 * device, then pipelines the rows of A and C in slabs of at most
 * max(256, M/8 rounded up to 256) rows through three device slots: while
 * one slab's GEMM runs on `stream`, the next slab's A rows (and, with
 * use_acc, its C rows) are copied in on an internal stream and the earlier
 * slabs' C rows are copied out on another.  `stream` waits for the last copy, so
 * C on the host is complete once `stream` is: synchronize it before reading
 * C.  The host buffers must hold their values when the call is made and
 * stay unchanged until `stream` has completed it; consecutive calls on one
 * handle overlap (one call's copies in run while the previous call's
 * copies out finish).  Page-locked (pinned) host buffers let the copies
 * overlap; pageable ones work but the copies then block the calling thread.  The handle owns
 * the device staging buffers (B, B_scale and the three slots), which grow
 * lazily in stream order on `stream`, and two internal streams.  Use one
 * stream per handle.  K == 0 synchronizes `stream` and then zeroes C (use_acc
 * = 0) or leaves it unchanged.  Errors as for mxgemm_run; MXGEMM_ERR_CUDA if
 * a copy cannot be enqueued. */
int mxgemm_run_host(mxgemm_handle_t h, int64_t M, int64_t N, int64_t K,
                    const void *A, const void *A_scale, const void *B,
                    const void *B_scale, void *C, int use_acc, int out_dtype,
                    mxgemm_stream_t stream);

/* MX quantization on the GPU: a real matrix X (R x C, row-major, dense) to
 * E4M3 codes with one E8M0 scale per block of 32 values -- the operands of
 * mxgemm_run.  Per block (OCP Microscaling Formats v1.0 conversion, E4M3
 * maximum 448):
 *   scale  = clamp(127 + ceil(log2(amax / 448)), 0, 254); 127 when amax = 0
 *   code_i = nearest E4M3 value to clamp(x_i * 2^(127 - scale), +-448),
 *            ties to even, sign kept.
 *   x_dtype    : MXGEMM_IN_F32 or MXGEMM_IN_BF16.
 *   along_cols : 0 -> blocks run along each row (C % 32 == 0); scales is
 *                R x (C/32): X = A (M x K) gives A and A_scale.
 *                1 -> blocks run down each column (R % 32 == 0); scales is
 *                C x (R/32), row j holding column j's scales: X = B (K x N)
 *                gives B and B_scale.
 *   X, codes, scales : device pointers; X and codes 16-byte aligned
 *                (MXGEMM_ERR_MISALIGNED).  codes is R x C bytes.
 * X must hold finite values (the codes of non-finite inputs are
 * unspecified).  Needs no handle: nothing is allocated; enqueued on
 * `stream`.  Errors as for mxgemm_run. */
typedef enum { MXGEMM_IN_F32 = 0, MXGEMM_IN_BF16 = 1 } mxgemm_in_dtype_t;
int mxgemm_quantize(const void *X, int x_dtype, int64_t R, int64_t C, int along_cols,
                    void *codes, void *scales, mxgemm_stream_t stream);

/* mxgemm_quantize with stochastic rounding of the codes: the FP32 -> FP8
 * rounding with caller-supplied random bits ("TLX API Quick Reference",
 * section "Utility", tlx.stoch_round).  The scales are those of
 * mxgemm_quantize.  Element (i, j) is scaled to the FP32 value
 * y = X[i][j] * 2^(127 - scale); with lo <= |y| < lo + q the E4M3
 * magnitudes around |y| (|y| clamped to 448) and r = rand_bits[i * C + j],
 * the code is lo + q when r < 2^32 * (|y| - lo) / q, else lo (so it rounds up
 * with probability (|y| - lo) / q); the sign is kept.
 *   rand_bits : device pointer, R x C uint32 words, row-major (the index of
 *               X, for either block direction), 16-byte aligned
 *               (MXGEMM_ERR_MISALIGNED); read only.  NULL is invalid.
 * Other arguments, layouts and errors as for mxgemm_quantize. */
int mxgemm_quantize_sr(const void *X, int x_dtype, int64_t R, int64_t C, int along_cols,
                       const void *rand_bits, void *codes, void *scales,
                       mxgemm_stream_t stream);

/* mxgemm_quantize with both choices: rand_bits NULL rounds to nearest
 * (mxgemm_quantize), else stochastically (mxgemm_quantize_sr);
 * scale_layout (an mxgemm_scale_layout_t) is the layout of `scales`.
 * MXGEMM_SCALES_PACKED writes the order a run with MXGEMM_OPT_SCALE_LAYOUT
 * = MXGEMM_SCALES_PACKED reads: along_cols = 0 gives A_scale of an M x K
 * matrix X (M = R, K = C), along_cols = 1 gives B_scale of a K x N matrix X
 * (K = R, N = C).  The whole packed area (mxgemm_scale_bytes) is written,
 * the padding entries as 127; `scales` then needs 16-byte alignment
 * (MXGEMM_ERR_MISALIGNED).  Other arguments and errors as for the two
 * entry points above. */
int mxgemm_quantize_ex(const void *X, int x_dtype, int64_t R, int64_t C, int along_cols,
                       const void *rand_bits, int scale_layout, void *codes, void *scales,
                       mxgemm_stream_t stream);

/* Bytes of the scales that mxgemm_quantize_ex writes for an R x C matrix
 * (and a run reads): row-major R * (C/32) or C * (R/32); packed as above.
 * The block dimension (C, or R with along_cols) must be a multiple of 32
 * (MXGEMM_ERR_INVALID_VALUE).  Host-only, no device work. */
int mxgemm_scale_bytes(int64_t R, int64_t C, int along_cols, int scale_layout,
                       int64_t *bytes_out);

/* Set an option (mxgemm_option_t) on the handle; applies to later runs. */
int mxgemm_set_option(mxgemm_handle_t h, int option, int64_t value);

/* Synchronize `stream`, then read and clear the handle's device status word.
 * *status_out receives MXGEMM_OK or MXGEMM_ERR_TIMEOUT; *detail_out (may be
 * NULL) receives where the first failing wait was (role | stage << 8 |
 * tile << 16), 0 when none.  Roles: 0x01 producer (free stage), 0x02 MMA
 * issuer (free accumulator), 0x03 MMA issuer (full stage), 0x04 MMA issuer
 * (final commit), 0x05 epilogue (full accumulator), 0x06 epilogue (stream-K
 * partials), 0x07 / 0x08 cluster-launch-control response / free slot,
 * 0x09 scale loader (free stage), 0x0A scale loader (staged scale rows),
 * 0x0B scale loader (staging load at exit), 0x0C producer (scale loader's
 * first staging load), 0x11 producer (drain at exit). */
int mxgemm_get_device_status(mxgemm_handle_t h, mxgemm_stream_t stream,
                             int *status_out, int *detail_out);

/* Timing hook: record the CUDA events `ev_before` and `ev_after`
 * (cudaEvent_t handles created by the caller; either may be NULL) on the
 * run's stream immediately before and after the GEMM kernel launch of every
 * later mxgemm_run on this handle, so that the kernel alone can be timed
 * with the caller's events.  Passing NULL, NULL turns the hook off.  The
 * handle does not own the events. */
int mxgemm_set_profile_events(mxgemm_handle_t h, void *ev_before, void *ev_after);

/* Number of kernels this handle has launched so far (the GEMM kernel and its
 * prepasses), in *count_out. */
int mxgemm_get_launch_count(mxgemm_handle_t h, int64_t *count_out);

/* Free the handle's device memory (synchronizes its device) and the handle
 * (the counterpart of mxgemm_create; the product is that of "TLX API Quick
 * Reference", section "Matrix Multiply (MMA)"). */
int mxgemm_destroy(mxgemm_handle_t h);

/* The same product as mxgemm_run, for callers that cannot allocate device
 * memory where they call it: a plug-in whose host framework owns all device
 * memory (and hands the plug-in only its inputs and outputs), or code that
 * must not allocate after start-up (an allocation there can fail, block on
 * other streams or fragment the caller's pool).  It takes no handle,
 * allocates nothing (no cudaMalloc, cudaFree or allocating library call) and
 * runs on the current device and the given stream.  The pages have no
 * counterpart to this entry point.
 *
 * Scratch: B re-pitched to a 16-byte row pitch when N % 16 != 0 goes to one
 * file-scope device array of 16 MiB, which every GPU that loads this library
 * holds until the process exits (the single-CTA kernel reads the scales in
 * their row-major layout and needs no other scratch).  A problem with
 * N % 16 != 0 needs K * round_up(N, 16) bytes rounded up to 1 KiB; more than
 * 16 MiB is rejected with MXGEMM_ERR_TOO_LARGE before anything is
 * enqueued.  All calls share that array and it keeps the last call's
 * contents, so calls whose work overlaps on the GPU (different streams, or
 * different host threads) race and must be serialised by the caller.
 *
 * The first call on a device does a one-time set-up for that device (device
 * check and lookup of the array's device address); make that first call
 * before starting any stream capture.  Arguments, layouts and use_acc are as
 * for mxgemm_run; it always uses single-CTA 128x256 tiles computed whole.  A
 * device-side wait that runs out records MXGEMM_ERR_TIMEOUT in a status word
 * of the current device (C is then incomplete); the word keeps the first
 * failure until mxgemm_noalloc_get_status reads and clears it. */
int mxgemm_run_noalloc(int64_t M, int64_t N, int64_t K, const void *A,
                       const void *A_scale, const void *B, const void *B_scale,
                       void *C, int use_acc, int out_dtype,
                       mxgemm_stream_t stream);

/* Synchronize `stream`, then read and clear the current device's status
 * word of mxgemm_run_noalloc: *status_out receives MXGEMM_OK or
 * MXGEMM_ERR_TIMEOUT (the first failure of any call since the last read),
 * *detail_out (may be NULL) where the wait was, with the codes of
 * mxgemm_get_device_status.  Allocates nothing: the word is copied into the
 * caller's host ints.  The first use on a device does the same one-time
 * set-up as mxgemm_run_noalloc.  No counterpart on the pages, as for
 * mxgemm_run_noalloc. */
int mxgemm_noalloc_get_status(mxgemm_stream_t stream, int *status_out, int *detail_out);

/* Options of mxgemm_run_noalloc, for the whole process (it has no handle):
 * MXGEMM_OPT_WAIT_TIMEOUT_NS (default 2e9) and the test hook
 * MXGEMM_OPT_TEST_STALL_PRODUCER (default 0), as for mxgemm_set_option;
 * other options are MXGEMM_ERR_INVALID_VALUE.  Applies to later calls. */
int mxgemm_noalloc_set_option(int option, int64_t value);

/* Static description of a status code. */
const char *mxgemm_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MXGEMM_H_ */
