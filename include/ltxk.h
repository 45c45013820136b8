/*
 * ltxk.h -- C ABI of libltxk.so: RMSNorm and fused RMSNorm + rotary position
 * embedding (RoPE) on one NVIDIA GB300 GPU (sm_103a), with the AdaLN and
 * residual-add norms, standalone RoPE from token positions and the tanh
 * GELU / GEGLU, in bfloat16 (the calls without a dtype), fp16 and fp32 (the
 * _dt calls).
 *
 * Where the operations come from
 *   RMSNorm: "cuda-kernels" skill page (Hugging Face), sections "Kernel-
 *   Specific Guidelines / RMSNorm" (layout [..., hidden_size], epsilon
 *   default 1e-6, the weight may be absent) and "RMSNorm Micro-benchmarks"
 *   (bf16 activations shaped [batch x seq x hidden]).  The pages print no
 *   formula; the operation implemented is, per row r of x [rows, hidden]:
 *       y[r, j] = bf16_rne( x[r, j] * w[j] / sqrt(mean_j x[r, j]^2 + eps) )
 *   computed in fp32 with one rounding to bfloat16 at the end.
 *   Fused form: "ltx-kernels" README, opening list (`ops_cpp`: fused element
 *   ops rms_norm_rope and rms_norm_split_rope) and the skill page's "Kernel-
 *   Specific Guidelines / RoPE" ([batch, seq, heads, head_dim] text layout,
 *   [batch, t*h*w, heads, head_dim] video layout).  The RMSNorm runs over the
 *   full hidden = heads * head_dim with the full-length weight; then, in
 *   registers and before the single bf16 rounding, every head is rotated pair
 *   by pair with c = cos[pos, p], s = sin[pos, p]:
 *       a' = a*c - b*s,   b' = a*s + b*c
 *   LTXK_ROPE_INTERLEAVED pairs (a, b) = (h*D + 2p, h*D + 2p + 1);
 *   LTXK_ROPE_SPLIT_HALF  pairs (a, b) = (h*D + p,  h*D + p + D/2).
 *
 * Conventions shared by every entry point
 *   - Tensor pointers are DEVICE pointers (or managed memory) of the current
 *     CUDA device.  bfloat16 data travel as void* (IEEE-754 binary32 upper
 *     halves, little-endian).  All tensors are dense and row-major.
 *     Page-locked host memory the device can address (cudaHostAlloc or
 *     cudaHostRegister; on GB300 through NVLink-C2C) may be passed as well:
 *     the kernels then read and write it across the host link themselves
 *     (zero-copy), with the same results.
 *   - The caller owns and allocates every buffer (the out-variant convention
 *     of the pages' `Tensor! out` ops); the library allocates no device
 *     memory and keeps no per-call state.
 *   - Work is queued asynchronously on `stream` (NULL = the legacy default
 *     stream); the call returns once the launch is queued.
 *   - Arguments are validated on the host BEFORE any CUDA call; on error
 *     nothing is launched and an ltxk_status is returned.
 *   - out == x (in place) is allowed: every row is read completely before
 *     any element of it is written.  Any other overlap of out with x, w or
 *     the tables is rejected with LTXK_ERR_OVERLAP.
 *   - rows == 0 is a no-op returning LTXK_OK.
 *   - Pointers need only the 2-byte (bf16) / 4-byte (fp32) alignment of
 *     their type.  16-byte-aligned pointers with hidden % 8 == 0 (and, for
 *     the fused form, head_dim % 8 == 0 interleaved or % 16 == 0 split-half)
 *     take the vectorised kernels; anything else takes the element-wise
 *     kernel, which computes the same values.  There is no CPU fallback.
 *   - Numerics: the sum of squares is kept in fp32, so rows whose sum of
 *     squares exceeds FLT_MAX (elements of magnitude about 2^63 and up)
 *     overflow; with eps == 0 an all-zero row yields NaN (0/0).
 */
#ifndef LTXK_H_
#define LTXK_H_

#include <stdint.h>

#if defined(__GNUC__)
#define LTXK_API __attribute__((visibility("default")))
#else
#define LTXK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t (a CUDA runtime stream handle). */
struct CUstream_st;
typedef struct CUstream_st* ltxk_stream_t;

typedef enum {
    LTXK_OK = 0,
    LTXK_ERR_NULL = 1,      /* a required pointer is NULL */
    LTXK_ERR_SHAPE = 2,     /* rows < 0, hidden <= 0, heads*head_dim overflow,
                               odd head_dim, seq_len <= 0, size limits */
    LTXK_ERR_ALIGN = 3,     /* a pointer lacks its element's alignment */
    LTXK_ERR_MODE = 4,      /* unknown RoPE pairing mode */
    LTXK_ERR_OVERLAP = 5,   /* out partially overlaps x, or overlaps w/cos/sin */
    LTXK_ERR_CUDA = 6,      /* a CUDA runtime call or the launch failed; see
                               ltxk_last_cuda_error() */
    LTXK_ERR_TIMEOUT = 7,   /* a kernel gave up waiting for a bulk copy (see
                               ltxk_fault_status) */
    LTXK_ERR_DTYPE = 8      /* unknown LTXK_DTYPE_* code */
} ltxk_status;

enum { LTXK_ROPE_INTERLEAVED = 0, LTXK_ROPE_SPLIT_HALF = 1 };

/* Element types of the rows, weight and conditioning vectors ("cuda-kernels"
 * skill page, "Supported Data Types": every kernel in three precision modes).
 * RoPE tables stay fp32 in every mode. */
enum { LTXK_DTYPE_BF16 = 0, LTXK_DTYPE_F16 = 1, LTXK_DTYPE_F32 = 2 };

/* Largest hidden size (elements per row) the library accepts. */
#define LTXK_MAX_HIDDEN (1 << 30)

/*
 * ltxk_rms_norm -- y = x * w / sqrt(mean(x^2) + eps) per row, bf16 in/out.
 *   out    [rows, hidden] bf16, written.
 *   x      [rows, hidden] bf16, read.
 *   w      [hidden] bf16, or NULL for a weight of ones (the pages'
 *          elementwise_affine=False case).
 *   rows   >= 0.  hidden in [1, LTXK_MAX_HIDDEN].
 *   eps    added to the mean square inside the square root (default on the
 *          pages: 1e-6).
 * Returns an ltxk_status.
 */
LTXK_API int ltxk_rms_norm(void* out, const void* x, const void* w, int64_t rows,
                  int64_t hidden, float eps, ltxk_stream_t stream);

/*
 * ltxk_rms_norm_rope -- RMSNorm over hidden = heads*head_dim, then RoPE per
 * head, with PER-ROW tables: row r uses cos[r, :] and sin[r, :].
 *   out, x  [rows, heads*head_dim] bf16.   w as for ltxk_rms_norm.
 *   cos,sin [rows, head_dim/2] fp32 (device).
 *   heads >= 1, head_dim >= 2 and even, mode = LTXK_ROPE_*.
 * For x shaped [batch, seq, heads*head_dim] with one [seq, head_dim/2] table
 * per sequence, use ltxk_rms_norm_rope_seq instead of repeating the table.
 */
LTXK_API int ltxk_rms_norm_rope(void* out, const void* x, const void* w,
                       const float* cos, const float* sin, int64_t rows,
                       int heads, int head_dim, int mode, float eps,
                       ltxk_stream_t stream);

/*
 * ltxk_rms_norm_rope_seq -- as ltxk_rms_norm_rope, with tables shared by all
 * sequences of a batch: cos, sin are [seq_len, head_dim/2] and row r uses
 * table row (r mod seq_len), i.e. x is [batch, seq_len, heads*head_dim].
 * seq_len >= 1; rows need not be a multiple of seq_len.
 */
LTXK_API int ltxk_rms_norm_rope_seq(void* out, const void* x, const void* w,
                           const float* cos, const float* sin, int64_t rows,
                           int heads, int head_dim, int mode, float eps,
                           int64_t seq_len, ltxk_stream_t stream);

/*
 * ltxk_rms_norm_adaln -- AdaLN-modulated RMSNorm, the DiT conditioning of
 * the "cuda-kernels" page ("Kernel-Specific Guidelines / AdaLN"):
 *     y[r, j] = bf16_rne( n[r, j] * (1 + scale[c, j]) + shift[c, j] ),
 *     n = x * w / sqrt(mean(x^2) + eps) (the RMSNorm above, fp32),
 *     c = r / rows_per_cond.
 *   out, x        [rows, hidden] bf16.   w [hidden] bf16 or NULL (ones: the
 *                 pages' weightless LTX-Video block norm).
 *   scale, shift  [ceil(rows / rows_per_cond), hidden] bf16: one vector per
 *                 conditioning row (per batch item for x [B, S, hidden] with
 *                 rows_per_cond = S), shared by rows_per_cond rows.
 *   rows_per_cond >= 1.
 * out may equal x; it must not overlap w, scale or shift.
 */
LTXK_API int ltxk_rms_norm_adaln(void* out, const void* x, const void* w,
                                 const void* scale, const void* shift,
                                 int64_t rows, int64_t hidden,
                                 int64_t rows_per_cond, float eps,
                                 ltxk_stream_t stream);

/*
 * ltxk_add_rms_norm -- fused residual add + RMSNorm, the add-then-norm that
 * precedes each block norm:
 *     h[r, j] = bf16_rne( x[r, j] + residual[r, j] )     -> residual_out
 *     y[r, j] = bf16_rne( h[r, j] * w[j] / sqrt(mean_j h[r, j]^2 + eps) ) -> out
 * The norm reads the rounded h, exactly as the unfused add then norm would.
 *   out, residual_out, x, residual  [rows, hidden] bf16.  w [hidden] or NULL.
 * out and residual_out must be disjoint.  Either may be exactly one of the
 * inputs (in place, e.g. residual_out == residual to update the residual
 * stream); partial overlaps are rejected.  Reads 4 and writes 4 bytes per
 * element.
 */
LTXK_API int ltxk_add_rms_norm(void* out, void* residual_out, const void* x,
                               const void* residual, const void* w,
                               int64_t rows, int64_t hidden, float eps,
                               ltxk_stream_t stream);

/*
 * The same four row operations for rows of element type `dtype`
 * (LTXK_DTYPE_BF16, _F16 or _F32); x, out, w and (AdaLN) scale and shift,
 * (residual add) residual and residual_out all have that type, and every
 * output is one round-to-nearest-even of the fp32 result to it.
 *   - Arguments, layouts and overlap rules are those of the bf16 calls
 *     above; pointers need the alignment of the element type (2 or 4
 *     bytes), 16-byte alignment (and hidden % 8 == 0) takes the vector
 *     kernels.
 *   - ltxk_rms_norm_rope_dt takes tables [seq_len, head_dim/2] with row r
 *     using table row r mod seq_len, as ltxk_rms_norm_rope_seq (seq_len =
 *     rows gives per-row tables).
 *   - Numerics: for fp16, x*w is exact in fp32 as for bf16, so every output
 *     is within 1 fp16 ulp of the exact value.  For fp32 rows, x*w itself
 *     rounds, and the output carries the fp32 error of the sum of squares,
 *     rsqrtf and one or two products (a few ulp; more under cancellation in
 *     RoPE or AdaLN).  fp16 outputs beyond 65504 round to infinity.
 * An unknown dtype returns LTXK_ERR_DTYPE before any other check.
 */
LTXK_API int ltxk_rms_norm_dt(void* out, const void* x, const void* w, int64_t rows,
                              int64_t hidden, float eps, int dtype, ltxk_stream_t stream);
LTXK_API int ltxk_rms_norm_rope_dt(void* out, const void* x, const void* w,
                                   const float* cos, const float* sin, int64_t rows,
                                   int heads, int head_dim, int mode, float eps,
                                   int64_t seq_len, int dtype, ltxk_stream_t stream);
LTXK_API int ltxk_rms_norm_adaln_dt(void* out, const void* x, const void* w,
                                    const void* scale, const void* shift, int64_t rows,
                                    int64_t hidden, int64_t rows_per_cond, float eps,
                                    int dtype, ltxk_stream_t stream);
LTXK_API int ltxk_add_rms_norm_dt(void* out, void* residual_out, const void* x,
                                  const void* residual, const void* w, int64_t rows,
                                  int64_t hidden, float eps, int dtype,
                                  ltxk_stream_t stream);

/*
 * ltxk_rope -- standalone rotary position embedding with the rotation angles
 * computed on the device from token positions: no cos/sin tables in memory
 * ("cuda-kernels" skill page, "Kernel-Specific Guidelines / RoPE": 1D text
 * [batch, seq, heads, head_dim], 3D video [batch, t*h*w, heads, head_dim];
 * LTX-Video computes its own rotary angles).
 *   out, x   [rows, heads*head_dim] of element type `dtype`; out == x (in
 *            place) is allowed, any other overlap returns LTXK_ERR_OVERLAP.
 *   Row r is token s = r mod (grid_t*grid_h*grid_w) (x is [batch, tokens,
 *   heads, head_dim] with the token index inner), with coordinates
 *     (s / (grid_h*grid_w), (s / grid_w) mod grid_h, s mod grid_w).
 *   The head_dim/2 rotation pairs split into consecutive groups of pairs_t,
 *   pairs_h, pairs_w pairs (axis t, then h, then w; they must add up to
 *   head_dim/2).  Pair k of an axis with n pairs turns by
 *     angle = coordinate * theta^(-k/n),
 *   and every head's pair (a, b) becomes (a cos - b sin, a sin + b cos),
 *   rounded once.  mode = LTXK_ROPE_* selects the pairing as for the fused
 *   form.  1D text: grid (seq_len, 1, 1), pairs (head_dim/2, 0, 0), which is
 *   the usual theta^(-2k/head_dim).
 *   head_dim even, at most 512; theta > 0.
 * Numerics: angles are formed and reduced in fp64, cos/sin in fp32 with a
 * correction for the reduced angle's fp32 remainder (a few 1e-8 absolute for
 * coordinates below 2^24), and the rotation uses Kahan's 2x2-determinant
 * algorithm.  An output is therefore within 1 ulp of the exact value, except
 * where a' or b' cancels: its error is then bounded by a few fp32 ulps of
 * |a| + |b|.
 */
LTXK_API int ltxk_rope(void* out, const void* x, int64_t rows, int heads, int head_dim,
                       int mode, int64_t grid_t, int64_t grid_h, int64_t grid_w,
                       int pairs_t, int pairs_h, int pairs_w, double theta, int dtype,
                       ltxk_stream_t stream);

/*
 * ltxk_rope_tables -- the cos and sin tables of the fused RMSNorm + RoPE
 * (ltxk_rms_norm_rope_seq's cos/sin inputs) for token positions, computed on
 * the device with ltxk_rope's angles: row s of each table holds, for the
 * head_dim/2 pairs, cos and sin of the angle ltxk_rope gives token
 * s mod (T*H*W) (same coordinates, pair split and frequencies).
 *   cos_out, sin_out  [tokens, head_dim/2] fp32 on the device, 4-byte
 *                     aligned; they must not overlap (LTXK_ERR_OVERLAP).
 *   tokens >= 0 (0 is a no-op); tokens * head_dim <= 2^40.
 *   head_dim, grid_*, pairs_*, theta  as for ltxk_rope (head_dim <= 512).
 * Each value is within about 2 * 2^-24 of the exact cos / sin for
 * coordinates below 2^24.  Writes 8 bytes per pair and token.
 */
LTXK_API int ltxk_rope_tables(float* cos_out, float* sin_out, int64_t tokens, int head_dim,
                              int64_t grid_t, int64_t grid_h, int64_t grid_w, int pairs_t,
                              int pairs_h, int pairs_w, double theta, ltxk_stream_t stream);

/*
 * ltxk_gelu_tanh -- elementwise tanh-approximated GELU, bf16 -> bf16:
 *   y = x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))
 * ("cuda-kernels" skill page, "Kernel-Specific Guidelines / GEGLU vs GELU":
 * the approximate GELU of LTX-Video's feed-forward blocks).  Computed in
 * fp32, rounded once to bf16 (nearest even).
 *   out, x  n contiguous bf16 values on the device; out == x (in place) is
 *           allowed, any other overlap returns LTXK_ERR_OVERLAP.
 *   n       in [0, 2^40]; n == 0 is a no-op.
 * Pointers need 2-byte alignment; 16-byte aligned pointers take the vector
 * kernel.  Reads 2 and writes 2 bytes per element.
 */
LTXK_API int ltxk_gelu_tanh(void* out, const void* x, int64_t n,
                            ltxk_stream_t stream);

/*
 * ltxk_geglu -- gated GELU over the last dimension (same page and section:
 * GEGLU halves the last dimension):
 *   out[r, j] = x[r, j] * gelu_tanh(x[r, hidden + j]),  j < hidden
 * i.e. the first half of each input row is the value, the second half the
 * gate, and the product of the fp32 value and the fp32 gelu is rounded once.
 *   x    [rows, 2*hidden] bf16, row-major contiguous.
 *   out  [rows, hidden] bf16; must not overlap x (LTXK_ERR_OVERLAP).
 *   rows >= 0 (0 is a no-op); hidden in [1, LTXK_MAX_HIDDEN];
 *        rows * hidden <= 2^40.
 * hidden % 8 == 0 with 16-byte aligned pointers takes the vector kernel.
 * Reads 4 and writes 2 bytes per output element.
 */
LTXK_API int ltxk_geglu(void* out, const void* x, int64_t rows, int64_t hidden,
                        ltxk_stream_t stream);

/*
 * ltxk_gelu_tanh_dt, ltxk_geglu_dt -- ltxk_gelu_tanh and ltxk_geglu for one
 * element type (LTXK_DTYPE_BF16, _F16 or _F32; input and output share it):
 * the page's "Supported Data Types" (__half, __nv_bfloat16, float).  Same
 * arguments, layout and errors; pointers need the element's alignment, and an
 * unknown dtype returns LTXK_ERR_DTYPE.  bf16 gives exactly the bits of the
 * calls above.  fp16 is rounded once from the same fp32 evaluation.  The
 * vector kernels want 16-byte aligned pointers and, for GEGLU, hidden % 8 == 0
 * (fp32: hidden % 4 == 0); anything else takes the element kernel.  fp32
 * carries the fp32 evaluation's error:
 *   |y - gelu| <= 2^-24 (32 + 5 |q| / (1 + 2^q)) |gelu| + 2^-148,
 * with q = (2 / ln 2) sqrt(2 / pi) (x + 0.044715 x^3) (the |q| term is the
 * fp32 rounding of q, magnified by 2^q's sensitivity in the left tail).
 * Bytes per element: 2, 2 or 4 read and written (GEGLU: twice the reads).
 */
LTXK_API int ltxk_gelu_tanh_dt(void* out, const void* x, int64_t n, int dtype,
                               ltxk_stream_t stream);
LTXK_API int ltxk_geglu_dt(void* out, const void* x, int64_t rows, int64_t hidden,
                           int dtype, ltxk_stream_t stream);

/*
 * ltxk_rms_norm_host -- ltxk_rms_norm for x and y in HOST memory, pipelined.
 * The rows are cut into chunks; chunk i is copied in on streams[i % n],
 * normalised in place in staging slot i % n, and copied out, so the copy-in,
 * kernel and copy-out of consecutive chunks overlap.  Asynchronous: the
 * results are in out_host once every stream in `streams` has finished.
 *   out_host, x_host [rows, hidden] bf16 in host memory; page-locked memory
 *                 (cudaHostAlloc / torch pin_memory) lets the copies overlap.
 *   w             [hidden] bf16 on the device, or NULL (ones).
 *   staging       device memory of staging_bytes, 256-byte aligned, owned by
 *                 the caller; split into n_streams slots of at least one row.
 *   streams       n_streams (1 .. LTXK_HOST_MAX_STREAMS) streams, ideally
 *                 distinct non-default streams.
 * When out_host and x_host are both page-locked host memory the device can
 * address (cudaHostAlloc, cudaHostRegister, torch pin_memory), the call
 * instead queues one kernel on streams[0] that reads x and writes y across
 * the host link directly (zero-copy; on GB300 over NVLink-C2C, both
 * directions at once); staging is then unused.  out_host may equal x_host
 * (in place) but must not partly overlap it (LTXK_ERR_OVERLAP).
 * The library allocates nothing.  Returns an ltxk_status; argument errors
 * are reported before any copy is queued.
 */
#define LTXK_HOST_MAX_STREAMS 8
LTXK_API int ltxk_rms_norm_host(void* out_host, const void* x_host, const void* w,
                                int64_t rows, int64_t hidden, float eps,
                                void* staging, int64_t staging_bytes,
                                const ltxk_stream_t* streams, int n_streams);

/*
 * ltxk_fault_status -- did any kernel on the current device give up waiting
 * since the last call?  The TMA-ring kernel bounds each wait for a bulk copy
 * of a row (about two seconds); a wait that runs out sets a device fault
 * word, lets the warp's other copies land, and ends the warp without writing
 * the rows it had left.  This call waits for the device to finish
 * (cudaDeviceSynchronize), reads and clears that word, and returns LTXK_OK,
 * LTXK_ERR_TIMEOUT, or LTXK_ERR_CUDA.  The word lives in the library's
 * static device memory (4 bytes per device); nothing is allocated.
 */
LTXK_API int ltxk_fault_status(void);

/*
 * ltxk_set_path -- process-wide choice of kernel family for the vectorised
 * cases (for tuning and for testing every family on the same shapes):
 * LTXK_PATH_AUTO (default), LTXK_PATH_REGISTERS (rows loaded straight into
 * registers) or LTXK_PATH_TMA (rows streamed through a shared-memory ring by
 * bulk copies; used where one warp can own a row, hidden <= 4096).  All
 * families compute the same values.  Returns the previous setting, or -1
 * for an unknown value (the setting is then unchanged).
 */
enum { LTXK_PATH_AUTO = 0, LTXK_PATH_REGISTERS = 1, LTXK_PATH_TMA = 2 };
LTXK_API int ltxk_set_path(int path);

/*
 * ltxk_diag_missing_copy -- diagnostic for the bounded waits: runs the
 * TMA-ring RMSNorm kernel on x [rows, hidden] (16-byte aligned, hidden a
 * multiple of 8 and at most 4096) with the bulk copy of every warp's first
 * row never issued, so that those waits run out after wait_limit_ns
 * nanoseconds (1e3 .. 1e10).  No copy is left in flight.  Afterwards
 * ltxk_fault_status() returns LTXK_ERR_TIMEOUT; rows whose copies did land
 * may have been written to out.  Returns an ltxk_status for the launch.
 */
LTXK_API int ltxk_diag_missing_copy(void* out, const void* x, int64_t rows,
                                    int64_t hidden, uint64_t wait_limit_ns,
                                    ltxk_stream_t stream);

/*
 * ltxk_rms_norm_noalloc -- the same RMSNorm as ltxk_rms_norm, for callers
 * that cannot allocate device memory: for example an engine whose device
 * memory all comes from its own pre-sized pool, or a latency-critical loop
 * where an allocation's implicit device synchronisation is not acceptable.
 * The pages have no counterpart to it.
 *
 * It runs the TMA-ring kernel, whose only device memory beyond x, w and out
 * is one fault word for its bounded waits.  That word lives in a file-scope
 * static device array of LTXK_NOALLOC_SCRATCH_WORDS 32-bit words (256 bytes)
 * that every GPU loading the library holds until the process exits; the call
 * allocates nothing and calls no cudaMalloc or cudaFree.
 *   out, x, w : as for ltxk_rms_norm, but 16-byte aligned (w may be NULL).
 *   hidden    : a multiple of 8 and at most LTXK_NOALLOC_MAX_HIDDEN (one warp
 *               per row); larger or ragged rows return LTXK_ERR_SHAPE.
 * The first call on a device resolves the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Each call clears the fault word on `stream`
 * before its kernel.  A wait that runs out sets the word and leaves that
 * warp's remaining rows unwritten; ltxk_noalloc_fault_status() reads the
 * word back (and clears it), so check it after a call whose output matters.
 * All calls share the array, which keeps the last call's contents, so calls
 * that overlap on the GPU (other streams, other threads) race on it: on the
 * fault word, one call's clear can erase another call's fault.
 */
#define LTXK_NOALLOC_SCRATCH_WORDS 64
#define LTXK_NOALLOC_MAX_HIDDEN 4096
LTXK_API int ltxk_rms_norm_noalloc(void* out, const void* x, const void* w,
                                   int64_t rows, int64_t hidden, float eps,
                                   ltxk_stream_t stream);

/*
 * ltxk_noalloc_fault_status -- waits for the current device to finish
 * (cudaDeviceSynchronize), then reads the fault word of
 * ltxk_rms_norm_noalloc's static array.  Returns LTXK_ERR_TIMEOUT if a
 * bounded wait of the last call ran out (and clears the word), LTXK_OK if
 * not, LTXK_ERR_CUDA if a CUDA call failed.  Allocates nothing.  Like the
 * entry point it serves, the pages have no counterpart to it.
 */
LTXK_API int ltxk_noalloc_fault_status(void);

/*
 * ltxk_diag_noalloc_missing_copy -- diagnostic for the bounded waits of
 * ltxk_rms_norm_noalloc: the same call (no weight, eps 1e-6) with the bulk
 * copy of every warp's first row never issued, so that those waits run out
 * after wait_limit_ns nanoseconds (1e3 .. 1e10).  No copy is left in
 * flight.  Afterwards ltxk_noalloc_fault_status() returns LTXK_ERR_TIMEOUT.
 * Returns an ltxk_status for the launch (the entry point's checks).
 */
LTXK_API int ltxk_diag_noalloc_missing_copy(void* out, const void* x, int64_t rows,
                                            int64_t hidden, uint64_t wait_limit_ns,
                                            ltxk_stream_t stream);

/* Human-readable name of an ltxk_status (static string, never NULL). */
LTXK_API const char* ltxk_status_string(int status);

/* cudaError_t value behind the calling thread's last LTXK_ERR_CUDA (0 if
 * none yet). */
LTXK_API int ltxk_last_cuda_error(void);

/* ---- launch plan (host-only introspection; no CUDA call) -------------- */

enum {
    LTXK_KERNEL_NONE = 0,       /* rows == 0: nothing to launch */
    LTXK_KERNEL_ROWS_VEC = 1,   /* 16-byte vectors, row in registers */
    LTXK_KERNEL_ROWS_ELEM = 2,  /* element-wise, two passes over the row */
    LTXK_KERNEL_ROWS_TMA = 3    /* one warp per row, rows streamed by bulk
                                   copies through a shared-memory ring */
};

enum {
    LTXK_OP_RMS_NORM = 0,
    LTXK_OP_RMS_NORM_ROPE = 1,
    LTXK_OP_RMS_NORM_ADALN = 2,
    LTXK_OP_ADD_RMS_NORM = 3
};

typedef struct {
    int kernel;          /* LTXK_KERNEL_* */
    int group_warps;     /* warps that share one row */
    int vec_per_lane;    /* 16-byte vectors each lane keeps in registers */
    int block_threads;   /* threads per CTA */
    int rows_per_cta;    /* rows a CTA works on at a time */
    int stages;          /* TMA ring: row buffers per warp (else 0) */
    int smem_bytes;      /* dynamic shared memory per CTA: the TMA ring, or AdaLN's
                            staged conditioning row (register kernel, 16-bit rows) */
} ltxk_plan;

/*
 * ltxk_plan_launch -- the kernel choice the entry points make, for the
 * given problem, under the current ltxk_set_path setting.  `vector_ok` says
 * whether every pointer is 16-byte aligned.  `mode` is ignored for
 * LTXK_OP_RMS_NORM.  Returns an ltxk_status (the same shape and mode checks
 * as the entry points).
 */
LTXK_API int ltxk_plan_launch(int op, int64_t rows, int64_t hidden, int head_dim,
                     int mode, int vector_ok, ltxk_plan* plan);

/* ltxk_plan_launch for rows of element type `dtype` (LTXK_DTYPE_*). */
LTXK_API int ltxk_plan_launch_dt(int op, int dtype, int64_t rows, int64_t hidden,
                                 int head_dim, int mode, int vector_ok, ltxk_plan* plan);

#ifdef __cplusplus
}
#endif

#endif /* LTXK_H_ */
