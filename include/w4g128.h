/*
 * w4g128 -- int4 weight-only, group-128 (int4-g128) weight-streaming GEMV for
 * one NVIDIA GB300 GPU (sm_103a).  Plain C ABI: host/device pointers, sizes
 * and a CUDA stream passed as void*.  No C++ exceptions cross it.
 *
 * The operation (Token Rush README: intro bullet "4.25 bits per weight" and
 * the "Quantization" section define the format; the "bandwidth ceiling"
 * paragraph and the progress table -- steps 3, 8-9, 13-14, 20, 28 -- define
 * the decode GEMV, its split-K form, the M-row speculative verify and the
 * lm_head row slice):
 *
 *     y[m][n] = bf16( sum_k x[m][k] * w[k][n] ),   w[k][n] = min[g][n] + q[k][n] * scale[g][n],
 *     g = k / 128,  q in 0..15,  1 <= M <= 16,
 *
 * with bf16 x, scale, min and y, fp32 accumulation and one final
 * round-to-nearest-even to bf16.  Results are accepted when
 * |y - y_exact| <= 4e-3 * sum_k |x[m][k] w[k][n]| + one bf16 ulp of y_exact.
 *
 * ---------------------------------------------------------------------------
 * CANONICAL INPUT FORMAT (what callers hand to w4g128_pack)
 *   codes  uint32 [K/8][N] row-major: code of row k = 8j + i of column n is in
 *          bits 4i..4i+3 of word (j, n).
 *   scales bf16   [K/128][N] row-major, mins bf16 [K/128][N] row-major.
 *   x      bf16   [M][K] row-major;  y  bf16 [M][N] row-major.
 *   Shapes: K % 128 == 0, N % 16 == 0, 128 <= K <= 65536, 16 <= N <= 2^24.
 *
 * PACKED LAYOUT (what the kernels stream; exactly 4.25 bits per weight)
 *   G = K/128 groups, T = N/16 column tiles of 16 columns, grouped into
 *   quads of 4 tiles (64 columns); quad q holds nt(q) = min(4, T - 4q) tiles.
 *   Each (tile t, group g) is a block of 1088 bytes.  Block (t, g), with
 *   q = t / 4 and i = t % 4, starts at byte
 *        q*G*4352 + g*nt(q)*1088 + i*1088,
 *   so one quad's blocks for one group are contiguous, a quad is one
 *   contiguous run over all groups, and the whole matrix is one sequential
 *   stream in (quad, group) order.  The columns of the first Q' quads are a
 *   contiguous byte prefix: a column slice of N' = 64*Q' columns (such as the
 *   first 131072 lm_head rows) is used in place by passing N'.
 *   Block bytes [0, 1024): codes.  Half h (0, 1) starts at 512*h; lane l
 *   (0..31) at +16*l; little-endian uint32 word j (0..3) at +4*j.  With
 *   r = l / 4, c = l % 4 and k0 = 128g + 64h + 16j, nibble p = 4b + 2a + e
 *   (bits 4p..4p+3) of that word holds the code of row k0 + 2c + 8a + b of
 *   column 16t + r + 8e.  (So one word is exactly the 16x16 weight operand
 *   fragment one lane holds for a 16x8x16 warp MMA, and nibbles p and p+4 are
 *   the two rows of one 32-bit operand register.)
 *   Block bytes [1024, 1088): 8 entries of 8 bytes; entry r holds the
 *   little-endian bf16 values scale, min of column 16t + r and scale, min of
 *   column 16t + r + 8, for group g.
 *
 * WORKSPACE
 *   Every compute call takes a caller-owned device workspace `ws` (16-byte
 *   aligned, size from the matching *_workspace_bytes query).  It holds the
 *   per-call activation package, the split-K partial sums, the arrival
 *   counters of the M = 1 fold and a status word.  Each call re-initialises
 *   what it needs: no zeroing is required, and the content after a call is
 *   unspecified except for the
 *   status word (w4g128_workspace_status).  A workspace must not be used by
 *   two calls that can run at the same time (e.g. on two streams).
 *
 * CONVENTIONS
 *   - All array pointers are device pointers owned by the caller; the library
 *     allocates nothing per call (the only device memory it holds is the
 *     fixed scratch array behind w4g128_gemv_noalloc).  packed, ws: 16-byte
 *     aligned; x, y, codes, scales, mins: 4-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Argument errors are returned before anything is
 *     launched.  Launch failures return W4G128_ERR_CUDA.
 *   - Output is bitwise deterministic for a given shape and M (independent of
 *     the grid size and of the SM count).
 *   - x and y must not overlap; y must not overlap packed or ws.
 *   - Finite inputs whose sums stay within fp32 range.  The kernels carry x
 *     as fp16 scaled by one power of two per (128-row group, row): every
 *     x within 2^29 of its group's largest magnitude is exact there, and
 *     every product x * code is exact in fp32.  When all weights of a column
 *     are zero (min = -q * scale exactly) the factorised sum leaves a
 *     rounding residual of order 2^-24 * 1024 * scale * sum|x| instead of 0.
 */
#ifndef W4G128_H
#define W4G128_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define W4G128_API __attribute__((visibility("default")))
#else
#define W4G128_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  W4G128_OK = 0,
  W4G128_ERR_INVALID_ARG = 1, /* null pointer, M outside 1..W4G128_MAX_M, count outside 1..W4G128_MAX_MATRICES */
  W4G128_ERR_SHAPE = 2,       /* K % 128, N % 16, or a size outside the limits above */
  W4G128_ERR_ALIGN = 3,       /* a pointer is not aligned as required */
  W4G128_ERR_WORKSPACE = 4,   /* ws_bytes smaller than the workspace query returns */
  W4G128_ERR_CUDA = 5,        /* a CUDA runtime call or a launch failed */
  W4G128_ERR_DEVICE = 6,      /* the current device is not compute capability 10.3 */
  W4G128_ERR_TIMEOUT = 7,     /* (status word only) a bounded device-side wait gave up */
  W4G128_ERR_INTERNAL = 8     /* (status word only) a kernel found its launch inconsistent and skipped its work */
} w4g128_status;

#define W4G128_MAX_M 16
#define W4G128_MAX_MATRICES 512

/* Raw bf16 bit pattern. */
typedef uint16_t w4g128_bf16;

/* Human-readable name of a status code (static string). */
W4G128_API const char* w4g128_status_string(int status);

/* Exact byte size of the packed form of a K x N matrix: K*N/2 + 4*(K/128)*N,
 * i.e. 4 bits per code plus one bf16 scale and one bf16 minimum per 128
 * weights, 4.25 bits per weight (Token Rush README, intro bullet "4.25 bits
 * per weight" and the "Quantization" section).  Returns 0 for an invalid
 * shape. */
W4G128_API size_t w4g128_packed_bytes(int K, int N);

/* Canonical -> packed layout (a bit permutation; bit-exact).  The format is
 * the pages' group-wise asymmetric int4 with one bf16 scale and minimum per
 * 128 weights (Token Rush README, "Quantization" section); the packed byte
 * order is this library's own (PACKED LAYOUT above).  codes, scales, mins and
 * packed are device pointers (caller-owned); packed must hold
 * w4g128_packed_bytes(K, N) bytes and is written in full, nothing past it.
 * Runs once per weight matrix, not per decode step.  Asynchronous on
 * `stream`; argument errors are returned before anything is launched. */
W4G128_API int w4g128_pack(const uint32_t* codes, const w4g128_bf16* scales, const w4g128_bf16* mins,
                           int K, int N, void* packed, void* stream);

/* Exact inverse of w4g128_pack (for round-trip checks and export): the
 * canonical codes, scales and mins of the "Quantization" section's format
 * (Token Rush README) back from the packed layout.  Device pointers, caller-
 * owned; same shapes and alignment as w4g128_pack.  Asynchronous on
 * `stream`. */
W4G128_API int w4g128_unpack(const void* packed, int K, int N, uint32_t* codes, w4g128_bf16* scales,
                             w4g128_bf16* mins, void* stream);

/* bf16 weights w[K][N] (row-major, device) -> the canonical format that
 * w4g128_pack takes: codes [K/8][N], scales and mins [K/128][N] (device,
 * caller-owned).  Token Rush README, "Quantization": 128 weights per bf16
 * scale and minimum; round-to-nearest (search = 0), or round-to-nearest with
 * the per-group range search that clips outliers (search = 1).  Per group of
 * 128 rows of one column, with lo / hi its smallest / largest weight, a
 * candidate p spans [p lo, p hi] in 15 steps: scale = bf16((p hi - p lo) /
 * 15), min = bf16(p lo), q = clamp(round_half_even((w - min) / scale), 0, 15)
 * (0 when scale = 0); search = 1 tries p = 1.00, 0.99, ..., 0.80 and keeps
 * the smallest sum of (w - (min + q scale))^2 over the group (the widest on
 * ties).  Every step is one fp32 operation rounded to nearest (no fused
 * multiply-add), so the result is bit-exact and deterministic.  Weights must
 * be finite with |w| < 2^126.  A one-time preprocessing call, not part of the
 * weight stream. */
W4G128_API int w4g128_quantize(const w4g128_bf16* w, int K, int N, int search, uint32_t* codes,
                               w4g128_bf16* scales, w4g128_bf16* mins, void* stream);

/* Workspace bytes needed by w4g128_gemm_verify(M, K, N) on the current
 * device (and by w4g128_gemv, M = 1): the activation packages, the split-K
 * partial sums (Token Rush README, progress table steps 8-9: the split-K
 * GEMV's partial sums), the fold counters and the status word.  The size
 * depends on the SM count of the current device.  Returns 0 for invalid
 * arguments or when the current device is not compute capability 10.3. */
W4G128_API size_t w4g128_workspace_bytes(int M, int K, int N);

/* y[1][N] = x[1][K] . dequant(W): the batch-1 decode GEMV (streamed by TMA
 * bulk copies, the dequantised weights fed to the warp MMA with the one x row
 * in every B column, split-K with a deterministic last-arriver reduction).
 * Bitwise identical to w4g128_gemm_verify at M = 1.  Token Rush README,
 * progress table steps 3 and 8-9. */
W4G128_API int w4g128_gemv(const void* packed, const w4g128_bf16* x, w4g128_bf16* y, int K, int N,
                           void* ws, size_t ws_bytes, void* stream);

/* y[M][N] = x[M][K] . dequant(W) for 1 <= M <= W4G128_MAX_M (16): the
 * speculative M-row verify step (one weight pass for M draft rows, on the
 * tensor cores via warp MMA; the pages draft 7 tokens, M = 9..16 serves longer
 * drafts with two 8-row MMA tiles per weight fragment).  Row m of the result
 * is bitwise identical to this call on row m alone (M = 1), for every M: a
 * verify pass reproduces exactly what the same arithmetic gives one token at
 * a time; w4g128_gemv is this call at M = 1.  Token Rush README, progress
 * table steps 13-14 and 28. */
W4G128_API int w4g128_gemm_verify(const void* packed, const w4g128_bf16* x, w4g128_bf16* y, int M, int K,
                                  int N, void* ws, size_t ws_bytes, void* stream);

/* One matrix of a multi-matrix weight stream. */
typedef struct {
  const void* packed;     /* packed weights (device) */
  const w4g128_bf16* x;   /* [M][K] activations (device) */
  w4g128_bf16* y;         /* [M][N] output (device) */
  int K;
  int N;
} w4g128_matrix;

/* Workspace bytes for w4g128_decode_step or w4g128_verify_step over these
 * matrices at this M (Token Rush README, progress table step 4 and the
 * "bandwidth ceiling" paragraph: one pass over every weight of a step); the
 * same parts as w4g128_workspace_bytes, for all matrices at once.  `mats`
 * is a host array; only K and N are read.  Returns 0 for invalid
 * arguments. */
W4G128_API size_t w4g128_decode_step_workspace_bytes(const w4g128_matrix* mats, int count, int M);

/* Streams every matrix of `mats` (a HOST array of `count` descriptors,
 * 1 <= count <= W4G128_MAX_MATRICES) in one persistent launch: y_i = x_i .
 * dequant(W_i) for each i, as a whole decode step reads every weight once
 * (Token Rush README, progress table step 4 and the "bandwidth ceiling"
 * paragraph).  Every M runs the warp-MMA kernel.
 * The split-K segments (512 rows) and their summation order depend only on
 * each matrix's shape, so every y_i is bitwise identical to what a separate
 * w4g128_gemv (M = 1) or w4g128_gemm_verify call returns, whatever the SM
 * count or the other matrices.  The descriptor array is read during the call
 * and may be reused afterwards.  The matrices' N may sum to at most 2^30
 * (W4G128_ERR_SHAPE beyond). */
W4G128_API int w4g128_decode_step(const w4g128_matrix* mats, int count, int M, void* ws, size_t ws_bytes,
                                  void* stream);

/* w4g128_decode_step for activations that live in host memory between
 * steps: copies x_bytes from x_host to x_dev, streams the matrices, then
 * copies y_bytes from y_dev to y_host -- three operations issued in that
 * order on `stream` by one call, so a step whose input arrives from and
 * whose output returns to the host costs one library call.  The pages keep
 * the token on the device for the whole step (Token Rush README, progress
 * table step 4: the whole decode step captured as one graph); this entry
 * serves callers whose activations cross the host boundary every step.
 * The descriptors' x must lie inside [x_dev, x_dev + x_bytes) and their y
 * inside [y_dev, y_dev + y_bytes) (device, caller-owned); x_host and y_host
 * are host buffers.  Pinned (device-mapped) buffers with 16-byte aligned
 * ends and sizes that are multiples of 16 are moved by two small kernels
 * that keep the step's kernels overlapping the previous call (a copy-engine
 * copy between kernels would not); other buffers by cudaMemcpyAsync (with
 * pageable memory the CUDA runtime may return only after staging them).
 * Do not change x_host before the call has run.  x_bytes / y_bytes may be
 * 0 (no move).  Returns what w4g128_decode_step
 * returns, or W4G128_ERR_CUDA if a copy could not be issued; argument
 * errors are returned before anything is issued. */
W4G128_API int w4g128_decode_step_host(const w4g128_matrix* mats, int count, int M, const void* x_host,
                                       void* x_dev, size_t x_bytes, void* y_host, const void* y_dev,
                                       size_t y_bytes, void* ws, size_t ws_bytes, void* stream);

/* The verify step over a list of matrices: row m of each y_i is bitwise
 * identical to w4g128_gemm_verify on matrix i and row m alone, so decoding
 * at M = 1 and verifying drafts at M > 1 give the same bits for the same
 * token (the exact speculative-decoding property; Token Rush README, progress
 * table step 28).  It computes exactly what w4g128_decode_step does (one
 * arithmetic serves every M); same arguments and workspace query. */
W4G128_API int w4g128_verify_step(const w4g128_matrix* mats, int count, int M, void* ws, size_t ws_bytes,
                                  void* stream);

/* The product folded into the residual add and RMS norm that follow it
 * (Token Rush README, progress table steps 8-9: the split-K partial sums are
 * added up in the norm rather than in a pass of their own).  The pages name
 * the norm only; this is the pre-norm transformer's residual update followed
 * by RMS normalisation (Zhang and Sennrich, 2019), per row m over the N
 * columns:
 *   h[m][n]   = bf16( residual[m][n] + (x . dequant(W))[m][n] )
 *   out[m][n] = bf16( gamma[n] h[m][n] / sqrt( mean_n h[m][n]^2 + eps ) )
 * The product is the one w4g128_gemm_verify computes, kept in fp32; the
 * residual is added to it in fp32 and h rounded once, so with residual = -0.0
 * h is bit for bit that call's y.  The norm reads the rounded h (the value the residual
 * stream keeps): mean_n h^2 is summed in fp32 in an order fixed by N alone,
 * and every step after it is one correctly rounded fp32 operation, so out is
 * deterministic.  The residual add happens where the split-K sums are
 * folded; one small kernel, launched behind the product's kernels, then
 * normalises the rows.  If the call's status word reports an error, out is
 * left unwritten.
 *   x [M][K], residual, h, out [M][N], gamma [N]: bf16, device, row-major,
 *   caller-owned; 1 <= M <= W4G128_MAX_M.  h may be the residual itself
 *   (updated in place); out must not overlap x, residual or h
 *   (W4G128_ERR_INVALID_ARG when it is one of them).  residual, gamma, h,
 *   out: 4-byte aligned.  eps: finite and >= 0.  verify: 0 or 1 (both
 *   name the one arithmetic every M uses).  ws as for
 *   w4g128_gemm_verify (w4g128_workspace_bytes(M, K, N) bytes). */
W4G128_API int w4g128_gemm_add_rmsnorm(const void* packed, const w4g128_bf16* x, const w4g128_bf16* residual,
                                       const w4g128_bf16* gamma, float eps, w4g128_bf16* h, w4g128_bf16* out,
                                       int M, int K, int N, int verify, void* ws, size_t ws_bytes,
                                       void* stream);

/* Size of the fixed device scratch array behind w4g128_gemv_noalloc (16 MiB). */
#define W4G128_NOALLOC_SCRATCH_BYTES (16u << 20)

/* The pages have no counterpart to this entry point; it is a convenience of
 * this library.  Same result as w4g128_gemv (the same kernels, bit for bit),
 * for callers that cannot give the library a workspace because they must not
 * allocate device memory: plugin hooks of another runtime that owns the
 * device memory budget, fixed-pool serving processes, and latency-critical
 * threads that must not call cudaMalloc/cudaFree (those calls can synchronise
 * the device).  It allocates no device memory: the workspace is a fixed
 * W4G128_NOALLOC_SCRATCH_BYTES array that every GPU loading the library holds
 * until the process exits.  Shapes whose workspace would exceed it (the
 * limit is reached near K*N = 2^31 weights; a 5120 x 248320 lm_head needs
 * 10 MB) return W4G128_ERR_WORKSPACE before anything is launched.  The first
 * call on each device loads the array's module and looks up its device
 * address (every call repeats the lookup, so a reset device is handled);
 * make that first call before any stream capture.  All calls share the one
 * array, so calls that can overlap on the GPU (other streams, other host
 * threads) race and corrupt each other; serialise them (calls in order on
 * one stream are fine).  The status word of the last call is read with
 * w4g128_noalloc_status. */
W4G128_API int w4g128_gemv_noalloc(const void* packed, const w4g128_bf16* x, w4g128_bf16* y, int K, int N,
                                   void* stream);

/* Reads the status word the last call on `ws` left (W4G128_OK, or
 * W4G128_ERR_TIMEOUT if a bounded device wait gave up).  Synchronises
 * `stream`. */
W4G128_API int w4g128_workspace_status(const void* ws, int* status_out, void* stream);

/* The status word the last w4g128_gemv_noalloc call on the current device
 * left in the library's scratch array (W4G128_OK, or W4G128_ERR_TIMEOUT if a
 * bounded device wait gave up, in which case that call's y is incomplete).
 * No counterpart in the pages, like the entry point it serves.  Synchronises
 * `stream`. */
W4G128_API int w4g128_noalloc_status(int* status_out, void* stream);

/* The schedule w4g128_decode_step (count matrices; count = 1 for
 * w4g128_gemv / w4g128_gemm_verify) takes for these shapes at M rows on the
 * current device, for diagnostics and tests; launches nothing and reads only
 * K, N and x of `mats` (a HOST array; x may be NULL, read as 16-byte
 * aligned).  No counterpart in the pages: it reports how this library lays
 * the weight stream over the SMs.  Writes min(n, W4G128_SCHEDULE_FIELDS)
 * values to out (host):
 *   [0] 1 when every streaming CTA builds its own activation packages
 *       (M = 1), 0 with the separate package kernel;
 *   [1] streaming CTAs;  [2] warps per streaming CTA;
 *   [3] second pass: 0 none, 1 boundary fold of quads split between CTAs
 *       (M = 1), 2 per-quad reduce, 3 per-warp reduce (M >= 2);
 *   [4] 1 when each quad is split over the two CTAs of a thread-block
 *       cluster and folded in the first one's shared memory, else 0;
 *   [5] ring slots per streaming warp;  [6] workspace bytes;
 *   [7] work items (quad, 512-row segment) of all matrices.
 * Returns W4G128_OK, W4G128_ERR_INVALID_ARG / W4G128_ERR_SHAPE for the
 * arguments w4g128_decode_step would reject, W4G128_ERR_DEVICE without an
 * sm_103 device. */
#define W4G128_SCHEDULE_FIELDS 8
W4G128_API int w4g128_schedule(const w4g128_matrix* mats, int count, int M, long long* out, int n);

/* Workspace bytes w4g128_selftest_wait needs. */
#define W4G128_SELFTEST_WS_BYTES 512u

/* Diagnostic of the bounded device-side waits; the pages have no
 * counterpart (no wait in this library's kernels can spin forever: each
 * gives up after a time limit and records W4G128_ERR_TIMEOUT in the status
 * word instead).  Launches one small kernel on `stream` that clears the
 * status word of `ws`, stores 1 (set_flag = 1) or 0 (set_flag = 0) in a flag
 * word of `ws`, and then waits with the library's bounded flag wait for the
 * flag to be nonzero, for at most limit_ns nanoseconds (1 .. 2e9).  With
 * set_flag = 0 nothing ever sets the flag: the wait runs out and
 * w4g128_workspace_status(ws) then reads W4G128_ERR_TIMEOUT; with
 * set_flag = 1 it reads W4G128_OK.  Either way the kernel returns on its own
 * and `ws` is usable by any later call (every call re-initialises what it
 * needs).  ws: device, 16-byte aligned, ws_bytes >= W4G128_SELFTEST_WS_BYTES.
 *
 * Every compute entry point of this header also honours the environment
 * variable W4G128_FAULT, read once per process, for tests of callers' error
 * handling: "launch" makes it return W4G128_ERR_CUDA and "workspace"
 * W4G128_ERR_WORKSPACE after argument validation, without touching the
 * device. */
W4G128_API int w4g128_selftest_wait(void* ws, size_t ws_bytes, unsigned long long limit_ns, int set_flag,
                                    void* stream);

#ifdef __cplusplus
}
#endif

#endif /* W4G128_H */
