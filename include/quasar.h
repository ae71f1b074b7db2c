/*
 * quasar.h -- C ABI of libquasar.so, the GB300 (sm_103a) W8A8 verification
 * path of Quasar quantized self-speculative decoding.
 *
 * Source of the method: "Quasar: Quantized Self-Speculative Acceleration for
 * Rapid Inference via Memory-Efficient Verification" (arXiv 2603.01399), in
 * its gist.science summaries.  Sections cited below are the summaries'
 * technical sections: pt §2 "Metodologia", zh §2 "方法论", ko §2 "방법론".
 *
 * Common conventions
 *  - Every pointer argument is DEVICE memory owned by the caller unless the
 *    comment says otherwise.  No call allocates device memory and none keeps
 *    per-call state.  The library image owns two fixed device objects, held
 *    by every GPU that loads it until the process exits: a 32-bit error word
 *    read by quasar_get_device_error(), and the QUASAR_NOALLOC_SCRATCH_BYTES
 *    array used only by quasar_w8a8_linear_noalloc().
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Host-side argument checks happen first; a call that
 *    fails them returns an error code and launches nothing.
 *  - Matrices are row-major.  "ld" arguments are row strides in elements.
 *  - Base pointers of BF16 / INT8 matrices must be 16-byte aligned and their
 *    row strides multiples of 16 bytes (TMA and 128-bit loads); fp32 / int32
 *    vectors must be 4-byte aligned.  Violations return
 *    QUASAR_ERR_UNSUPPORTED.
 *  - Inputs are finite by contract; NaN/Inf behaviour is unspecified.
 *  - Results are deterministic: integer work is exact and every floating
 *    point reduction has a fixed order.
 */
#ifndef QUASAR_H
#define QUASAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Binary-compatible with cudaStream_t. */
typedef struct CUstream_st* quasar_stream_t;

typedef enum {
  QUASAR_OK = 0,
  QUASAR_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad value   */
  QUASAR_ERR_UNSUPPORTED = 2,   /* alignment / shape outside the contract   */
  QUASAR_ERR_WORKSPACE = 3,     /* workspace missing or too small           */
  QUASAR_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed         */
  QUASAR_ERR_TIMEOUT = 5        /* a device-side bounded wait ran out        */
} quasar_status_t;

/* Static, NUL-terminated description of a status code (host only). */
const char* quasar_status_string(int status);

/* Library ABI version, (major << 16) | minor. */
int quasar_version(void);

/* Device-side error word.  Kernels never trap: a bounded wait that runs out
 * (an mbarrier that is never completed, see the kernels) records its site in
 * a device word and the kernel returns early.  This call synchronises
 * `stream`, reads and clears the word, and returns QUASAR_OK or
 * QUASAR_ERR_TIMEOUT (also QUASAR_ERR_CUDA if the synchronisation fails).
 * If `site` is non-NULL (HOST pointer) it receives the recorded site code.
 * After a timeout, any workspace in use must be zero-filled again. */
quasar_status_t quasar_get_device_error(quasar_stream_t stream, uint32_t* site);

/* Self-test of the bounded waits (this library's failure handling; the pages
 * have no counterpart): launches one CTA whose thread waits on an mbarrier
 * that nothing completes.  The wait runs out after `limit_ns` (1 us .. 10 s),
 * records site code 12 in the device error word and the kernel returns; the
 * context stays usable and quasar_get_device_error reports
 * QUASAR_ERR_TIMEOUT.  Returns QUASAR_ERR_INVALID_ARG for a limit out of
 * range, else the launch status. */
quasar_status_t quasar_selftest_wait_timeout(uint64_t limit_ns, quasar_stream_t stream);

/* Tensor-pipe rate probe (a measurement utility; the pages have no
 * counterpart).  Runs one CTA per SM that issues `iters` groups of four MMAs
 * of one form and records, in `out` (DEVICE, >= 4 * SM-count 64-bit slots,
 * caller-owned, overwritten), per CTA b: out[4b] = clock64 cycles of the MMA
 * loop (0 if its bounded wait ran out), out[4b+1] = MMAs issued, out[4b+2] =
 * tcgen05.st instructions of the store traffic (form 2), out[4b+3] = cycles
 * that traffic ran.  Forms: 0 = tcgen05.mma kind::f16 M = 128, N = n, K = 16,
 * A in TMEM and B in shared memory; 1 = the same with A in shared memory;
 * 2 = form 0 while 16 warps store into another TMEM region (the W8A8 tcgen05
 * kernel's converter traffic); 3 = mma.sync m16n8k16 fp16 -> fp32 from
 * registers, 16 warps (n ignored); 4 / 5 = form 0 with each group's K steps
 * spread over 2 / 4 independent accumulators (n <= 128 / 64); 6 = form 1
 * with M = 64; 7 = tcgen05.mma.cta_group::2 kind::f16 over a cluster of two
 * CTAs on two SMs, M = 256 (128 A rows in each CTA's TMEM), N = n (n / 2 B
 * rows in each CTA's shared memory), issued by the even CTA, which records
 * the counts (n <= 224; out[4b+2] = the TMEM address CTA b's paired
 * allocation returned); 8 = form 7 with A in shared memory.  n: 16 .. 256,
 * a multiple of 16 (forms other than 3); 1 <= iters <= 2^20.  Asynchronous
 * on `stream`; returns
 * QUASAR_ERR_INVALID_ARG / QUASAR_ERR_UNSUPPORTED for bad arguments. */
quasar_status_t quasar_probe_tensor_rate(int form, int n, int iters, unsigned long long* out,
                                         int out_slots, quasar_stream_t stream);

/* Bound for the device-side waits, in nanoseconds (default 2e9 = 2 s).
 * Host-side setting applied to the next launches; 0 restores the default. */
quasar_status_t quasar_set_wait_limit_ns(uint64_t ns);

/* ------------------------------------------------------------------------
 * A0  Offline calibration of the smoothing vector.
 *
 * zh §2: the smoothing factor s is calibrated offline so that
 * Y = (W·diag(s)^-1)·(diag(s)·X); s multiplies the activations and divides
 * the weights.  Computed here as
 *   smooth[k] = max_n|W[n][k]|^(1-alpha) / max_m|Xcal[m][k]|^alpha
 * (SmoothQuant's migration factor inverted, so outlier activation channels
 * shrink), in fp64 and rounded once to fp32; smooth[k] = 1 when either
 * maximum is 0.  alpha == 0.5 uses IEEE sqrt and division (correctly
 * rounded, bit-reproducible); other alpha in (0,1) use pow().
 *
 *   Xcal    [Mcal][ldx] BF16 calibration activations, Mcal >= 1
 *   W       [N][ldw]    BF16 weights (all output rows that share this input,
 *                       e.g. fused q/k/v), N >= 1, K >= 1
 *   smooth  [K] fp32 output
 *   workspace: >= quasar_calibrate_workspace_size(K) bytes, any contents;
 *              the call clears what it uses.
 * ------------------------------------------------------------------------ */
size_t quasar_calibrate_workspace_size(int K);
quasar_status_t quasar_calibrate_smooth(const void* Xcal_bf16, int Mcal, int ldx,
                                        const void* W_bf16, int N, int ldw, int K,
                                        float alpha, float* smooth,
                                        void* workspace, size_t ws_bytes,
                                        quasar_stream_t stream);

/* ------------------------------------------------------------------------
 * A1  Offline weight packing (fold diag(smooth)^-1, per-channel INT8).
 *
 * pt §2 step 1 / zh §2 / ko §2: weights are smoothed and quantized to INT8
 * offline.  Per output channel n, in fp32 with IEEE rounding:
 *   w'[k]  = float(W[n][k]) / smooth[k]
 *   a      = max_k |w'[k]|
 *   sw[n]  = a / 127                 (0 if a == 0)
 *   Wq[n][k] = clamp(rne(w'[k] * (127 / a)), -127, 127)   (0 if a == 0)
 *
 * Packed layout (what quasar_w8a8_linear streams): the codes are stored in
 * blocks of 128 rows x 128 K, block (tn, kb) at byte offset
 * (tn * KB + kb) * 16384 with KB = ceil(K/128), so each block is 16 KB of
 * contiguous memory.  Inside a block, row r (n = 128*tn + r) takes bytes
 * [128r, 128r + 128); its 16-byte chunk c (k = 128*kb + 16c .. +15) sits at
 * chunk position c ^ (r % 8).  Each byte holds the code plus 128 (the code
 * with its sign bit flipped), so widening it needs no sign fix-up.  Rows
 * n >= N and columns k >= K of the last tiles hold code 0 (byte 0x80).
 * Size: quasar_packed_weight_bytes(N, K).
 *
 *   W      [N][ldw] BF16, ldw >= K, ldw % 8 == 0
 *   smooth [K] fp32, nonzero
 *   Wp     packed INT8 output (K % 16 == 0)
 *   sw     [N] fp32 output
 * ------------------------------------------------------------------------ */
size_t quasar_packed_weight_bytes(int N, int K);
quasar_status_t quasar_pack_weights(const void* W_bf16, int ldw, const float* smooth,
                                    int N, int K, int8_t* Wp, float* sw,
                                    quasar_stream_t stream);

/* Relayout row-major INT8 codes Wq [N][K] (K % 16 == 0) into the packed
 * layout above, for callers that quantized their weights themselves. */
quasar_status_t quasar_tile_weights(const int8_t* Wq, int N, int K, int8_t* Wp,
                                    quasar_stream_t stream);

/* ------------------------------------------------------------------------
 * A2  Online activation smoothing + per-token INT8 quantization.
 *
 * pt §2 step 2 / zh §2: during verification the BF16 input activations are
 * smoothed and quantized on the fly.  Per token m, in fp32:
 *   x'[k] = float(X[m][k]) * smooth[k]
 *   a     = max_k |x'[k]|
 *   sa[m] = a / 127                  (0 if a == 0)
 *   Xq[m][k] = clamp(rne(x'[k] * (127 / a)), -127, 127)   (0 if a == 0)
 *
 *   X      [M][ldx] BF16, ldx >= K, ldx % 8 == 0; M >= 0 (M == 0: no-op)
 *   smooth [K] fp32
 *   Xq     [M][K] INT8 output (K % 16 == 0)
 *   sa     [M] fp32 output
 * ------------------------------------------------------------------------ */
quasar_status_t quasar_smooth_quant_act(const void* X_bf16, int ldx, const float* smooth,
                                        int M, int K, int8_t* Xq, float* sa,
                                        quasar_stream_t stream);

/* ------------------------------------------------------------------------
 * A2 for qkv and gate_up: RMSNorm, then smooth + quantize, in one launch.
 *
 * pt §2 step 2 / zh §2: the BF16 input of a verify linear is smoothed and
 * quantized on the fly; here that input is the RMSNorm of the residual
 * stream and is formed on the way in.  Per token m, with K values:
 *   ss = sum_k float(X[m][k])^2         (each square exact in fp64; fp64 sum)
 *   r  = fp32_rn( 1 / sqrt(ss / K + eps) )   (fp64, IEEE division and sqrt)
 *   t[k] = bf16_rne(float(X[m][k]) * r),  h[k] = bf16_rne(float(t[k]) * gamma[k])
 *   then exactly quasar_smooth_quant_act on the row h.
 * The sum is taken in the kernel's own order, which can move ss by a few
 * fp64 ulps from the correctly rounded sum; r (and so the row's codes) can
 * differ from a correctly rounded evaluation only when 1 / sqrt(ss/K + eps)
 * lies within 2^-38 (relative) of an fp32 rounding midpoint.
 *
 *   X      [M][ldx] BF16, ldx >= K, ldx % 8 == 0, 16-byte aligned; M >= 0
 *   gamma  [K] BF16 (the norm's weight), 16-byte aligned
 *   eps    > 0 and finite (1e-6 for Qwen3)
 *   smooth [K] fp32 (the linear's smoothing vector), 16-byte aligned
 *   Xq     [M][K] INT8 output (K % 16 == 0, K <= 12288), sa [M] fp32 output
 *   Returns QUASAR_ERR_UNSUPPORTED for K % 16 != 0, K > 12288, ldx < K,
 *   ldx % 8 != 0 or a misaligned pointer; QUASAR_ERR_INVALID_ARG for K <= 0,
 *   eps <= 0 or not finite, or a null pointer.
 * ------------------------------------------------------------------------ */
quasar_status_t quasar_rmsnorm_smooth_quant(const void* X_bf16, int ldx, const void* gamma_bf16,
                                            float eps, const float* smooth, int M, int K,
                                            int8_t* Xq, float* sa, quasar_stream_t stream);

/* ------------------------------------------------------------------------
 * A2 for the MLP block's down projection: SiLU(gate) * up, then smooth +
 * quantize, in one launch.
 *
 * zh §2 / pt §2: the verifier dequantizes to BF16 ahead of the nonlinear
 * layers; the MLP's down linear then smooths and quantizes its input like any
 * other.  Per token m and k < I, in fp32:
 *   g = float(GU[m][k]), u = float(GU[m][I + k])   (gate half, then up half)
 *   h[k]  = bf16_rne( (g / (1 + exp(-g))) * u )     (one rounding to BF16)
 *   then exactly quasar_smooth_quant_act on the row h (x' = float(h) * smooth).
 * exp is a fixed fp32 algorithm so that the codes are a fixed function of the
 * inputs: Cody and Waite's reduction t = n ln2 + r (ln2 as a 15-bit head
 * 0x3F317200 plus a tail 0x35BFBE8E, n = rint(t * 0x3FB8AA3B)), the degree-7
 * Taylor polynomial of e^r by Horner with fp32 coefficients 1/k!, times 2^n,
 * every step one correctly rounded fp32 operation, the argument -g clamped
 * to [-87, 88]; it is within 2 ulp of e^t.
 *
 *   GU     [M][ldgu] BF16 (the gate_up linear's output: gate in columns
 *          0..I-1, up in I..2I-1), ldgu >= 2 I, ldgu % 8 == 0, 16-byte
 *          aligned; M >= 0 (M == 0: no-op)
 *   smooth [I] fp32 (down's smoothing vector), 16-byte aligned
 *   Xq     [M][I] INT8 output (I % 16 == 0), sa [M] fp32 output
 *   Returns QUASAR_ERR_UNSUPPORTED for I % 16 != 0, ldgu < 2 I or
 *   ldgu % 8 != 0, QUASAR_ERR_INVALID_ARG for I <= 0, I > 2^29 or a null
 *   pointer.  Feed Xq, sa to quasar_w8a8_linear with down's packed weights.
 * ------------------------------------------------------------------------ */
quasar_status_t quasar_silu_mul_smooth_quant(const void* GU_bf16, int ldgu, const float* smooth,
                                             int M, int I, int8_t* Xq, float* sa,
                                             quasar_stream_t stream);

/* ------------------------------------------------------------------------
 * A3 + A4  W8A8 linear: exact INT8 GEMM with fused BF16 dequant epilogue.
 *
 * pt §2 steps 3-4 / ko §2: the matmul runs on INT8 operands and the result
 * is dequantized back to BF16 before the nonlinear layers:
 *   acc[m][n] = sum_k Xq[m][k] * Wq[n][k]          (exact, int32)
 *   Y[m][n]   = bf16_rne((float(acc[m][n]) * sa[m]) * sw[n])
 *
 *   Xq [M][K] INT8 row-major, sa [M] fp32 (from quasar_smooth_quant_act)
 *   Wp packed INT8 weights, sw [N] fp32 (from quasar_pack_weights or
 *      quasar_tile_weights)
 *   Y  [M][ldy] BF16 output, ldy >= N, ldy % 8 == 0
 *   Sizes: M >= 0 (0 = no-op), 16 <= K <= 131072 with K % 16 == 0 (the int32
 *   accumulator cannot overflow: 127*127*131072 < 2^31), N >= 8 with
 *   N % 8 == 0.  Tuned for M <= 256 (verification passes); larger M works.
 *   Two kernels serve it: the register-path kernel for M <= 24, and for
 *   M <= 32 when N <= 8192; the tcgen05 kernel otherwise.
 *   The kernel is launched with programmatic dependent launch: it may start
 *   streaming Wp before the previous kernel on `stream` has finished, and it
 *   reads Xq / sa and writes Y and the workspace only after that kernel's
 *   writes are visible.
 *   workspace: >= quasar_w8a8_linear_workspace_size(M, N, K) bytes of device
 *   memory whose first quasar_w8a8_linear_workspace_zeroed_bytes(M, N, K)
 *   bytes (split-K counters and, on the tcgen05 kernel, int32 partial
 *   sums) are ZERO when the call starts; the rest may hold anything.  The call leaves
 *   all quasar_w8a8_linear_workspace_size(M, N, K) bytes zero-filled again
 *   when it completes without a device error, so one zero-filled workspace
 *   can serve every linear on a stream (but see the one-call entry below,
 *   which leaves scratch behind).  Calls that share a workspace must not run
 *   concurrently.  After QUASAR_ERR_TIMEOUT from quasar_get_device_error the
 *   workspace must be zero-filled again.
 * ------------------------------------------------------------------------ */
size_t quasar_w8a8_linear_workspace_size(int M, int N, int K);
size_t quasar_w8a8_linear_workspace_zeroed_bytes(int M, int N, int K);
quasar_status_t quasar_w8a8_linear(const int8_t* Xq, const float* sa,
                                   const int8_t* Wp, const float* sw,
                                   int M, int N, int K,
                                   void* Y_bf16, int ldy,
                                   void* workspace, size_t ws_bytes,
                                   quasar_stream_t stream);

/* ------------------------------------------------------------------------
 * W4A8 variant (NEXT-4; the pages' future ultra-low-bit verifier, as a
 * kernel variant only -- no accuracy claim).
 *
 * pt §2 step 1 with 4-bit codes: per output channel n, in fp32 as A1,
 *   w' = float(W[n][k]) / smooth[k],  a = max_k |w'|,  sw[n] = a / 7,
 *   Wq4[n][k] = clamp(rne(w' * (7 / a)), -7, 7)        (0 if a == 0)
 * and then the A3 + A4 linear with the same exact integer sums and the same
 * epilogue: Y = bf16_rne((float(acc) * sa[m]) * sw[n]).
 *
 * Packed 4-bit layout: blocks of 128 rows x 128 K, block (tn, kb) at byte
 * offset (tn * KB + kb) * 8192; row r (n = 128 tn + r) takes bytes
 * [64 r, 64 r + 64); its 16-byte chunk c (k = 128 kb + 32 c .. +31) sits
 * at chunk position c ^ ((r >> 1) & 3).  Byte j = 4 w + b of a chunk holds
 * code(k0 + 4 w + b) + 8 in its low nibble and code(k0 + 16 + 4 w + b) + 8
 * in its high nibble (k0 = 128 kb + 32 c).  Rows n >= N and columns k >= K
 * hold code 0 (nibble 8).  Size: quasar_packed_weight_bytes_w4(N, K).
 *
 *   quasar_pack_weights_w4: W [N][ldw] BF16 (ldw >= K, ldw % 8 == 0),
 *     smooth [K] fp32 -> Wp4 (K % 16 == 0), sw [N] fp32.
 *   quasar_tile_weights_w4: row-major codes [N][K] in [-8, 7] -> Wp4.
 *   quasar_w4a8_linear: as quasar_w8a8_linear with Wp4 for Wp, same
 *     argument rules, limits and error codes, any M >= 0 (the register-path
 *     kernel for a few tokens, the tcgen05 kernel above, both reading the
 *     4-bit blocks directly); workspace: quasar_w8a8_linear_workspace_size
 *     (M, N, K) bytes under the same contract (the first
 *     quasar_w8a8_linear_workspace_zeroed_bytes(M, N, K) zero on entry and
 *     left zero).
 * ------------------------------------------------------------------------ */
size_t quasar_packed_weight_bytes_w4(int N, int K);
quasar_status_t quasar_pack_weights_w4(const void* W_bf16, int ldw, const float* smooth,
                                       int N, int K, int8_t* Wp4, float* sw,
                                       quasar_stream_t stream);
quasar_status_t quasar_tile_weights_w4(const int8_t* Wq4, int N, int K, int8_t* Wp4,
                                       quasar_stream_t stream);
quasar_status_t quasar_w4a8_linear(const int8_t* Xq, const float* sa,
                                   const int8_t* Wp4, const float* sw,
                                   int M, int N, int K,
                                   void* Y_bf16, int ldy,
                                   void* workspace, size_t ws_bytes,
                                   quasar_stream_t stream);

/* A2 + A3 + A4 in one call: smooth + quantize the BF16 activations and run
 * the W8A8 linear on the codes.
 *   Y[m][n] is bit-identical to quasar_smooth_quant_act(X, smooth) followed by
 *   quasar_w8a8_linear on its outputs (same codes, same sa, same epilogue),
 *   with the codes and scales kept in the workspace instead of caller
 *   buffers.  On the register-path kernel it is one launch: its CTAs quantize
 *   the token rows themselves (row r by CTA r mod grid, with the quantizer's
 *   arithmetic) and publish them to the others through a counter in the
 *   workspace's zeroed prefix before any CTA reads a code; this needs every
 *   CTA of the launch resident at once, which the library's grid sizing
 *   gives on an otherwise idle device (where it cannot, the quantizer runs
 *   as a launch of its own first).  A wait for the rows that runs out is
 *   reported like any other bounded wait (site 11).  On the tcgen05 kernel
 *   it is the two launches (and the quantizer also writes the codes as fp16
 *   in the workspace for tiles of >= 64 tokens: the linear's token operand).
 *   X [M][ldx] BF16 (ldx >= K, ldx % 8 == 0, 16-byte aligned), smooth [K]
 *   fp32 (16-byte aligned), Wp / sw / Y / sizes as for quasar_w8a8_linear.
 *   workspace: >= quasar_w8a8_linear_fused_workspace_size(M, N, K) bytes;
 *   its first quasar_w8a8_linear_workspace_zeroed_bytes(M, N, K) bytes
 *   must be zero on entry as for quasar_w8a8_linear, and its first
 *   quasar_w8a8_linear_workspace_size(M, N, K) bytes are zero again on
 *   return; the bytes after those hold the codes and scales afterwards
 *   (scratch).  A later call on the same buffer whose zero prefix reaches
 *   into that scratch needs it cleared first (or a buffer of its own).
 * ------------------------------------------------------------------------ */
size_t quasar_w8a8_linear_fused_workspace_size(int M, int N, int K);
quasar_status_t quasar_w8a8_linear_fused(const void* X_bf16, int ldx, const float* smooth,
                                         const int8_t* Wp, const float* sw,
                                         int M, int N, int K,
                                         void* Y_bf16, int ldy,
                                         void* workspace, size_t ws_bytes,
                                         quasar_stream_t stream);

/* A3 alone: the exact int32 accumulator acc[M][N] (row stride N) instead of
 * Y, same kernel and workspace contract.  For checking and for callers
 * with their own epilogue. */
quasar_status_t quasar_int8_gemm_s32(const int8_t* Xq, const int8_t* Wp,
                                     int M, int N, int K, int32_t* acc,
                                     void* workspace, size_t ws_bytes,
                                     quasar_stream_t stream);

/* The same W8A8 linear for callers that cannot hand the library a
 * workspace: code hosted inside another runtime or plugin interface that
 * owns every device buffer and offers no scratch, or serving loops that
 * forbid device allocation once they are running.  (This entry point is a
 * library convenience; the paper has no counterpart.)  It allocates nothing:
 * its split-K scratch is one fixed array of QUASAR_NOALLOC_SCRATCH_BYTES in
 * the library's device image, which every GPU that loads the library keeps
 * until the process exits.
 *   - Arguments, outputs and results are those of quasar_w8a8_linear.
 *   - Returns QUASAR_ERR_WORKSPACE when quasar_w8a8_linear_workspace_size(M,
 *     N, K) exceeds QUASAR_NOALLOC_SCRATCH_BYTES (8 MiB: e.g. M x N up to
 *     about two million output elements on the tcgen05 kernel, and every
 *     register-path shape, whose partial sums need at most 5.3 MB).
 *   - The first call on a device looks up the array's device address with
 *     that device current; make that first call before any stream capture.
 *   - Each call clears the part of the array it uses on `stream` before the
 *     kernel runs, so it does not depend on what a previous call left.
 *   - All calls in the process share the one array: calls that may overlap
 *     on the GPU (different streams, or different host threads) race and
 *     must be serialized by the caller. */
#define QUASAR_NOALLOC_SCRATCH_BYTES (8u << 20)
quasar_status_t quasar_w8a8_linear_noalloc(const int8_t* Xq, const float* sa,
                                           const int8_t* Wp, const float* sw,
                                           int M, int N, int K,
                                           void* Y_bf16, int ldy,
                                           quasar_stream_t stream);

/* ------------------------------------------------------------------------
 * A5  Verification: accepted prefix length per sequence.
 *
 * zh §2 / ko §2: drafted tokens are checked against the dequantized,
 * high-precision logits with rejection sampling; pt §4: greedy (T = 0)
 * acceptance length.  Row j of sequence b scores the position that draft
 * j fills; row D is the bonus position after the last draft.
 *   T == 0:  ok_j = (draft[b][j] == argmax_v logits[b][j][v]), the lowest
 *            index wins ties (values compared as BF16 numbers).
 *   T  > 0:  p_j = softmax(float(logits[b][j][:]) / T)[draft[b][j]] in fp32;
 *            ok_j = (u[b][j] < p_j).  The drafter is treated as
 *            deterministic (its proposal probability is 1).
 *   n_acc[b] = first j with !ok_j, or D.
 *   next_token[b] (optional, T == 0 only) = argmax of row n_acc[b]: the
 *   correction token on a rejection or the bonus token after D accepts.
 *
 *   logits [B][D+1][V] BF16, rows `ldl` elements apart (ldl >= V,
 *          ldl % 8 == 0), row (b, j) at logits + (b*(D+1) + j)*ldl
 *   draft  [B][D] int32, values in [0, V)
 *   u      [B][D] fp32 in [0,1); required iff T > 0, else may be NULL
 *   n_acc  [B] int32 output
 *   next_token [B] int32 output or NULL; must be NULL when T > 0
 *   Sizes: B >= 0 (0 = no-op), D >= 0, V >= 1.
 *   workspace: >= quasar_verify_accept_workspace_size(B, D, V) bytes,
 *   ZERO-FILLED before first use and left zero-filled by the call (same
 *   contract as quasar_w8a8_linear).
 * ------------------------------------------------------------------------ */
size_t quasar_verify_accept_workspace_size(int B, int D, int V);
quasar_status_t quasar_verify_accept(const void* logits_bf16, int ldl,
                                     const int32_t* draft, int B, int D, int V,
                                     float temperature, const float* u,
                                     int32_t* n_acc, int32_t* next_token,
                                     void* workspace, size_t ws_bytes,
                                     quasar_stream_t stream);

/* A5 with T > 0 and the lossless next token.
 *
 * zh §2 (lossless rejection sampling on the high-precision logits).  The
 * acceptance test is that of quasar_verify_accept for T > 0.  With the
 * deterministic drafter, the speculative-sampling correction at the first
 * rejected position j is a draw from norm(max(0, p_j - onehot(draft_j))),
 * i.e. p_j without the draft token, renormalised; after D acceptances the
 * bonus token is a draw from p_D.  next_token[b] is that draw by inverse
 * CDF: the smallest v whose cumulative weight exp(logit/T - max) exceeds
 * u_next[b] times the row's total (fp32; the draft token carries no
 * weight); a row with no weight left gives the lowest index other than the
 * draft.  Emitted tokens are then distributed as the target softmax
 * whatever the drafts are.
 *   temperature > 0 (finite); u [B][D] as above (may be NULL iff D == 0);
 *   u_next [B] fp32 in [0, 1); next_token [B] int32 output (both required);
 *   other arguments, sizes and the workspace as quasar_verify_accept.
 * ------------------------------------------------------------------------ */
quasar_status_t quasar_verify_sample(const void* logits_bf16, int ldl,
                                     const int32_t* draft, int B, int D, int V,
                                     float temperature, const float* u,
                                     const float* u_next,
                                     int32_t* n_acc, int32_t* next_token,
                                     void* workspace, size_t ws_bytes,
                                     quasar_stream_t stream);

/* ------------------------------------------------------------------------
 * BF16 lm_head weight packing (offline).
 *
 * The lm_head kernels stream the weight as contiguous 16 KB blocks, each
 * already in the layout the tensor cores read: 128 vocabulary rows x 64 K
 * values of BF16.  Block (t, kb) (t = vocabulary tile, kb = K block; KB =
 * ceil(K/64)) starts at byte (t*KB + kb) * 16384; inside it, row r (entry
 * v = 128t + r) occupies bytes r*128 .. r*128+127, and its 16-byte chunk c
 * (K values 64kb + 8c .. +7) sits at chunk position c ^ (r % 8).  Rows past
 * V and K values past K are zero.
 *   W   [V][ldw] BF16 row-major, ldw >= K, ldw % 8 == 0, 16-byte aligned
 *   K % 8 == 0; Wp: quasar_lm_head_packed_bytes(V, K) bytes, 16-byte aligned
 * ------------------------------------------------------------------------ */
size_t quasar_lm_head_packed_bytes(int V, int K);
quasar_status_t quasar_pack_lm_head(const void* W_bf16, int ldw, int V, int K,
                                    void* Wp, quasar_stream_t stream);

/* ------------------------------------------------------------------------
 * Fused BF16 lm_head + verification (the logits are never written).
 *
 * nl §2 / ko §2: the verifier's last matmul stays in BF16 and the drafts are
 * checked on its high-precision logits; zh §2: greedy or rejection
 * acceptance.  For token row c = b*(D+1) + j (j = D: the bonus position):
 *   l[c][v] = bf16_rne(fp32 sum_k H[c][k] * W[v][k])   (tensor cores, fp32
 *             accumulation in an unspecified order)
 * and then exactly the acceptance rule of quasar_verify_accept on l, with
 * the row reductions (max, lowest-index argmax, sum of exp((l - max)/T),
 * the draft's logit) taken inside the matmul's epilogue.
 *   H      [B*(D+1)][ldh] BF16 hidden states (final-norm output), row c as
 *          above; ldh >= K, ldh % 8 == 0; 16-byte aligned
 *   Wp     the lm_head weight W [V][K] packed by quasar_pack_lm_head
 *   K      hidden size, K % 8 == 0
 *   draft  [B][D] int32 in [0, V); u [B][D] fp32 in [0,1), required iff
 *          T > 0 and D > 0; n_acc [B] int32 output; next_token [B] int32
 *          (argmax of row n_acc) or NULL, and NULL when T > 0
 *   Sizes: B >= 0 (0 = no-op), D >= 0, V >= 1, B*(D+1) <= 512
 *          (QUASAR_ERR_UNSUPPORTED above).
 *   workspace: >= quasar_lm_head_verify_workspace_size(B, D, V) bytes,
 *   256-byte aligned, ZERO-FILLED before first use and left zero-filled by
 *   the call (same contract as quasar_w8a8_linear).
 * Two launches (the matmul with its epilogue, then one CTA per row merging
 * the per-tile records); asynchronous on `stream`.
 * ------------------------------------------------------------------------ */
size_t quasar_lm_head_verify_workspace_size(int B, int D, int V);
quasar_status_t quasar_lm_head_verify(const void* H_bf16, int ldh,
                                      const void* Wp, int K,
                                      const int32_t* draft, int B, int D, int V,
                                      float temperature, const float* u,
                                      int32_t* n_acc, int32_t* next_token,
                                      void* workspace, size_t ws_bytes,
                                      quasar_stream_t stream);

/* The fused lm_head + verification for T > 0 with the lossless next token:
 * the acceptance test of quasar_lm_head_verify at T > 0, then next_token[b]
 * drawn exactly as quasar_verify_sample draws it (inverse CDF on u_next[b]
 * over row n_acc's softmax without the rejected draft, or over the bonus
 * row after D acceptances).  The vocabulary tile holding the draw is found
 * from the per-tile records; its 128 logits are recomputed from Wp and H
 * (fp32 sums, one rounding to BF16) for the walk inside it.
 *   temperature > 0; u as above; u_next [B] fp32 in [0, 1); next_token [B]
 *   int32 output (both required); everything else as quasar_lm_head_verify.
 * ------------------------------------------------------------------------ */
quasar_status_t quasar_lm_head_verify_sample(const void* H_bf16, int ldh,
                                             const void* Wp, int K,
                                             const int32_t* draft, int B, int D, int V,
                                             float temperature, const float* u,
                                             const float* u_next,
                                             int32_t* n_acc, int32_t* next_token,
                                             void* workspace, size_t ws_bytes,
                                             quasar_stream_t stream);

/* The same BF16 lm_head kernel writing its logits instead:
 *   logits[m][v] = bf16_rne(fp32 sum_k H[m][k] * W[v][k]),
 *   logits [M][ldl] BF16 (ldl >= V), 2-byte aligned; 0 <= M <= 512;
 *   H, Wp, K as above.  No workspace.  For checking the matmul on its own
 *   and for callers that need the logits tensor.
 * ------------------------------------------------------------------------ */
quasar_status_t quasar_lm_head_logits(const void* H_bf16, int ldh,
                                      const void* Wp, int M, int V, int K,
                                      void* logits_bf16, long long ldl,
                                      quasar_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QUASAR_H */
