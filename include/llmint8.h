/*
 * llmint8.h -- C ABI of the LLM.int8() mixed-precision decomposed matmul on one
 * NVIDIA B300 (sm_103a).
 *
 * The operation (Y = X.W, decomposed):
 *   A0  weights get one absmax scale per output column and int8 codes
 *       q = round(w * 127/absmax)            ("LLM.int8() paper walkthrough",
 *       section 2.1; "LLM.int8() quantization pitfalls guide", section 1)
 *   A1  a K-column of X holding any |x| > threshold is an outlier dimension
 *       (paper walkthrough, section 2.3; default threshold 6.0)
 *   A2  the other columns of X get one absmax scale per row and int8 codes;
 *       outlier columns get code 0            (paper walkthrough, 2.1 and 2.3)
 *   A3  C = Xq . Wq, exact integer accumulation
 *   A4  F = X[:, outliers] . W[outliers, :] in fp16 with fp32 accumulation
 *       (paper walkthrough, 2.3; pitfalls guide, 3.2)
 *   A5  Y = fp16( C * rowScaleX[i] * colScaleW[n] / 127^2 + F )
 *       (pitfalls guide, 3.3: dequantize the 8-bit result, then add)
 *
 * Code rule: scale_factor = fp32(127 / absmax); q = round-half-away-from-zero(
 * fp32(x * scale_factor)), clamped to [-127, 127]; absmax 0 gives code 0.
 * Scales are stored as the absmax values themselves (fp32).
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers to caller-owned memory; the library
 *     allocates nothing and keeps no pointer after the call returns.
 *   - fp16 arrays are IEEE binary16, passed as void*.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). All work is
 *     enqueued asynchronously on it; the call returns without synchronizing.
 *   - Argument errors are detected on the host before anything is enqueued and
 *     leave all buffers untouched.  LLMINT8_ECUDA means a CUDA runtime call or a
 *     kernel launch failed; work enqueued before the failure may have run.
 *   - Sizes: 1 <= M, 1 <= K <= 65536, 1 <= N (else LLMINT8_EINVAL; M = 0 is
 *     an empty problem and is rejected, not silently accepted); K and N must be
 *     multiples of 16 and all pointers 16-byte aligned (else LLMINT8_EALIGN).
 *   - Inputs must be finite; NaN or Inf inputs give unspecified codes and Y.
 *   - The device must be compute capability 10.3 (else LLMINT8_EUNSUPPORTED).
 */
#ifndef LLMINT8_H
#define LLMINT8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LLMINT8_OK = 0,
    LLMINT8_EINVAL = 1,       /* bad size, NULL pointer, NaN threshold, missing operand */
    LLMINT8_EALIGN = 2,       /* K or N not a multiple of 16, or a pointer not 16-byte aligned */
    LLMINT8_EWORKSPACE = 3,   /* workspace NULL or smaller than llmint8_workspace_bytes() */
    LLMINT8_ECUDA = 4,        /* a CUDA runtime call or kernel launch failed */
    LLMINT8_ETIMEOUT = 5,     /* a bounded device-side wait gave up (see llmint8_device_status) */
    LLMINT8_EUNSUPPORTED = 6  /* current device is not sm_103 */
} llmint8_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *llmint8_status_str(int status);

/* Largest M served by the decode (GEMV) path; larger M uses the tensor-core GEMM. */
#define LLMINT8_DECODE_MAX_M 16

/*
 * A0 -- quantize a weight matrix once, before any forward call.
 *
 *   W         in   fp16 [K, N] row-major (the retained fp16 weight; keep it: its
 *                  rows are gathered for outlier columns of X)
 *   Wq        out  int8 [N, K] row-major, i.e. K contiguous per output column:
 *                  Wq[n*K + k] = round-half-away(W[k,n] * fp32(127 / colScaleW[n]))
 *   colScaleW out  fp32 [N], colScaleW[n] = max_k |W[k, n]| over ALL K rows
 *
 * Source: paper walkthrough, section 2.1 (per-column weight scale); Lightning
 * Fabric 8-bit page, section 2.2 (one scale per output channel).
 */
llmint8_status llmint8_quantize_weight(const void *W, int K, int N, int8_t *Wq, float *colScaleW,
                                       void *stream);

/*
 * Bytes of device workspace llmint8_matmul* needs for this shape (16-byte
 * multiple).  For M > LLMINT8_DECODE_MAX_M it includes a per-call fp16 copy of
 * the weight codes (2*N*K bytes): sm_103a has no int8 tcgen05 MMA, so the
 * prefill path widens Wq into exact fp16 integers there, right before its
 * tensor-core GEMM (one bandwidth-bound kernel), and the persistent weight
 * storage stays Wq plus colScaleW (N*K + 4*N bytes).
 */
size_t llmint8_workspace_bytes(int M, int K, int N);

/*
 * A1..A5 -- Y = X.W, LLM.int8() decomposition with the given outlier threshold.
 *
 *   X          in   fp16 [M, K] row-major activations
 *   threshold  in   outlier test |x| > threshold (strict).  +INFINITY disables
 *                   the decomposition (pure vector-wise int8); 0 or a negative
 *                   value makes every nonzero column an outlier; NaN -> EINVAL.
 *   Wq, colScaleW   from llmint8_quantize_weight
 *   W16        in   the retained fp16 W [K, N]; may be NULL only if threshold is
 *                   +INFINITY
 *   Y          out  fp16 [M, N] row-major
 *   workspace  scratch device memory of at least llmint8_workspace_bytes(M,K,N)
 *              bytes; its contents on entry do not matter.  Two calls that share
 *              a workspace must be ordered (same stream or synchronized).
 *
 * Source: paper walkthrough, sections 2.1-2.3; pitfalls guide, sections 3.1-3.3.
 */
llmint8_status llmint8_matmul(const void *X, int M, int K, int N, float threshold,
                              const int8_t *Wq, const float *colScaleW,
                              const void *W16, void *Y, void *workspace, size_t workspace_bytes,
                              void *stream);

/*
 * llmint8_matmul between host buffers: enqueues on `stream` the copy of X_host
 * into the device buffer X, the same kernels as llmint8_matmul, and the copy of
 * Y into Y_host, then returns (asynchronous: synchronize the stream before
 * reading Y_host).  For callers whose activations and results live in host
 * memory; one call instead of three.
 *
 *   X_host  in   host fp16 [M, K] (page-locked memory keeps the copies
 *                asynchronous; pageable memory works but the copies then
 *                block the calling thread)
 *   X       out  device fp16 [M, K] staging buffer (receives X_host)
 *   Y       out  device fp16 [M, N]
 *   Y_host  out  host fp16 [M, N]
 *   other arguments as llmint8_matmul
 *
 * Errors as llmint8_matmul (all checked before the first copy is enqueued);
 * EINVAL also for a NULL X_host, Y_host or Y; ECUDA if a copy cannot be enqueued.
 */
llmint8_status llmint8_matmul_host(const void *X_host, void *X, int M, int K, int N, float threshold,
                                   const int8_t *Wq, const float *colScaleW,
                                   const void *W16, void *Y, void *Y_host, void *workspace,
                                   size_t workspace_bytes, void *stream);

/*
 * bfloat16 forms: the same steps on bf16 W, X and Y (all other arguments as the
 * fp16 entry points).  The codes, scales, outlier test and the int32 product are
 * computed from the fp32 values of the bf16 inputs exactly as from fp16 ones;
 * the outlier slice multiplies bf16 X and W values with fp32 accumulation and Y
 * is rounded to bf16 (nearest even).
 * llmint8_matmul_i32_bf16 writes the int32 accumulator C, as llmint8_matmul_i32.
 */
llmint8_status llmint8_quantize_weight_bf16(const void *W, int K, int N, int8_t *Wq, float *colScaleW,
                                            void *stream);
llmint8_status llmint8_matmul_bf16(const void *X, int M, int K, int N, float threshold,
                                   const int8_t *Wq, const float *colScaleW,
                                   const void *W16, void *Y, void *workspace, size_t workspace_bytes,
                                   void *stream);
llmint8_status llmint8_matmul_i32_bf16(const void *X, int M, int K, int N, float threshold,
                                       const int8_t *Wq, const float *colScaleW,
                                       int32_t *C, void *workspace, size_t workspace_bytes, void *stream);

/*
 * llmint8_matmul without a full fp16 copy of W (int8 weight storage only).  The
 * outlier slice (A4) needs row k of W for every outlier column k of X: it is
 * W16c[row_map[k], :] when 0 <= row_map[k] < w16_rows (rows the caller chose to
 * keep in fp16, e.g. the columns that were outliers on calibration data), and
 * otherwise the dequantized codes, w_hat[k, n] = fp16(fp32(Wq[n, k]) *
 * fp32(colScaleW[n] / 127)) with each step rounded to nearest even.  The int8
 * part (A3) and the merge (A5) are those of llmint8_matmul; with every row kept
 * the result equals llmint8_matmul's.  Memory: w16_rows * N * 2 + K * 4 bytes
 * instead of K * N * 2 for the fp16 copy.
 *
 *   W16c       in   fp16 [w16_rows, N] kept rows (from llmint8_pack_w16_rows);
 *                   may be NULL when w16_rows = 0
 *   row_map    in   int32 [K] device array, or NULL when no row is kept
 *   w16_rows   in   number of kept rows (>= 0); map entries >= w16_rows count as
 *                   not kept
 *   other arguments as llmint8_matmul (without W16)
 *
 * Errors as llmint8_matmul; EINVAL also for w16_rows < 0, or w16_rows > 0 with a
 * NULL W16c or row_map; EALIGN for a W16c that is not 16-byte aligned.
 * Source: paper walkthrough, section 2.3 (the outlier slice in fp16); pitfalls
 * guide, section 1 (codes dequantized by their scale); Lightning Fabric 8-bit
 * page, section 2.2 (one scale per output column).
 */
llmint8_status llmint8_matmul_w8(const void *X, int M, int K, int N, float threshold,
                                 const int8_t *Wq, const float *colScaleW,
                                 const void *W16c, const int32_t *row_map, int w16_rows, void *Y,
                                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * Builds the kept rows for llmint8_matmul_w8 from a full fp16 W [K, N] (once, at
 * load time; the full copy can be freed afterwards): row_map[k] = -1 for every
 * k, then for each r < w16_rows, W16c[r, :] = W16[rows[r], :] and
 * row_map[rows[r]] = r.  A listed row outside [0, K) gets a zero row in W16c and
 * no map entry.
 *
 *   W16        in   fp16 [K, N] device
 *   rows       in   int32 [w16_rows] device, the rows to keep (may be NULL when
 *                   w16_rows = 0)
 *   W16c       out  fp16 [w16_rows, N] device (may be NULL when w16_rows = 0)
 *   row_map    out  int32 [K] device
 *
 * Errors: EINVAL for a NULL W16 or row_map, K or N <= 0, K > 65536, w16_rows < 0,
 * or w16_rows > 0 with a NULL rows or W16c; EALIGN if N is not a multiple of 16
 * or W16 or W16c is not 16-byte aligned; ECUDA if a launch fails.  Asynchronous
 * on `stream`.
 */
llmint8_status llmint8_pack_w16_rows(const void *W16, int K, int N, const int32_t *rows, int w16_rows,
                                     void *W16c, int32_t *row_map, void *stream);

/*
 * Plain vector-wise int8 variant: llmint8_matmul with threshold = +INFINITY and
 * no fp16 weight.  Row scales run over all K columns; Y = fp16(C * sx * sw / 127^2).
 * Source: pitfalls guide, section 1 (plain absmax int8, no outlier handling).
 */
llmint8_status llmint8_matmul_int8(const void *X, int M, int K, int N, const int8_t *Wq,
                                   const float *colScaleW, void *Y,
                                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * The two halves of llmint8_matmul, for callers that schedule them apart (and
 * for timing the GEMM stage alone).  llmint8_matmul(args) enqueues exactly
 * llmint8_xpass(X, M, K, N, threshold, workspace) followed by
 * llmint8_gemm(args) on the same stream.
 *
 * llmint8_xpass -- steps A1 and A2 (paper walkthrough, sections 2.1 and 2.3):
 *   reads X fp16 [M, K]; writes into `workspace` the outlier column set, the row
 *   scales, the codes (see llmint8_workspace_layout) and, for M > 16, the
 *   gathered outlier columns of X.  Same argument rules as llmint8_matmul.
 *
 * llmint8_gemm -- steps A3, A4 and A5 (pitfalls guide, sections 3.2-3.3):
 *   consumes a workspace that an llmint8_xpass with the same X, M, K, N and
 *   threshold filled earlier on the same stream (undefined otherwise); X is read
 *   again for the outlier values.  For M > 16 it first widens Wq into the
 *   workspace's fp16 code scratch.  Writes Y fp16 [M, N].
 */
llmint8_status llmint8_xpass(const void *X, int M, int K, int N, float threshold, void *workspace,
                             size_t workspace_bytes, void *stream);
llmint8_status llmint8_gemm(const void *X, int M, int K, int N, float threshold, const int8_t *Wq,
                            const float *colScaleW, const void *W16, void *Y,
                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * A1 + A2 into caller buffers (the pages' quantization of the activations,
 * paper walkthrough sections 2.1 and 2.3; pitfalls guide, section 1):
 *   Xq         out  int8 [M, K] row-major codes, outlier columns 0
 *   rowScaleX  out  fp32 [M], absmax of each row over the non-outlier columns
 *   workspace  scratch of at least llmint8_workspace_bytes(M, K, 16) bytes; it
 *              receives the outlier column set (llmint8_read_outliers)
 * Same rules as llmint8_matmul for X, M, K and threshold; EINVAL for a NULL Xq
 * or rowScaleX, EALIGN for one that is not 16-byte aligned.  Asynchronous.
 */
llmint8_status llmint8_quantize_x(const void *X, int M, int K, float threshold, int8_t *Xq, float *rowScaleX,
                                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * Synchronizes `stream`, then copies the outlier column set (A1, paper
 * walkthrough section 2.3) that the last llmint8_quantize_x / llmint8_matmul*
 * call on `workspace` found for rows of K columns:
 *   count     out  number of outlier columns (host int)
 *   idx_host  out  host int32 [capacity]: the first min(count, capacity)
 *                  column indices, ascending (may be NULL when capacity = 0)
 * EINVAL for NULL workspace or count, K outside [1, 65536], capacity < 0, or a
 * stored count outside [0, K] (a workspace no X pass of this K has filled);
 * ECUDA if synchronization or a copy fails.
 */
llmint8_status llmint8_read_outliers(const void *workspace, int K, int *count, int32_t *idx_host, int capacity,
                                     void *stream);

/*
 * Decode chain (1 <= M <= 4 rows, fp16): a matmul whose GEMV also prepares the
 * X pass of the next layer, when its output Y is that layer's input.  The
 * pages place the small-batch cost of the method in the per-forward handling
 * of the activations (paper walkthrough, section 5.4); here the outlier
 * columns of Y (A1 for the next threshold, paper walkthrough section 2.3) and
 * the row absmax of Y over the other columns (A2: sections 2.1 and 2.3) are
 * computed in the GEMV's epilogue and left in a "chain state", so the next call
 * runs one kernel and no X pass.  The codes, row scales and outlier set are
 * those llmint8_matmul derives from the same X (bit for bit; after a call given
 * a state they are left in the workspace fields of llmint8_workspace_layout),
 * and Y agrees with llmint8_matmul's within the stated tolerance (the outlier
 * slice is summed in another order).
 *
 *   X               in   fp16 [M, K] device (the previous layer's Y)
 *   threshold       in   outlier threshold of X, used only without state_in
 *   state_in        in   chain state of X written by the previous call's
 *                        state_out (same M, N of that call = K here), or NULL:
 *                        then the usual X pass runs first
 *   Wq, colScaleW, W16, Y   as llmint8_matmul
 *   next_threshold  in   threshold the flags of Y are taken for (not NaN)
 *   state_out       out  chain state of Y (llmint8_chain_state_bytes(M, N)
 *                        bytes, 16-byte aligned), or NULL
 *   state_in_bytes, state_out_bytes
 *                   in   sizes of the two state buffers (ignored for a NULL
 *                        state): at least llmint8_chain_state_bytes(M, K) and
 *                        llmint8_chain_state_bytes(M, N), else LLMINT8_EINVAL
 *   workspace       scratch as llmint8_matmul (error word, X-pass results)
 *
 * Chain state layout (llmint8_chain_state_layout): a 256-byte header (int32 M,
 * N, nparts, float threshold), then uint8 flags [N] (1 = outlier column, 0 =
 * not; no other values), then float [nparts][M] partial row maxima (the row
 * scale is their maximum; non-negative).  A caller may fill one by hand with
 * nparts = 1; M and N in the header must match the call that reads it (M and
 * K of that call) and 1 <= nparts <= N / 16.  The kernel checks this header
 * before it reads anything else of the state: a mismatch leaves Y unwritten and
 * records LLMINT8_EINVAL in the workspace error word (llmint8_device_status).
 *
 * Errors as llmint8_matmul; EUNSUPPORTED for M > 4, K < 512, or M * K too
 * large for shared memory; EINVAL if state_in == state_out, W16 is NULL while
 * outliers are possible, or next_threshold is NaN with a state_out; EALIGN for
 * a state pointer that is not 16-byte aligned.  state_in must not overlap Y or
 * state_out.  One kernel per call with state_in, else the X pass kernels plus
 * one.  Asynchronous on `stream`.
 */
size_t llmint8_chain_state_bytes(int M, int N);
llmint8_status llmint8_chain_state_layout(int M, int N, size_t *offsets /* [3]: flags, parts, total */);
llmint8_status llmint8_matmul_chain(const void *X, int M, int K, int N, float threshold, const void *state_in,
                                    size_t state_in_bytes, const int8_t *Wq, const float *colScaleW,
                                    const void *W16, void *Y, float next_threshold, void *state_out,
                                    size_t state_out_bytes, void *workspace, size_t workspace_bytes,
                                    void *stream);
/*
 * llmint8_matmul_chain that also writes the exact int32 accumulator of step A3,
 * C int32 [M, N] = sum_k Xq[i,k] * Wq[n,k] (introspection: the codes the chain
 * kernel derives from a state are then checkable bit for bit).  Same arguments
 * and errors, plus C (16-byte aligned, not NULL).
 */
llmint8_status llmint8_matmul_chain_i32(const void *X, int M, int K, int N, float threshold, const void *state_in,
                                        size_t state_in_bytes, const int8_t *Wq, const float *colScaleW,
                                        const void *W16, void *Y, float next_threshold, void *state_out,
                                        size_t state_out_bytes, int32_t *C, void *workspace,
                                        size_t workspace_bytes, void *stream);

/*
 * Allocation-free variant of llmint8_matmul.  The pages describe no such call;
 * it exists for callers that cannot allocate device memory when they run the
 * matmul: latency-critical loops that must not risk the device-wide
 * synchronization of cudaMalloc/cudaFree, hosts whose device memory is owned by
 * another allocator (a framework's caching pool, an embedding runtime), and
 * plug-ins that are handed device pointers but no allocation rights.
 *
 * Same arguments and results as llmint8_matmul minus the workspace: the scratch
 * space is a static 8 MiB device array inside the library (held by every GPU
 * that loads it until the process exits).  The call allocates nothing.
 *   - Shapes whose llmint8_workspace_bytes(M, K, N) exceeds 8 MiB return
 *     LLMINT8_EWORKSPACE (the 7B-like decode shapes need well under 1 MiB).
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - All calls share the array and it keeps the last call's contents; every
 *     call resets the parts that must start at zero.  Calls whose work overlaps
 *     on the GPU (other streams, other host threads without ordering) race on
 *     it: order them.
 *   - The device error word lives in the array and is not readable through
 *     llmint8_device_status.
 */
llmint8_status llmint8_matmul_noalloc(const void *X, int M, int K, int N, float threshold,
                                      const int8_t *Wq, const float *colScaleW,
                                      const void *W16, void *Y, void *stream);

/* ----------------------------------------------------------------------------
 * Introspection (tests and diagnostics; not on the hot path)
 * ------------------------------------------------------------------------- */

/*
 * Same arguments and kernels as llmint8_matmul, but the GEMM epilogue writes
 * the exact integer accumulator of step A3 instead of Y:
 *   C  out  int32 [M, N] row-major, C[i,n] = sum_k Xq[i,k] * Wq[n,k]
 * (|C| <= K * 127^2 < 2^31 for every accepted K <= 65536).  The fp16 outlier
 * product is not part of C; threshold still decides which columns of X are
 * zeroed, and W16 is not needed.
 */
llmint8_status llmint8_matmul_i32(const void *X, int M, int K, int N, float threshold,
                                  const int8_t *Wq, const float *colScaleW,
                                  int32_t *C, void *workspace, size_t workspace_bytes,
                                  void *stream);

/*
 * A3 alone on codes the caller chooses: C = Xq . Wq^T, exact int32, through the
 * same kernels the matmul uses (the int8 GEMV for M <= LLMINT8_DECODE_MAX_M;
 * above, the codes of Xq and Wq widened to exact fp16 integers and the
 * tensor-core GEMM with its 1024-long fp32 chunks drained into int32).  The
 * int8 x int8 -> int32 product the pages rescale afterwards ("Lightning Fabric
 * 8-bit" page, section 2.2; paper walkthrough, section 2.3).
 *
 *   Xq         in   int8 [M, K] row-major, any values in [-127, 127] (-128 is
 *                   accepted and multiplied as -128, but |C| < 2^31 is then the
 *                   caller's concern)
 *   Wq         in   int8 [N, K] row-major (the layout llmint8_quantize_weight
 *                   writes), values as Xq
 *   C          out  int32 [M, N] row-major, C[i,n] = sum_k Xq[i,k] * Wq[n,k]
 *   workspace  at least llmint8_workspace_bytes(M, K, N) bytes (its code and
 *              weight-code scratch are overwritten)
 *
 * EINVAL for NULL Xq, Wq or C or sizes as llmint8_matmul; EALIGN for K or N not
 * a multiple of 16 or an unaligned pointer; EWORKSPACE as llmint8_matmul.
 * Asynchronous on `stream`.
 */
llmint8_status llmint8_gemm_i32(const int8_t *Xq, const int8_t *Wq, int M, int K, int N, int32_t *C,
                                void *workspace, size_t workspace_bytes, void *stream);

/*
 * Number of kernels one llmint8_matmul (write_i32 = 0) or llmint8_matmul_i32
 * (write_i32 = 1) call launches for this shape and threshold (pass +INFINITY
 * for llmint8_matmul_int8): the outlier scan (not run at +INFINITY, nor for
 * M <= 16 with K <= 4096, where the row-quantization CTAs form one cluster and
 * find the outlier columns themselves), the row quantization, for M > 16 with a
 * finite threshold and write_i32 = 0 the gather of the outlier rows of W16
 * (unless the row quantization writes them: K <= 4096 and ceil(M/8) * 8 >=
 * N/16), for M > 16 the widening of the weight codes to fp16, and the GEMV or
 * GEMM.
 * The bf16 entry points launch the same kernels; llmint8_matmul_w8 launches the
 * gather for every M > 16 with a finite threshold (one more kernel when
 * K <= 4096).  -1 for arguments the call would reject as EINVAL.
 * Host-only; touches no device.
 */
int llmint8_kernels_per_call(int M, int K, int N, float threshold, int write_i32);

/* Workspace fields whose offsets llmint8_workspace_layout reports. */
enum {
    LLMINT8_WS_STATUS = 0,       /* uint32: device error word (0 = OK, else an llmint8_status) */
    LLMINT8_WS_OUTLIER_COUNT = 1,/* int32: number of outlier columns found by the last call */
    LLMINT8_WS_OUTLIER_IDX = 2,  /* int32 [count]: outlier column indices, ascending */
    LLMINT8_WS_ROW_SCALE = 3,    /* fp32 [M]: rowScaleX (absmax over non-outlier columns) */
    LLMINT8_WS_CODES = 4,        /* [M, K] row-major codes of X: int8 when M <= 16 (the
                                    decode path), else the same codes stored as exact fp16
                                    values (the tensor-core operand format) */
    LLMINT8_WS_NFIELDS = 5
};

/*
 * Byte offsets of the fields above inside a workspace used by a call with the
 * same (M, K, N).  After a llmint8_matmul* call has completed, the fields hold
 * that call's intermediate results.  offsets must hold LLMINT8_WS_NFIELDS values.
 */
llmint8_status llmint8_workspace_layout(int M, int K, int N, size_t *offsets);

/*
 * Synchronize `stream`, then read and clear the device error word of `workspace`.
 * Every llmint8_matmul* call clears the word when it starts, so it reports the
 * last call that used this workspace (or the last llmint8_selftest_timeout).
 * Returns LLMINT8_OK, or the status a kernel recorded (LLMINT8_ETIMEOUT when a
 * bounded wait gave up), or LLMINT8_ECUDA if synchronization itself failed.
 */
llmint8_status llmint8_device_status(void *workspace, void *stream);

/*
 * Self-test of the bounded-wait machinery: launches one small kernel that waits
 * on a shared-memory barrier that nothing ever completes, giving up after
 * `spin_limit` polls (1 .. 1e7).  It then records LLMINT8_ETIMEOUT in the
 * workspace error word and returns; no GPU hang, trap or fault is involved.
 * The workspace needs at least 256 bytes.
 */
llmint8_status llmint8_selftest_timeout(void *workspace, int spin_limit, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LLMINT8_H */
