/*
 * fa.h -- C ABI of libfa.so, exact scaled-dot-product attention on one GB300.
 *
 * The method.  Attention O = softmax(Q K^T * scale) V is computed block by
 * block in on-chip memory (lexicon page "FlashAttention" (urworte.de),
 * section "Methodische Grundlagen": "Blockweise Verarbeitung"), with the
 * score, normalisation and weighting steps fused into one pass
 * ("Verschmelzung der Schritte") and the row normalisation kept as a running
 * statistic that corrects earlier partial results when a larger score shows
 * up ("Fortlaufende Normierung").  The backward pass recomputes the scores
 * instead of storing them ("Neuberechnung statt Speicherung").  The result
 * equals the conventional computation up to rounding ("Exaktheit").  The
 * N x N score matrix never reaches device memory, so memory grows linearly
 * in N (page "FlashAttention-2 (DE)" (systems-analysis.info), section
 * "Hintergrund").
 *
 * Conventions shared by every call below.
 *  - Tensors q, k, v, o, dO, dq, dk, dv are bf16, contiguous [B, H, N, d]
 *    (d fastest), except in the *_strided calls, which take any layout
 *    whose d elements are contiguous.  lse is fp32, contiguous [B, H, N].
 *    All pointers are
 *    device pointers owned by the caller, 16-byte aligned, non-null, and
 *    the library keeps none of them after the call returns.  The library
 *    owns only a device status word per device, and for fa_bwd and its
 *    strided and packed forms one side stream and two events per host
 *    thread and device.
 *  - B, H, N >= 1; d is 64 or 128 (FA_ERR_UNSUPPORTED otherwise);
 *    B*H*ceil(N/128) < 2^31 (one backward CTA per head and block of 128
 *    rows must fit a launch grid) and B*H*N*d < 2^39 elements per tensor
 *    (1 TiB of bf16: TMA byte strides stay below 2^40), which admits every
 *    tensor a GPU's memory can hold; element offsets are 64-bit
 *    throughout.
 *  - causal is 0 or 1.  With causal = 1, key j is visible to query i iff
 *    j <= i (square mask, aligned at the top-left).  Fully masked tiles are
 *    skipped.
 *  - scale is any finite float (the usual value is 1/sqrt(d)).
 *  - lse[i] = ln sum_{j visible} exp(scale * q_i . k_j): the natural-log
 *    logsumexp of the SCALED scores.
 *  - Outputs must not overlap inputs.
 *  - Every call is asynchronous on `stream` (0 = the legacy default
 *    stream) and validates all arguments on the host before any CUDA call;
 *    an invalid call launches nothing and returns an error code.
 *  - A kernel whose internal pipeline wait runs past its time limit stops,
 *    records FA_ERR_DEVICE_TIMEOUT in a per-device status word and returns;
 *    fa_device_status() reads and clears it.  Kernels never trap.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARGUMENT = 1, /* null/misaligned pointer, bad size, non-finite scale, bad flag */
    FA_ERR_UNSUPPORTED = 2,      /* head dimension other than 64 or 128 */
    FA_ERR_WORKSPACE = 3,        /* caller workspace smaller than fa_bwd_workspace_bytes() */
    FA_ERR_CUDA = 4,             /* a CUDA runtime/driver call or launch failed */
    FA_ERR_DEVICE_TIMEOUT = 5    /* a kernel gave up on a pipeline wait (see fa_device_status) */
} fa_status_t;

/*
 * Forward pass: o = softmax(q k^T * scale) v and lse (see conventions).
 * Page "FlashAttention" (urworte.de), "Methodische Grundlagen": tiling,
 * fused steps and running normalisation; page "FlashAttention-2 (DE)",
 * "Technische Architektur", section 2: the work of one head is spread over
 * the SMs by query block.
 *   q, k, v : inputs  [B, H, N, d] bf16
 *   o       : output  [B, H, N, d] bf16
 *   lse     : output  [B, H, N] fp32
 * Bitwise reproducible from run to run for the same inputs.
 */
FA_API fa_status_t fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                   int B, int H, int N, int d, int causal, float scale,
                   cudaStream_t stream);

/*
 * Bytes of device workspace fa_bwd needs for these sizes: D = rowsum(dO * O)
 * and the logsumexp in log2 units, each fp32 [B, H, Np] with N padded up to
 * Np, the next multiple of 128, each rounded up to 256 bytes.  Linear in N.
 * Returns 0 for sizes fa_bwd would reject.
 */
FA_API size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward pass: gradients of a loss L through o = attention(q, k, v), given
 * dO = dL/do and the lse saved by fa_fwd.  The scores and probabilities are
 * recomputed from q, k and lse; nothing of size N x N is stored (page
 * "FlashAttention" (urworte.de), "Methodische Grundlagen", paragraph
 * "Neuberechnung statt Speicherung").
 *   q, k, v, o, dO : inputs  [B, H, N, d] bf16 (o as written by fa_fwd)
 *   lse            : input   [B, H, N] fp32 (as written by fa_fwd)
 *   dq, dk, dv     : outputs [B, H, N, d] bf16
 *   workspace      : device scratch of at least fa_bwd_workspace_bytes()
 *                    bytes, 256-byte aligned, or NULL to let the library
 *                    take it with cudaMallocAsync/cudaFreeAsync on `stream`.
 * No atomics are used: dq, dk and dv are bitwise reproducible run to run.
 * The dK/dV kernel runs on `stream` and the dQ kernel next to it on a side
 * stream of the library's (one per host thread and device, created on the
 * first call with two events, kept until the process exits); `stream`
 * waits for both before any work enqueued after the call, so the ordering
 * a caller sees is that of a single stream.
 */
FA_API fa_status_t fa_bwd(const void *q, const void *k, const void *v, const void *o,
                   const void *dO, const float *lse, void *dq, void *dk, void *dv,
                   int B, int H, int N, int d, int causal, float scale,
                   void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Strided layouts.  The same two passes on tensors in any layout whose d
 * elements are contiguous: element (b, h, n, c) of a tensor lies at
 *     base + b * strides[0] + h * strides[1] + n * strides[2] + c
 * (strides in elements, int64, one array of three per tensor).  This covers
 * [B, N, H, d] ("BNHD", the layout of many frameworks' projections), the
 * q, k, v slices of one packed [B, N, 3, H, d] projection, and any padded
 * row pitch; the page "FlashAttention-2 (DE)" (systems-analysis.info),
 * section "Anwendung und Integration in das Oekosystem", names the
 * frameworks this is for.  Rules: every stride of a dimension of extent > 1
 * is a positive multiple of 8 elements (16 bytes) below 2^39 (the stride of
 * an extent-1 dimension is ignored); inputs may share memory with each
 * other (a packed projection); each output's elements are all distinct and
 * no output overlaps an input, another output or the workspace (checked on
 * the address ranges spanned).  lse stays contiguous [B, H, N].  Everything
 * else is as in fa_fwd / fa_bwd; with contiguous strides the results are
 * bitwise those of fa_fwd / fa_bwd.
 */
FA_API fa_status_t fa_fwd_strided(const void *q, const int64_t *q_strides, const void *k,
                                  const int64_t *k_strides, const void *v, const int64_t *v_strides,
                                  void *o, const int64_t *o_strides, float *lse, int B, int H, int N,
                                  int d, int causal, float scale, cudaStream_t stream);

FA_API fa_status_t fa_bwd_strided(const void *q, const int64_t *q_strides, const void *k,
                                  const int64_t *k_strides, const void *v, const int64_t *v_strides,
                                  const void *o, const int64_t *o_strides, const void *dO,
                                  const int64_t *dO_strides, const float *lse, void *dq,
                                  const int64_t *dq_strides, void *dk, const int64_t *dk_strides,
                                  void *dv, const int64_t *dv_strides, int B, int H, int N, int d,
                                  int causal, float scale, void *workspace, size_t workspace_bytes,
                                  cudaStream_t stream);

/*
 * Packed variable-length sequences ("varlen").  B sequences of different
 * lengths stored back to back along one row axis of T rows: sequence b is
 * rows [cu_seqlens[b], cu_seqlens[b+1]) of every tensor, and attends only
 * to itself (causal = 1: key j visible to query i iff j <= i, positions
 * counted from the sequence's first row).
 *   q, k, v, o, dO, dq, dk, dv : [T, H, d] bf16 with element strides
 *                    strides[0] between rows and strides[1] between heads
 *                    (d contiguous; same rules as the strided calls)
 *   lse          : [H, T] fp32, contiguous
 *   cu_seqlens   : device array of B + 1 int32 row offsets, 4-byte aligned:
 *                  0 = cu[0] <= cu[1] <= ... <= cu[B] = T, every length
 *                  cu[b+1] - cu[b] at most max_seqlen.  The kernels read it
 *                  on the device, so the host cannot check it; they clamp
 *                  every offset into [0, T] and every length to max_seqlen,
 *                  so a malformed array gives wrong results for the
 *                  sequences it describes, never an access outside the
 *                  tensors.  Zero-length sequences are allowed.
 *   max_seqlen   : the longest sequence (sizes the launch and the workspace)
 * The backward workspace is fa_bwd_workspace_bytes(B, H, max_seqlen, d).
 * The pages describe attention per sequence; packing several sequences into
 * one call is this library's reading of the framework integration that the
 * page "FlashAttention-2 (DE)", section "Anwendung und Integration in das
 * Oekosystem", names.
 */
FA_API fa_status_t fa_fwd_varlen(const void *q, const int64_t *q_strides, const void *k,
                                 const int64_t *k_strides, const void *v, const int64_t *v_strides,
                                 void *o, const int64_t *o_strides, float *lse,
                                 const int *cu_seqlens, int B, int H, int T, int max_seqlen, int d,
                                 int causal, float scale, cudaStream_t stream);

FA_API fa_status_t fa_bwd_varlen(const void *q, const int64_t *q_strides, const void *k,
                                 const int64_t *k_strides, const void *v, const int64_t *v_strides,
                                 const void *o, const int64_t *o_strides, const void *dO,
                                 const int64_t *dO_strides, const float *lse, void *dq,
                                 const int64_t *dq_strides, void *dk, const int64_t *dk_strides,
                                 void *dv, const int64_t *dv_strides, const int *cu_seqlens, int B,
                                 int H, int T, int max_seqlen, int d, int causal, float scale,
                                 void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * FP8 forward: the forward pass with Q, K, V given as e4m3 codes (OCP FP8
 * E4M3: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinities, 0x7F/0xFF NaN) and one fp32 scale per tensor: element value =
 * decoded code * q_scale (k_scale, v_scale).  Both products run on the
 * tensor core's 8-bit path.  The page "FlashAttention-2 (DE)", section
 * "Vergleich mit nachfolgenden Versionen" / "FlashAttention-3", names
 * low-precision FP8 as a FlashAttention-3 addition without a formula; what
 * this call computes, per row i (log2 units, x_ij = scale * log2(e) *
 * q_i . k_j on the decoded, scaled values, masked keys excluded):
 *   M_i = ceil(max_j x_ij);  w_ij = e4m3 rounding (nearest, ties to even)
 *   of 2^(x_ij - M_i + 8), at most 256;
 *   o_i = sum_j w_ij v_j / sum_j w_ij  (bf16);
 *   lse_i = ln 2 * (M_i - 8 + log2 sum_j 2^(x_ij - M_i + 8))  (fp32, exact
 *   logsumexp of the scaled scores, as in fa_fwd).
 * The weights are what an FP8 tensor-core product of P and V can apply; the
 * integer M_i makes them independent of how the keys are tiled (outside
 * e4m3's subnormal range, 2^(x - M + 8) < 2^-6, where the rounding grid of
 * a tiled pass may be finer).
 *   q8, k8, v8 : [B, H, N, d] e4m3 codes (1 byte each), contiguous
 *   o          : [B, H, N, d] bf16, lse : [B, H, N] fp32, contiguous
 *   d must be 128 (FA_ERR_UNSUPPORTED otherwise); the tensor scales must
 *   be finite; other conventions as above.
 */
FA_API fa_status_t fa_fwd_fp8(const void *q8, const void *k8, const void *v8, float q_scale,
                              float k_scale, float v_scale, void *o, float *lse, int B, int H, int N,
                              int d, int causal, float scale, cudaStream_t stream);

/*
 * Decode forward: Nq new query rows per (batch entry, head) against a cache
 * of keys and values, as in token-by-token generation.  The computation is
 * the forward pass above (o and lse, same definition and scale), with
 * rectangular shapes: per (b, h) the query rows are q[b, h, 0..Nq) and the
 * keys/values are the first len_b rows of the cache, len_b = cache_seqlens[b]
 * (all Nk rows when cache_seqlens is NULL).  The query rows are the LAST Nq
 * positions of the sequence: with causal = 1, query i sees key j iff
 * j <= len_b - Nq + i (mask aligned at the bottom-right; for Nq = 1 it is no
 * restriction); with causal = 0 it sees every key j < len_b.  A query row
 * that sees no key (len_b = 0, or causal with len_b - Nq + i < 0) gets
 * o = 0 and lse = -inf.
 *   q    : [B, H, Nq, d] bf16, element strides q_strides[3] (b, h, row)
 *   k, v : [B, H, Nk, d] bf16, element strides k_strides / v_strides (a
 *          cache stored [B, Nk, H, d] is strides {Nk*H*d, d, H*d})
 *   o    : [B, H, Nq, d] bf16, strides o_strides; must not overlap anything
 *   lse  : [B, H, Nq] fp32, contiguous
 *   cache_seqlens : NULL, or a device array of B int32 (4-byte aligned);
 *          the kernel clamps each value into [0, Nk], so a bad value gives a
 *          wrong result for its batch entry, never an access outside k, v
 *   1 <= Nq <= 8, Nk >= 1 (Nk <= 2^30), d 64 or 128, B*H < 2^24; strides
 *   follow the rules of the *_strided calls.
 *   workspace : device scratch of fa_decode_workspace_bytes(B, H, Nq, Nk, d)
 *          bytes (256-byte aligned; that size may be 0), or NULL to let the
 *          call take it with cudaMallocAsync/cudaFreeAsync on `stream`.
 * Work is split over the keys: each 128-key tile chunk of a head gives a
 * partial result normalised over its own keys and its logsumexp, and the
 * partials are merged with the same running-maximum correction the tiled
 * pass uses between key blocks; the chunk size depends on the shape only,
 * so the result is bitwise reproducible for the same inputs.  The
 * glossary page "FlashAttention" (blog.brdg.mn) places the method in model
 * serving next to the block-wise management of the key/value cache
 * (sections "Der Engpass ist der Weg zum Speicher, nicht das Rechnen" and
 * "Wo es verwechselt wird"); decoding against that cache is this call.
 * The cache's block management itself is not part of the library.
 */
FA_API size_t fa_decode_workspace_bytes(int B, int H, int Nq, int Nk, int d);

FA_API fa_status_t fa_fwd_decode(const void *q, const int64_t *q_strides, const void *k,
                                 const int64_t *k_strides, const void *v, const int64_t *v_strides,
                                 void *o, const int64_t *o_strides, float *lse,
                                 const int *cache_seqlens, int B, int H, int Nq, int Nk, int d,
                                 int causal, float scale, void *workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/*
 * Size in bytes of the fixed device array that fa_bwd_noalloc uses as its
 * scratch (8 MiB).  Every GPU that loads the library holds this array until
 * the process exits.  It covers B * H * Np <= 1,048,576 padded rows, where
 * Np is N rounded up to a multiple of 128 (for example B*H = 32 heads of
 * N = 32768).
 */
#define FA_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * Backward pass for callers that must not allocate device memory: the same
 * computation, arguments, layouts and results as fa_bwd, but with no
 * workspace argument and no allocation of any kind (no cudaMalloc,
 * cudaMallocAsync or cudaFree, and no side stream: its kernels run one
 * after the other on `stream`).  Its scratch lives in a fixed array of the
 * library (FA_NOALLOC_SCRATCH_BYTES); calls that would need more return
 * FA_ERR_WORKSPACE without launching anything.
 *
 * Who needs it: callers whose device memory is owned by someone else (a
 * framework's memory manager that must see every allocation) or planned up
 * front (a process that must not allocate once it runs), which can neither
 * pass fa_bwd a workspace nor let it take one.
 *
 * Set-up and sharing: every call looks up the array's device address in
 * the current context (cudaGetSymbolAddress, a host-side query; the first
 * lookup in a process may load the library's device code).  All calls share
 * the one array and it keeps the last
 * call's contents; nothing in it needs to start at zero.
 * Calls whose work overlaps on the GPU (other streams or host threads on
 * the same device) race on it, so the caller must order them.
 *
 * The pages describe no counterpart of this entry point.
 */
FA_API fa_status_t fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                                  const void *dO, const float *lse, void *dq, void *dk, void *dv,
                                  int B, int H, int N, int d, int causal, float scale,
                                  cudaStream_t stream);

/*
 * Synchronises `stream`, then returns the status word the kernels of the
 * current device recorded (FA_OK or FA_ERR_DEVICE_TIMEOUT) and resets it to
 * FA_OK.  Returns FA_ERR_CUDA if the synchronisation itself fails.
 */
FA_API fa_status_t fa_device_status(cudaStream_t stream);

/*
 * Diagnostic: the wait site (a small positive integer naming the pipeline
 * barrier) of the first timeout recorded on the current device since the
 * status word was last cleared, 0 if none, -1 if it cannot be read.  Call it
 * before fa_device_status(), which clears the record.
 */
FA_API int fa_debug_last_wait_site(void);

/*
 * Diagnostic timing hook: the next fa_bwd call made by this host thread
 * records, on its stream, `start` right before the launch of its dK/dV
 * kernel, `mid` between that kernel and its dQ kernel, and `stop` right
 * after the dQ kernel, so both kernels can be timed with
 * cudaEventElapsedTime (that call runs the two kernels one after the
 * other on its stream, not side by side).  The events are created and owned by the caller;
 * the hook is used once and then cleared.  Returns FA_ERR_INVALID_ARGUMENT
 * if any event is NULL.
 */
FA_API fa_status_t fa_debug_time_next_bwd(cudaEvent_t start, cudaEvent_t mid, cudaEvent_t stop);

/* A static, NUL-terminated description of a status code. */
FA_API const char *fa_status_string(fa_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
