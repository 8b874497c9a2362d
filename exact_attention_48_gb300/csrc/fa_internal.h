// fa_internal.h -- host-side declarations shared by the translation units of
// libfa.so (kernel parameter blocks and launchers).  Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime_api.h>
#include <cstdint>

#include "../../include/fa.h"

namespace fa {

// Where a kernel gave up waiting (second word of the device status block).
enum WaitSite : int {
  kSiteQFull = 1,
  kSiteKFull,
  kSiteKEmpty,
  kSiteVFull,
  kSiteVEmpty,
  kSiteSFull,
  kSitePReady,
  kSitePvDone,
  kSiteDoFull,
  kSiteDoEmpty,
  kSiteDsReady,
  kSiteDqFull,
  kSiteDqEmpty,
  kSiteKvFull,
  kSiteMmaDone,
  kSiteKvEmpty,
  kSiteQEmpty,
};

// Element strides of a [B, H, N, d] bf16 tensor whose d elements are
// contiguous: element (b, h, n, c) is at base + b*b + h*h + n*n + c.
struct Strides {
  long long b, h, n;
};

// Offset of row n of head bh (= b*H + h) of a strided tensor.
__host__ __device__ inline long long row_offset(const Strides &s, int bh, int H, int n) {
  return static_cast<long long>(bh / H) * s.b + static_cast<long long>(bh % H) * s.h + static_cast<long long>(n) * s.n;
}

// Rows of the sequence of batch entry b: [start, start + len) of the
// tensors' row axis.  Batched mode (cu == null): every sequence is rows
// [0, N) of its own batch slot.  Packed ("varlen") mode: sequence b is rows
// [cu[b], cu[b+1]) of one packed row axis of T rows, N is the longest
// sequence; the bounds are clamped into [0, T] and the length to N, so that
// no access leaves the tensors whatever the array holds.
struct SeqRange {
  int start, len;
};
__device__ inline SeqRange seq_range(const int *cu, int b, int N, int T) {
  if (!cu) return SeqRange{0, N};
  int s = cu[b], e = cu[b + 1];
  s = s < 0 ? 0 : (s > T ? T : s);
  e = e < s ? s : (e > T ? T : e);
  const int len = e - s;
  return SeqRange{s, len < N ? len : N};
}

struct FwdParams {
  __nv_bfloat16 *o;   // [B, H, N, d] with strides so
  float *lse;         // [BH, N] contiguous
  Strides so;
  int H;
  const int *cu_seqlens;       // packed mode: B+1 row offsets (device); null in batched mode
  int T;                       // packed mode: rows of the packed row axis
  long long lse_b, lse_h;      // lse index = b*lse_b + h*lse_h + row (row on the tensors' row axis)
  int *status;        // device status block (2 ints)
  int N;
  int BH;
  int num_qblk;       // ceil(N / 256): one CTA per 256 query rows
  int persist_ctas;   // > 0: persistent launch of this many CTAs walking the 256-row tiles
  float scale_log2;   // scale * log2(e)
  int neg;            // scale < 0
};

struct BwdParams {
  const __nv_bfloat16 *q;     // [B, H, N, d] with strides sq (likewise every bf16 tensor below)
  const __nv_bfloat16 *o;
  const __nv_bfloat16 *dout;
  const float *lse;           // [BH, N]
  float *delta;               // [BH, Np]  D = rowsum(dO * O), Np = 128 * num_blk, 0 past N
  float *lse2;                // [BH, Np]  lse * log2(e), +inf past N
  __nv_bfloat16 *dq;
  __nv_bfloat16 *dk;
  __nv_bfloat16 *dv;
  Strides sq, so, sdo, sdq, sdk, sdv;
  int H;
  const int *cu_seqlens;       // as in FwdParams
  int T;
  long long lse_b, lse_h;
  int *status;
  int N;
  int BH;
  int num_blk;                // ceil(N / 128)
  float scale;
  float scale_log2;
  int head_major;             // causal: order the blocks head by head (heaviest first inside a head)
  int pairs_kv, pairs_q;      // causal: one CTA per pair of mirror blocks (j, nb-1-j) of a head in the
                              // dK/dV kernel, in the dQ kernel
};

// Decode forward: Nq (<= 8) query rows per head against Nk cached keys.
// The keys of a head are cut into chunks of `chunk` 128-key tiles; item
// it = split * BH + bh is chunk `split` of head bh.  With splits > 1 each
// item writes its normalised partial O and log2-domain logsumexp to
// part_o / part_lse and a second kernel merges them.
struct DecodeParams {
  const __nv_bfloat16 *q;     // [B, H, Nq, d] strides sq
  __nv_bfloat16 *o;           // [B, H, Nq, d] strides so
  float *lse;                 // [B, H, Nq] contiguous (natural log)
  Strides sq, so;
  const int *cache_len;       // [B] valid keys per batch entry (device), or null: all Nk
  float *part_o;              // [BH][splits][Nq][d] fp32 (splits > 1)
  float *part_lse;            // [BH][splits][Nq] fp32, log2 units (splits > 1)
  int *status;
  int H, BH, Nq, Nk;
  int chunk, splits, items;
  int causal;                 // query i sees keys j <= len - Nq + i
  float scale_log2;           // scale * log2(e)
};

// tq: q as [B, H, Nq, d] with boxes of 16 rows (used by the tensor-core kernel).
cudaError_t launch_decode(int d, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tq,
                          const DecodeParams &p, int grid, cudaStream_t stream);

// FP8 forward (e4m3 Q, K, V with tensor scales; d = 128).
struct Fp8FwdParams {
  __nv_bfloat16 *o;   // [B, H, N, d] with strides so
  float *lse;         // [B, H, N] contiguous
  Strides so;
  int H;
  int *status;
  int N;
  int BH;
  int num_qblk;       // ceil(N / 256)
  float scale_log2;   // scale * q_scale * k_scale * log2(e)
  float v_scale;
  int neg;            // scale_log2 < 0
};

cudaError_t launch_fwd_fp8(bool causal, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const Fp8FwdParams &p, cudaStream_t stream);

// Tensor maps over [B, H, N, d] bf16 tensors viewed as 4-D (d, N, H, B)
// with the tensors' strides, box (64, 128, 1, 1), 128-byte swizzle.
cudaError_t launch_fwd(int d, bool causal, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const FwdParams &p, cudaStream_t stream);

// ev[0..2] (all null or all set) are recorded before the dK/dV kernel,
// between it and the dQ kernel, and after the dQ kernel; the two kernels
// then run one after the other.  Without events and with `concurrent`, the
// dQ kernel runs on a side stream next to the dK/dV kernel, joined before
// the call returns.
cudaError_t launch_bwd(int d, bool causal, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const CUtensorMap &tdo, const BwdParams &p,
                       cudaStream_t stream, const cudaEvent_t *ev, bool concurrent);

}  // namespace fa

// The backward pass of fa_bwd with its two main kernels one after the
// other on `stream` (no side stream): used by fa_bwd_noalloc.  Internal
// (hidden visibility: not exported from libfa.so).
extern "C" fa_status_t fa_bwd_sequential(const void *q, const void *k, const void *v, const void *o, const void *dO,
                              const float *lse, void *dq, void *dk, void *dv, int B, int H, int N, int d,
                              int causal, float scale, void *workspace, size_t workspace_bytes,
                              cudaStream_t stream);

namespace fa {

}  // namespace fa
