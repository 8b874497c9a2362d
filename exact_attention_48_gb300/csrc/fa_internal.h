// fa_internal.h -- host-side declarations shared by the translation units of
// libfa.so (kernel parameter blocks and launchers).  Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime_api.h>
#include <cstdint>

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
};

struct FwdParams {
  __nv_bfloat16 *o;   // [BH, N, d]
  float *lse;         // [BH, N]
  int *status;        // device status block (2 ints)
  int N;
  int BH;
  int num_qblk;       // ceil(N / 256): one CTA per 256 query rows
  float scale_log2;   // scale * log2(e)
  int neg;            // scale < 0
};

struct BwdParams {
  const __nv_bfloat16 *q;     // [BH, N, d]
  const __nv_bfloat16 *o;     // [BH, N, d]
  const __nv_bfloat16 *dout;  // [BH, N, d]
  const float *lse;           // [BH, N]
  float *delta;               // [BH, Np]  D = rowsum(dO * O), Np = 128 * num_blk, 0 past N
  float *lse2;                // [BH, Np]  lse * log2(e), +inf past N
  __nv_bfloat16 *dq;          // [BH, N, d]
  __nv_bfloat16 *dk;          // [BH, N, d]
  __nv_bfloat16 *dv;          // [BH, N, d]
  int *status;
  int N;
  int BH;
  int num_blk;                // ceil(N / 128)
  float scale;
  float scale_log2;
};

// Three tensor maps over a [BH, N, d] bf16 tensor viewed as 3-D (d, N, BH),
// box (64, 128, 1), 128-byte swizzle.
cudaError_t launch_fwd(int d, bool causal, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const FwdParams &p, cudaStream_t stream);

// ev[0..2] (all null or all set) are recorded before the dK/dV kernel,
// between it and the dQ kernel, and after the dQ kernel.
cudaError_t launch_bwd(int d, bool causal, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const CUtensorMap &tdo, const BwdParams &p,
                       cudaStream_t stream, const cudaEvent_t *ev);

}  // namespace fa
