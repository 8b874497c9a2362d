// fa_api.cu -- the C ABI of libfa.so: argument validation, TMA descriptor
// encoding, workspace handling, the device status word and the launches.
// The operations themselves are defined in include/fa.h.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace fa {
namespace {

// Status block per device: [0] = FA_OK or FA_ERR_DEVICE_TIMEOUT, [1] = wait site.
__device__ int g_status[2];

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// [BH, N, d] bf16 viewed as 3-D (d, N, BH); one box is 64 columns (128
// bytes, the swizzle span) x 128 rows of one head.  Rows past N read as 0.
bool encode_bhnd(CUtensorMap *map, const void *base, int BH, int N, int d) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int *status_ptr() {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
  return static_cast<int *>(p);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-side checks shared by both passes; no CUDA call happens before them.
fa_status_t check_common(int B, int H, int N, int d, int causal, float scale) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARGUMENT;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARGUMENT;
  if (d != 64 && d != 128) return d < 1 ? FA_ERR_INVALID_ARGUMENT : FA_ERR_UNSUPPORTED;
  const long long elems = static_cast<long long>(B) * H * N * d;
  if (elems >= (1LL << 31)) return FA_ERR_INVALID_ARGUMENT;
  return FA_OK;
}

// Events the next fa_bwd call of this thread records around its kernels.
thread_local cudaEvent_t t_bwd_ev[3] = {nullptr, nullptr, nullptr};

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

const char *fa_status_string(fa_status_t s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported head dimension (d must be 64 or 128)";
    case FA_ERR_WORKSPACE: return "workspace too small";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_DEVICE_TIMEOUT: return "a kernel timed out waiting inside its pipeline";
  }
  return "unknown status";
}

fa_status_t fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int N, int d,
                   int causal, float scale, cudaStream_t stream) {
  fa_status_t st = check_common(B, H, N, d, causal, scale);
  if (st != FA_OK) return st;
  const void *ptrs[5] = {q, k, v, o, lse};
  for (const void *x : ptrs)
    if (!x || !aligned16(x)) return FA_ERR_INVALID_ARGUMENT;
  const size_t tb = static_cast<size_t>(B) * H * N * d * 2, lb = static_cast<size_t>(B) * H * N * 4;
  for (const void *in : {q, k, v})
    if (overlaps(in, tb, o, tb) || overlaps(in, tb, lse, lb)) return FA_ERR_INVALID_ARGUMENT;
  if (overlaps(o, tb, lse, lb)) return FA_ERR_INVALID_ARGUMENT;

  const int BH = B * H;
  CUtensorMap tq, tk, tv;
  if (!encode_bhnd(&tq, q, BH, N, d) || !encode_bhnd(&tk, k, BH, N, d) || !encode_bhnd(&tv, v, BH, N, d))
    return FA_ERR_CUDA;
  FwdParams p{};
  p.o = static_cast<__nv_bfloat16 *>(o);
  p.lse = lse;
  p.status = status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  p.N = N;
  p.BH = BH;
  p.num_qblk = (N + 255) / 256;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.neg = scale < 0.0f ? 1 : 0;
  return launch_fwd(d, causal != 0, tq, tk, tv, p, stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (check_common(B, H, N, d, 0, 1.0f) != FA_OK) return 0;
  const size_t padded_rows = static_cast<size_t>(B) * H * ((N + 127) / 128) * 128;
  return 2 * round256(padded_rows * 4);
}

fa_status_t fa_bwd(const void *q, const void *k, const void *v, const void *o, const void *dO, const float *lse,
                   void *dq, void *dk, void *dv, int B, int H, int N, int d, int causal, float scale, void *workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
  fa_status_t st = check_common(B, H, N, d, causal, scale);
  if (st != FA_OK) return st;
  const void *ptrs[9] = {q, k, v, o, dO, lse, dq, dk, dv};
  for (const void *x : ptrs)
    if (!x || !aligned16(x)) return FA_ERR_INVALID_ARGUMENT;
  const size_t tb = static_cast<size_t>(B) * H * N * d * 2, lb = static_cast<size_t>(B) * H * N * 4;
  const void *ins[6] = {q, k, v, o, dO, lse};
  const size_t in_sz[6] = {tb, tb, tb, tb, tb, lb};
  void *outs[3] = {dq, dk, dv};
  for (int i = 0; i < 6; ++i)
    for (void *out : outs)
      if (overlaps(ins[i], in_sz[i], out, tb)) return FA_ERR_INVALID_ARGUMENT;
  if (overlaps(dq, tb, dk, tb) || overlaps(dq, tb, dv, tb) || overlaps(dk, tb, dv, tb)) return FA_ERR_INVALID_ARGUMENT;
  const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
  if (workspace) {
    if (workspace_bytes < need) return FA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_INVALID_ARGUMENT;
    for (int i = 0; i < 6; ++i)
      if (overlaps(ins[i], in_sz[i], workspace, need)) return FA_ERR_INVALID_ARGUMENT;
    for (void *out : outs)
      if (overlaps(out, tb, workspace, need)) return FA_ERR_INVALID_ARGUMENT;
  }

  const int BH = B * H;
  CUtensorMap tq, tk, tv, tdo;
  if (!encode_bhnd(&tq, q, BH, N, d) || !encode_bhnd(&tk, k, BH, N, d) || !encode_bhnd(&tv, v, BH, N, d) ||
      !encode_bhnd(&tdo, dO, BH, N, d))
    return FA_ERR_CUDA;

  void *ws = workspace;
  bool owned = false;
  if (!ws) {
    if (cudaMallocAsync(&ws, need, stream) != cudaSuccess) return FA_ERR_CUDA;
    owned = true;
  }
  BwdParams p{};
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.o = static_cast<const __nv_bfloat16 *>(o);
  p.dout = static_cast<const __nv_bfloat16 *>(dO);
  p.lse = lse;
  const size_t padded_rows = static_cast<size_t>(BH) * ((N + 127) / 128) * 128;
  p.delta = static_cast<float *>(ws);
  p.lse2 = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + round256(padded_rows * 4));
  p.dq = static_cast<__nv_bfloat16 *>(dq);
  p.dk = static_cast<__nv_bfloat16 *>(dk);
  p.dv = static_cast<__nv_bfloat16 *>(dv);
  p.status = status_ptr();
  p.N = N;
  p.BH = BH;
  p.num_blk = (N + 127) / 128;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  fa_status_t rc = FA_OK;
  const cudaEvent_t ev[3] = {t_bwd_ev[0], t_bwd_ev[1], t_bwd_ev[2]};
  t_bwd_ev[0] = t_bwd_ev[1] = t_bwd_ev[2] = nullptr;
  if (!p.status || launch_bwd(d, causal != 0, tq, tk, tv, tdo, p, stream, ev[0] ? ev : nullptr) != cudaSuccess)
    rc = FA_ERR_CUDA;
  if (owned && cudaFreeAsync(ws, stream) != cudaSuccess) rc = FA_ERR_CUDA;
  return rc;
}

fa_status_t fa_device_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  int h[2] = {0, 0};
  if (cudaMemcpyFromSymbol(h, g_status, sizeof(h)) != cudaSuccess) return FA_ERR_CUDA;
  if (h[0] != 0) {
    const int zero[2] = {0, 0};
    if (cudaMemcpyToSymbol(g_status, zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
    return static_cast<fa_status_t>(h[0]);
  }
  return FA_OK;
}

fa_status_t fa_debug_time_next_bwd(cudaEvent_t start, cudaEvent_t mid, cudaEvent_t stop) {
  if (!start || !mid || !stop) return FA_ERR_INVALID_ARGUMENT;
  t_bwd_ev[0] = start;
  t_bwd_ev[1] = mid;
  t_bwd_ev[2] = stop;
  return FA_OK;
}

// Wait site of the last recorded timeout (0 if none); diagnostic only.
int fa_debug_last_wait_site(void) {
  int h[2] = {0, 0};
  if (cudaMemcpyFromSymbol(h, g_status, sizeof(h)) != cudaSuccess) return -1;
  return h[1];
}

}  // extern "C"
