// fa_noalloc.cu -- fa_bwd_noalloc: the backward pass for callers that must
// not allocate device memory.
//
// Some callers cannot let a library allocate: a framework that owns every
// device allocation through its own memory manager, or a process whose
// device memory is planned up front and must not grow or fragment while it
// runs.  Such callers can neither hand fa_bwd a workspace taken with
// cudaMalloc nor let it take one with cudaMallocAsync.  fa_bwd_noalloc
// gives them the same backward pass with its scratch (the per-row D and
// logsumexp arrays) in a fixed array of this library's own device memory.
// Its two main kernels run one after the other on the caller's stream (no
// side stream is created for it).
//
// The array is a file-scope __device__ variable of FA_NOALLOC_SCRATCH_BYTES
// bytes: every GPU that loads the library holds it until the process
// exits.  In host code its name only stands in for the device object, so
// every call looks up the array's device address on the current device with
// cudaGetSymbolAddress (a host-side query: it enqueues nothing).  The
// address is not cached: after cudaDeviceReset, or under another context on
// the same device, the module is loaded again and the array may move.  The
// first lookup in a process may load the module.
//
// Every call uses the same array and leaves its last contents there.
// Nothing in it has to start at zero: the first kernel of each call writes
// every element that the later kernels of that call read.  Calls whose work
// overlaps on the GPU (different streams, or different host threads, on the
// same device) race on the array; callers must order them.

#include <cmath>
#include <cstdint>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array in the current context.
fa_status_t scratch_address(void **out) {
  void *ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return FA_ERR_CUDA;
  *out = ptr;
  return FA_OK;
}

}  // namespace

extern "C" fa_status_t fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o, const void *dO,
                                      const float *lse, void *dq, void *dk, void *dv, int B, int H, int N, int d,
                                      int causal, float scale, cudaStream_t stream) {
  // Host-side checks first (no CUDA call before them): pointers, flags and
  // scale, then the size of the scratch the call needs.
  // fa_bwd_workspace_bytes returns 0 for sizes fa_bwd rejects; fa_bwd
  // reports those with its own code.
  const void *ptrs[9] = {q, k, v, o, dO, lse, dq, dk, dv};
  for (const void *x : ptrs)
    if (!x || (reinterpret_cast<uintptr_t>(x) & 15u)) return FA_ERR_INVALID_ARGUMENT;
  if ((causal != 0 && causal != 1) || !std::isfinite(scale)) return FA_ERR_INVALID_ARGUMENT;
  const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
  if (need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;
  if (need == 0)  // invalid sizes: let fa_bwd name the error, without touching the device
    return fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, causal, scale, nullptr, 0, stream);
  void *scratch = nullptr;
  const fa_status_t st = scratch_address(&scratch);
  if (st != FA_OK) return st;
  return fa_bwd_sequential(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, causal, scale, scratch,
                           FA_NOALLOC_SCRATCH_BYTES, stream);
}
