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

// A [B, H, N, d] bf16 tensor with element strides s (d contiguous) viewed
// as 4-D (d, N, H, B); one box is 64 columns (128 bytes, the swizzle span) x
// 128 rows of one head.  Rows past N read as 0.
bool encode_map(CUtensorMap *map, const void *base, int B, int H, int N, int d, const Strides &s,
                unsigned box_rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(s.n) * 2, static_cast<cuuint64_t>(s.h) * 2,
                           static_cast<cuuint64_t>(s.b) * 2};
  cuuint32_t box[4] = {64, box_rows, 1, 1};
  cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// An [B, H, N, d] e4m3 tensor (one byte per element, element strides s)
// as 4-D (d, N, H, B); one box is a whole 128-byte row x box_rows rows of
// one head, 128-byte swizzle.  Rows past N read as 0.
bool encode_map_u8(CUtensorMap *map, const void *base, int B, int H, int N, int d, const Strides &s,
                   unsigned box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(s.n), static_cast<cuuint64_t>(s.h), static_cast<cuuint64_t>(s.b)};
  cuuint32_t box[4] = {128, box_rows, 1, 1};
  cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(base), dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

Strides contiguous(int H, int N, int d) {
  return Strides{static_cast<long long>(H) * N * d, static_cast<long long>(N) * d, d};
}

// A caller's strides made usable: the stride of an extent-1 dimension is
// never used, so it is replaced by a harmless valid value; then every
// stride must be positive and a multiple of 8 elements (16 bytes: TMA and
// the 16-byte row accesses).  False if the layout is not supported.
bool normalise(const int64_t *in, int B, int H, int N, int d, Strides *out) {
  if (!in) return false;
  Strides s{in[0], in[1], in[2]};
  if (N == 1) s.n = d;  // d is 64 or 128: a multiple of 8
  if (H == 1) s.h = s.n * N;
  if (B == 1) s.b = s.h * H;
  const long long lim = 1LL << 40;  // TMA strides are below 2^40 bytes
  for (long long v : {s.b, s.h, s.n})
    if (v <= 0 || (v & 7) || v >= lim / 2) return false;
  *out = s;
  return true;
}

// Address span [lo, hi) of the elements of a strided tensor.
void span(const void *base, int B, int H, int N, int d, const Strides &s, uintptr_t *lo, uintptr_t *hi) {
  const uintptr_t b0 = reinterpret_cast<uintptr_t>(base);
  const long long last = (B - 1) * s.b + (H - 1) * s.h + (N - 1) * s.n + d;
  *lo = b0;
  *hi = b0 + static_cast<uintptr_t>(last) * 2;
}

// No two elements of the tensor share an address (each stride covers the
// extent of the smaller ones): required of the outputs.
bool injective(int B, int H, int N, int d, const Strides &s) {
  struct Dim { long long stride, extent; } dims[3] = {{s.b, B}, {s.h, H}, {s.n, N}};
  for (int i = 0; i < 3; ++i)
    for (int j = i + 1; j < 3; ++j)
      if (dims[j].stride < dims[i].stride) {
        Dim t = dims[i];
        dims[i] = dims[j];
        dims[j] = t;
      }
  long long covered = d;  // the contiguous d elements
  for (const Dim &x : dims) {
    if (x.extent == 1) continue;
    if (x.stride < covered) return false;
    covered = x.stride * x.extent;
  }
  return true;
}

bool spans_overlap(uintptr_t alo, uintptr_t ahi, uintptr_t blo, uintptr_t bhi) { return alo < bhi && blo < ahi; }

// Two tensors with the same strides s, whose layout is injective (each
// stride at least the extent of the smaller ones), and bases `delta`
// elements apart share an element iff delta = sum_k a_k s_k + c with
// |a_k| < extent_k and |c| < d.  With nested strides only the two integer
// quotients next to delta / s_k can work at each level, so this small
// search is exact.  (It lets the slices of one packed buffer, such as the
// q, k, v gradients of a [B, N, 3, H, d] projection, be outputs together.)
bool lattice_hit(long long rem, const long long (*dims)[2], int k, int d) {
  if (k == 3) return rem > -d && rem < d;
  const long long st = dims[k][0], ext = dims[k][1];
  if (ext == 1) return lattice_hit(rem, dims, k + 1, d);  // only a = 0: skip it
  const long long q = rem / st;
  for (long long a = q - 1; a <= q + 1; ++a)
    if (a > -ext && a < ext && lattice_hit(rem - a * st, dims, k + 1, d)) return true;
  return false;
}

// Whether two tensors of [B, H, N, d] may share an element.  Exact when
// both have the same injective strides; otherwise whether their address
// spans overlap.
bool may_overlap(const void *a, const Strides &sa, const void *b, const Strides &sb, int B, int H, int N, int d) {
  uintptr_t alo, ahi, blo, bhi;
  span(a, B, H, N, d, sa, &alo, &ahi);
  span(b, B, H, N, d, sb, &blo, &bhi);
  if (!spans_overlap(alo, ahi, blo, bhi)) return false;
  const bool same = sa.b == sb.b && sa.h == sb.h && sa.n == sb.n;
  if (!same || !injective(B, H, N, d, sa)) return true;
  long long dims[3][2] = {{sa.b, B}, {sa.h, H}, {sa.n, N}};
  for (int i = 0; i < 3; ++i)  // descending strides
    for (int j = i + 1; j < 3; ++j)
      if (dims[j][0] > dims[i][0])
        for (int c = 0; c < 2; ++c) {
          const long long t = dims[i][c];
          dims[i][c] = dims[j][c];
          dims[j][c] = t;
        }
  const long long delta_bytes = static_cast<long long>(reinterpret_cast<uintptr_t>(b) - reinterpret_cast<uintptr_t>(a));
  if (delta_bytes % 2) return true;
  return lattice_hit(delta_bytes / 2, dims, 0, d);
}

int *status_ptr() {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
  return static_cast<int *>(p);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr long long kMaxGridX = 2147483647LL;  // largest x extent of a launch grid
// Causal backward: pairs of mirror blocks per CTA up to this many blocks per
// sequence (short sequences, where a CTA's fixed cost weighs most; longer
// ones keep one block per CTA, heaviest first, which fills the last wave
// better).  Measured with pairs at every length, B*N = 16384, H = 16, d =
// 128: dK/dV +2..+11 % up to N = 4096 and -1..-3 % above; dQ +2..+7 % up to
// N = 1024, even at 2048, -2..-6 % above.  With many heads (the head-by-head
// order below) the dQ kernel takes pairs up to kPairMaxBlocksKv blocks too:
// B4 H32 N4096 backward 1.690 -> 1.657 ms, while B4 H16 N4096 (heaviest
// first over all heads) ran 0.7 % slower with them.
constexpr int kPairMaxBlocksKv = 32, kPairMaxBlocksQ = 16;
// Non-causal backward: pairs of mirror blocks per CTA up to this many blocks
// (all CTAs have equal work either way; a pair pays one CTA's fixed cost for
// two blocks).  Measured, B*N = 16384, H = 16: d = 128 +4 % at N = 512, +3 %
// at 1024, 0 at 2048, -2 % at 4096; d = 64 +10 %, +5 %, +1 %, -1 %.
constexpr int kPairMaxBlocksNonCausal = 16;
// Longest sequence, in 256-row tiles, for which the batched forward runs
// persistent CTAs.  Measured against one CTA per tile (forward only, L2
// flushed, B*N = 16384, H = 16):
//   d = 64:   +27 % at N = 512, +15 % at 1024, +7 % at 2048, +2.5 % at 4096,
//             +0.3 % at 8192, -0.7 % at 16384; causal +8.5 % at 512, +3 %
//             at 2048, -1 % at 8192;
//   d = 128:  +14 % at 512, +8 % at 1024, +2 % at 2048, -2 % at 4096, -5 %
//             at 8192; causal +12 %, +9 %, +5 %, +3 % (N = 4096; +3.7 % at
//             B4 H32), 0 % at 8192, -3 % at 16384.
int persist_max_qblk(int d, bool causal) {
  if (d == 64) return causal ? 16 : 32;
  return causal ? 16 : 8;
}

// Host-side checks shared by both passes; no CUDA call happens before them.
fa_status_t check_common(int B, int H, int N, int d, int causal, float scale) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARGUMENT;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARGUMENT;
  if (d != 64 && d != 128) return d < 1 ? FA_ERR_INVALID_ARGUMENT : FA_ERR_UNSUPPORTED;
  // The backward launches one CTA per (head, block of 128 rows): that count
  // must fit a grid's x extent.  Within it B*H*N < 2^38, so the element
  // count below cannot overflow.
  const long long bh = static_cast<long long>(B) * H;
  if (bh * ((N + 127) / 128) > kMaxGridX) return FA_ERR_INVALID_ARGUMENT;
  // TMA addresses a tensor with byte strides below 2^40: at most 2^39 bf16
  // elements (1 TiB) per tensor, more than a GPU's memory holds.
  const long long elems = bh * N * d;
  if (elems >= (1LL << 39)) return FA_ERR_INVALID_ARGUMENT;
  return FA_OK;
}

// Events the next fa_bwd call of this thread records around its kernels.
thread_local cudaEvent_t t_bwd_ev[3] = {nullptr, nullptr, nullptr};

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }


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

}  // extern "C"

namespace fa {
namespace {

// The row axis of the tensors.  Batched: B slots of N rows each.  Packed
// (cu != null): one slot of T rows holding the B sequences back to back,
// N the longest; the tensors' batch stride is then unused (0 in the kernels).
struct RowAxis {
  int B, N;
  const int *cu;
  int T;
  int slots() const { return cu ? 1 : B; }
  int rows() const { return cu ? T : N; }
};

// SMs of the current device (cached per host thread and device), 0 if unknown.
int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  thread_local int cached[64] = {0};
  if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

fa_status_t fwd_impl(const void *q, const Strides &sq, const void *k, const Strides &sk, const void *v,
                     const Strides &sv, void *o, const Strides &so, float *lse, const RowAxis &ax, int H, int d,
                     int causal, float scale, cudaStream_t stream) {
  const int B = ax.B, N = ax.N, SB = ax.slots(), R = ax.rows();
  fa_status_t st = check_common(B, H, N, d, causal, scale);
  if (st == FA_OK && ax.cu) st = check_common(1, H, R, d, causal, scale);
  if (st != FA_OK) return st;
  const void *ptrs[5] = {q, k, v, o, lse};
  for (const void *x : ptrs)
    if (!x || !aligned16(x)) return FA_ERR_INVALID_ARGUMENT;
  if (!injective(SB, H, R, d, so)) return FA_ERR_INVALID_ARGUMENT;
  const size_t lb = static_cast<size_t>(SB) * H * R * 4;
  uintptr_t olo, ohi, llo = reinterpret_cast<uintptr_t>(lse), lhi = llo + lb;
  span(o, SB, H, R, d, so, &olo, &ohi);
  const void *ins[3] = {q, k, v};
  const Strides *ins_s[3] = {&sq, &sk, &sv};
  for (int i = 0; i < 3; ++i) {
    uintptr_t lo, hi;
    span(ins[i], SB, H, R, d, *ins_s[i], &lo, &hi);
    if (may_overlap(ins[i], *ins_s[i], o, so, SB, H, R, d) || spans_overlap(lo, hi, llo, lhi))
      return FA_ERR_INVALID_ARGUMENT;
  }
  if (spans_overlap(olo, ohi, llo, lhi)) return FA_ERR_INVALID_ARGUMENT;

  CUtensorMap tq, tk, tv;
  if (!encode_map(&tq, q, SB, H, R, d, sq) || !encode_map(&tk, k, SB, H, R, d, sk) ||
      !encode_map(&tv, v, SB, H, R, d, sv))
    return FA_ERR_CUDA;
  FwdParams p{};
  p.o = static_cast<__nv_bfloat16 *>(o);
  p.lse = lse;
  p.so = so;
  if (ax.cu) p.so.b = 0;
  p.H = H;
  p.cu_seqlens = ax.cu;
  p.T = R;
  p.lse_b = ax.cu ? 0 : static_cast<long long>(H) * N;
  p.lse_h = R;
  p.status = status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  p.N = N;
  p.BH = B * H;
  p.num_qblk = (N + 255) / 256;
  // The batched forward of short sequences runs persistent CTAs (one per
  // SM) when there are more 256-row tiles than SMs.
  if (!ax.cu && p.num_qblk <= persist_max_qblk(d, causal != 0)) {
    const int sms = sm_count();
    if (sms > 0 && static_cast<long long>(p.BH) * p.num_qblk > sms) p.persist_ctas = sms;
  }
  p.scale_log2 = scale * 1.4426950408889634f;
  p.neg = scale < 0.0f ? 1 : 0;
  return launch_fwd(d, causal != 0, tq, tk, tv, p, stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status_t bwd_impl(const void *q, const Strides &sq, const void *k, const Strides &sk, const void *v,
                     const Strides &sv, const void *o, const Strides &so, const void *dO, const Strides &sdo,
                     const float *lse, void *dq, const Strides &sdq, void *dk, const Strides &sdk, void *dv,
                     const Strides &sdv, const RowAxis &ax, int H, int d, int causal, float scale, void *workspace,
                     size_t workspace_bytes, cudaStream_t stream, bool concurrent = true) {
  const int B = ax.B, N = ax.N, SB = ax.slots(), R = ax.rows();
  fa_status_t st = check_common(B, H, N, d, causal, scale);
  if (st == FA_OK && ax.cu) st = check_common(1, H, R, d, causal, scale);
  if (st != FA_OK) return st;
  const void *ptrs[9] = {q, k, v, o, dO, lse, dq, dk, dv};
  for (const void *x : ptrs)
    if (!x || !aligned16(x)) return FA_ERR_INVALID_ARGUMENT;
  void *outs[3] = {dq, dk, dv};
  const Strides *outs_s[3] = {&sdq, &sdk, &sdv};
  for (int i = 0; i < 3; ++i)
    if (!injective(SB, H, R, d, *outs_s[i])) return FA_ERR_INVALID_ARGUMENT;
  uintptr_t in_lo[6], in_hi[6], out_lo[3], out_hi[3];
  const void *ins[5] = {q, k, v, o, dO};
  const Strides *ins_s[5] = {&sq, &sk, &sv, &so, &sdo};
  for (int i = 0; i < 5; ++i) span(ins[i], SB, H, R, d, *ins_s[i], &in_lo[i], &in_hi[i]);
  in_lo[5] = reinterpret_cast<uintptr_t>(lse);
  in_hi[5] = in_lo[5] + static_cast<size_t>(SB) * H * R * 4;
  for (int i = 0; i < 3; ++i) span(outs[i], SB, H, R, d, *outs_s[i], &out_lo[i], &out_hi[i]);
  for (int j = 0; j < 3; ++j) {
    for (int i = 0; i < 5; ++i)
      if (may_overlap(ins[i], *ins_s[i], outs[j], *outs_s[j], SB, H, R, d)) return FA_ERR_INVALID_ARGUMENT;
    if (spans_overlap(in_lo[5], in_hi[5], out_lo[j], out_hi[j])) return FA_ERR_INVALID_ARGUMENT;  // lse
  }
  for (int i = 0; i < 3; ++i)
    for (int j = i + 1; j < 3; ++j)
      if (may_overlap(outs[i], *outs_s[i], outs[j], *outs_s[j], SB, H, R, d)) return FA_ERR_INVALID_ARGUMENT;
  const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
  if (workspace) {
    if (workspace_bytes < need) return FA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_INVALID_ARGUMENT;
    const uintptr_t wlo = reinterpret_cast<uintptr_t>(workspace), whi = wlo + need;
    for (int i = 0; i < 6; ++i)
      if (spans_overlap(in_lo[i], in_hi[i], wlo, whi)) return FA_ERR_INVALID_ARGUMENT;
    for (int j = 0; j < 3; ++j)
      if (spans_overlap(out_lo[j], out_hi[j], wlo, whi)) return FA_ERR_INVALID_ARGUMENT;
  }

  const int BH = B * H;
  CUtensorMap tq, tk, tv, tdo;
  if (!encode_map(&tq, q, SB, H, R, d, sq) || !encode_map(&tk, k, SB, H, R, d, sk) ||
      !encode_map(&tv, v, SB, H, R, d, sv) || !encode_map(&tdo, dO, SB, H, R, d, sdo))
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
  p.sq = sq;
  p.so = so;
  p.sdo = sdo;
  p.sdq = sdq;
  p.sdk = sdk;
  p.sdv = sdv;
  if (ax.cu) p.sq.b = p.so.b = p.sdo.b = p.sdq.b = p.sdk.b = p.sdv.b = 0;
  p.H = H;
  p.cu_seqlens = ax.cu;
  p.T = R;
  p.lse_b = ax.cu ? 0 : static_cast<long long>(H) * N;
  p.lse_h = R;
  p.status = status_ptr();
  p.N = N;
  p.BH = BH;
  p.num_blk = (N + 127) / 128;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  // Causal: head by head when the heaviest block (num_blk blocks of work)
  // is under a tenth of each SM's share (B*H*num_blk*(num_blk+1)/2 over the
  // 152 SMs), i.e. many short blocks: then L2 reuse within a head beats the
  // strict heaviest-first order (measured: B8 H16 N4096 +5..9 %, B1 H16
  // N16384 -2 %).
  p.head_major = (static_cast<long long>(BH) * (p.num_blk + 1) > 3040) ? 1 : 0;
  if (causal) {
    p.pairs_kv = (p.num_blk <= kPairMaxBlocksKv) ? 1 : 0;
    p.pairs_q = (p.num_blk <= kPairMaxBlocksQ || (p.head_major && p.num_blk <= kPairMaxBlocksKv)) ? 1 : 0;
  } else {
    p.pairs_kv = p.pairs_q = (p.num_blk <= kPairMaxBlocksNonCausal) ? 1 : 0;
  }
  fa_status_t rc = FA_OK;
  const cudaEvent_t ev[3] = {t_bwd_ev[0], t_bwd_ev[1], t_bwd_ev[2]};
  t_bwd_ev[0] = t_bwd_ev[1] = t_bwd_ev[2] = nullptr;
  if (!p.status ||
      launch_bwd(d, causal != 0, tq, tk, tv, tdo, p, stream, ev[0] ? ev : nullptr, concurrent) != cudaSuccess)
    rc = FA_ERR_CUDA;
  if (owned && cudaFreeAsync(ws, stream) != cudaSuccess) rc = FA_ERR_CUDA;
  return rc;
}

// ------------------------------------------------------------------ FP8 forward

fa_status_t fwd_fp8_impl(const void *q8, const void *k8, const void *v8, float sq, float sk, float sv, void *o,
                         float *lse, int B, int H, int N, int d, int causal, float scale, cudaStream_t stream) {
  fa_status_t st = check_common(B, H, N, d, causal, scale);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if (!std::isfinite(sq) || !std::isfinite(sk) || !std::isfinite(sv)) return FA_ERR_INVALID_ARGUMENT;
  const void *ptrs[5] = {q8, k8, v8, o, lse};
  for (const void *x : ptrs)
    if (!x || !aligned16(x)) return FA_ERR_INVALID_ARGUMENT;
  const size_t n8 = static_cast<size_t>(B) * H * N * d;  // bytes of each e4m3 input
  const uintptr_t olo = reinterpret_cast<uintptr_t>(o), ohi = olo + 2 * n8;
  const uintptr_t llo = reinterpret_cast<uintptr_t>(lse), lhi = llo + static_cast<size_t>(B) * H * N * 4;
  const void *ins[3] = {q8, k8, v8};
  for (const void *x : ins) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(x), hi = lo + n8;
    if (spans_overlap(lo, hi, olo, ohi) || spans_overlap(lo, hi, llo, lhi)) return FA_ERR_INVALID_ARGUMENT;
  }
  if (spans_overlap(olo, ohi, llo, lhi)) return FA_ERR_INVALID_ARGUMENT;
  const Strides s = contiguous(H, N, d);
  CUtensorMap tq, tk, tv;
  if (!encode_map_u8(&tq, q8, B, H, N, d, s, 128) || !encode_map_u8(&tk, k8, B, H, N, d, s, 128) ||
      !encode_map_u8(&tv, v8, B, H, N, d, s, 128))
    return FA_ERR_CUDA;
  Fp8FwdParams p{};
  p.o = static_cast<__nv_bfloat16 *>(o);
  p.lse = lse;
  p.so = s;
  p.H = H;
  p.status = status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  p.N = N;
  p.BH = B * H;
  p.num_qblk = (N + 255) / 256;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * sq * sk * 1.4426950408889634);
  p.v_scale = sv;
  p.neg = p.scale_log2 < 0.0f ? 1 : 0;
  return launch_fwd_fp8(causal != 0, tq, tk, tv, p, stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// ------------------------------------------------------------------ decode

constexpr int kDecodeMaxNq = 8;
constexpr int kDecodeModelCtas = 152;  // GB300's SMs: the persistent grid the split plan is made for
constexpr int kDecodeMaxSplits = 64;

struct DecodePlan {
  int chunk, splits;
};

// Chunk size (in 128-key tiles) for the persistent decode grid: the one
// whose round-robin assignment of (chunk, head) items to kDecodeModelCtas
// CTAs gives the smallest busiest-CTA load, counting each item's fixed
// merge cost as a quarter tile; ties go to larger chunks (fewer partials).
// A function of the shape alone, so the workspace size is too.
DecodePlan plan_decode(long long BH, int tiles) {
  thread_local long long last_bh = -1;
  thread_local int last_tiles = -1;
  thread_local DecodePlan last{1, 1};
  if (BH == last_bh && tiles == last_tiles) return last;
  const double alpha = 0.25;
  DecodePlan best{tiles, 1};
  double best_cost = 1e300;
  int prev = -1;
  for (int sp = 1; sp <= tiles && sp <= kDecodeMaxSplits; ++sp) {
    const int chunk = (tiles + sp - 1) / sp;
    if (chunk == prev) continue;
    prev = chunk;
    const int splits = (tiles + chunk - 1) / chunk;
    const int tail = tiles - (splits - 1) * chunk;
    const long long F = (splits - 1) * BH, I = splits * BH;
    const long long G = I < kDecodeModelCtas ? I : kDecodeModelCtas;
    double cost = 0.0;
    for (long long j = 0; j < G; ++j) {
      const long long nf = F / G + (j < F % G ? 1 : 0);
      const long long ni = I / G + (j < I % G ? 1 : 0);
      const double load = nf * (chunk + alpha) + (ni - nf) * (tail + alpha);
      cost = load > cost ? load : cost;
    }
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = DecodePlan{chunk, splits};
    }
  }
  last_bh = BH;
  last_tiles = tiles;
  last = best;
  return best;
}

fa_status_t check_decode(int B, int H, int Nq, int Nk, int d, int causal, float scale) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARGUMENT;
  if (Nq > kDecodeMaxNq) return FA_ERR_INVALID_ARGUMENT;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARGUMENT;
  if (d != 64 && d != 128) return d < 1 ? FA_ERR_INVALID_ARGUMENT : FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H >= (1LL << 24)) return FA_ERR_INVALID_ARGUMENT;
  if (Nk > (1 << 30)) return FA_ERR_INVALID_ARGUMENT;
  return FA_OK;
}

size_t decode_workspace(int B, int H, int Nq, int Nk, int d) {
  const long long BH = static_cast<long long>(B) * H;
  const DecodePlan pl = plan_decode(BH, (Nk + 127) / 128);
  if (pl.splits == 1) return 0;
  const size_t parts = static_cast<size_t>(BH) * pl.splits * Nq;
  return round256(parts * d * 4) + round256(parts * 4);
}

fa_status_t decode_impl(const void *q, const int64_t *q_strides, const void *k, const int64_t *k_strides,
                        const void *v, const int64_t *v_strides, void *o, const int64_t *o_strides, float *lse,
                        const int *cache_len, int B, int H, int Nq, int Nk, int d, int causal, float scale,
                        void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  fa_status_t st = check_decode(B, H, Nq, Nk, d, causal, scale);
  if (st != FA_OK) return st;
  const void *ptrs[5] = {q, k, v, o, lse};
  for (const void *x : ptrs)
    if (!x || !aligned16(x)) return FA_ERR_INVALID_ARGUMENT;
  if (cache_len && (reinterpret_cast<uintptr_t>(cache_len) & 3u)) return FA_ERR_INVALID_ARGUMENT;
  Strides sq, sk, sv, so;
  if (!normalise(q_strides, B, H, Nq, d, &sq) || !normalise(k_strides, B, H, Nk, d, &sk) ||
      !normalise(v_strides, B, H, Nk, d, &sv) || !normalise(o_strides, B, H, Nq, d, &so))
    return FA_ERR_INVALID_ARGUMENT;
  if (!injective(B, H, Nq, d, so)) return FA_ERR_INVALID_ARGUMENT;
  // no output may share memory with an input, the other output or the workspace
  uintptr_t lo[6], hi[6];  // q, k, v, cache_len, o, lse
  span(q, B, H, Nq, d, sq, &lo[0], &hi[0]);
  span(k, B, H, Nk, d, sk, &lo[1], &hi[1]);
  span(v, B, H, Nk, d, sv, &lo[2], &hi[2]);
  lo[3] = reinterpret_cast<uintptr_t>(cache_len);
  hi[3] = cache_len ? lo[3] + static_cast<size_t>(B) * 4 : lo[3];
  span(o, B, H, Nq, d, so, &lo[4], &hi[4]);
  lo[5] = reinterpret_cast<uintptr_t>(lse);
  hi[5] = lo[5] + static_cast<size_t>(B) * H * Nq * 4;
  for (int out = 4; out < 6; ++out)
    for (int i = 0; i < 6; ++i) {
      if (i == out || (out == 5 && i == 4)) continue;
      if (out == 4 && i == 0) {
        if (may_overlap(q, sq, o, so, B, H, Nq, d)) return FA_ERR_INVALID_ARGUMENT;
      } else if (spans_overlap(lo[i], hi[i], lo[out], hi[out])) {
        return FA_ERR_INVALID_ARGUMENT;
      }
    }
  const long long BH = static_cast<long long>(B) * H;
  const int tiles = (Nk + 127) / 128;
  const DecodePlan pl = plan_decode(BH, tiles);
  const size_t need = decode_workspace(B, H, Nq, Nk, d);
  if (workspace && need) {
    if (workspace_bytes < need) return FA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_INVALID_ARGUMENT;
    const uintptr_t wlo = reinterpret_cast<uintptr_t>(workspace), whi = wlo + need;
    for (int i = 0; i < 6; ++i)
      if (spans_overlap(lo[i], hi[i], wlo, whi)) return FA_ERR_INVALID_ARGUMENT;
  }

  CUtensorMap tk, tv, tq;  // q: boxes of 16 rows, the rows past Nq read as zeros
  if (!encode_map(&tk, k, B, H, Nk, d, sk) || !encode_map(&tv, v, B, H, Nk, d, sv) ||
      !encode_map(&tq, q, B, H, Nq, d, sq, 16))
    return FA_ERR_CUDA;
  const int sms = sm_count();
  if (sms <= 0) return FA_ERR_CUDA;
  void *ws = need ? workspace : nullptr;
  bool owned = false;
  if (need && !ws) {
    if (cudaMallocAsync(&ws, need, stream) != cudaSuccess) return FA_ERR_CUDA;
    owned = true;
  }
  DecodeParams p{};
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.o = static_cast<__nv_bfloat16 *>(o);
  p.lse = lse;
  p.sq = sq;
  p.so = so;
  p.cache_len = cache_len;
  const size_t parts = static_cast<size_t>(BH) * pl.splits * Nq;
  p.part_o = need ? static_cast<float *>(ws) : nullptr;
  p.part_lse = need ? reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + round256(parts * d * 4)) : nullptr;
  p.status = status_ptr();
  p.H = H;
  p.BH = static_cast<int>(BH);
  p.Nq = Nq;
  p.Nk = Nk;
  p.chunk = pl.chunk;
  p.splits = pl.splits;
  p.items = static_cast<int>(BH * pl.splits);
  p.causal = causal;
  p.scale_log2 = scale * 1.4426950408889634f;
  const int grid = p.items < sms ? p.items : sms;
  fa_status_t rc = FA_OK;
  if (!p.status || launch_decode(d, tk, tv, tq, p, grid, stream) != cudaSuccess) rc = FA_ERR_CUDA;
  if (owned && cudaFreeAsync(ws, stream) != cudaSuccess) rc = FA_ERR_CUDA;
  return rc;
}

}  // namespace
}  // namespace fa

extern "C" {

fa_status_t fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int N, int d,
                   int causal, float scale, cudaStream_t stream) {
  const Strides s = contiguous(H, N, d);
  return fwd_impl(q, s, k, s, v, s, o, s, lse, RowAxis{B, N, nullptr, 0}, H, d, causal, scale, stream);
}

fa_status_t fa_fwd_strided(const void *q, const int64_t *q_strides, const void *k, const int64_t *k_strides,
                           const void *v, const int64_t *v_strides, void *o, const int64_t *o_strides, float *lse,
                           int B, int H, int N, int d, int causal, float scale, cudaStream_t stream) {
  fa_status_t st = check_common(B, H, N, d, causal, scale);
  if (st != FA_OK) return st;
  Strides sq, sk, sv, so;
  if (!normalise(q_strides, B, H, N, d, &sq) || !normalise(k_strides, B, H, N, d, &sk) ||
      !normalise(v_strides, B, H, N, d, &sv) || !normalise(o_strides, B, H, N, d, &so))
    return FA_ERR_INVALID_ARGUMENT;
  return fwd_impl(q, sq, k, sk, v, sv, o, so, lse, RowAxis{B, N, nullptr, 0}, H, d, causal, scale, stream);
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (check_common(B, H, N, d, 0, 1.0f) != FA_OK) return 0;
  const size_t padded_rows = static_cast<size_t>(B) * H * ((N + 127) / 128) * 128;
  return 2 * round256(padded_rows * 4);
}

fa_status_t fa_bwd(const void *q, const void *k, const void *v, const void *o, const void *dO, const float *lse,
                   void *dq, void *dk, void *dv, int B, int H, int N, int d, int causal, float scale, void *workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
  const Strides s = contiguous(H, N, d);
  return bwd_impl(q, s, k, s, v, s, o, s, dO, s, lse, dq, s, dk, s, dv, s, RowAxis{B, N, nullptr, 0}, H, d, causal,
                  scale, workspace, workspace_bytes, stream);
}

fa_status_t fa_bwd_sequential(const void *q, const void *k, const void *v, const void *o, const void *dO,
                              const float *lse, void *dq, void *dk, void *dv, int B, int H, int N, int d,
                              int causal, float scale, void *workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
  const Strides s = contiguous(H, N, d);
  return bwd_impl(q, s, k, s, v, s, o, s, dO, s, lse, dq, s, dk, s, dv, s, RowAxis{B, N, nullptr, 0}, H, d, causal,
                  scale, workspace, workspace_bytes, stream, false);
}

fa_status_t fa_bwd_strided(const void *q, const int64_t *q_strides, const void *k, const int64_t *k_strides,
                           const void *v, const int64_t *v_strides, const void *o, const int64_t *o_strides,
                           const void *dO, const int64_t *dO_strides, const float *lse, void *dq,
                           const int64_t *dq_strides, void *dk, const int64_t *dk_strides, void *dv,
                           const int64_t *dv_strides, int B, int H, int N, int d, int causal, float scale,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  fa_status_t st = check_common(B, H, N, d, causal, scale);
  if (st != FA_OK) return st;
  Strides s[8];
  const int64_t *in[8] = {q_strides, k_strides, v_strides, o_strides, dO_strides, dq_strides, dk_strides, dv_strides};
  for (int i = 0; i < 8; ++i)
    if (!normalise(in[i], B, H, N, d, &s[i])) return FA_ERR_INVALID_ARGUMENT;
  return bwd_impl(q, s[0], k, s[1], v, s[2], o, s[3], dO, s[4], lse, dq, s[5], dk, s[6], dv, s[7],
                  RowAxis{B, N, nullptr, 0}, H, d, causal, scale, workspace, workspace_bytes, stream);
}

// Packed sequences: strides arrays of two (row, head); the batch stride of
// the one slot is derived (never used by the kernels).
static bool normalise_packed(const int64_t *in, int H, int T, int d, Strides *out) {
  if (!in) return false;
  const int64_t full[3] = {0, in[1], in[0]};
  if (!normalise(full, 1, H, T, d, out)) return false;
  return true;
}

fa_status_t fa_fwd_varlen(const void *q, const int64_t *q_strides, const void *k, const int64_t *k_strides,
                          const void *v, const int64_t *v_strides, void *o, const int64_t *o_strides, float *lse,
                          const int *cu_seqlens, int B, int H, int T, int max_seqlen, int d, int causal, float scale,
                          cudaStream_t stream) {
  fa_status_t st = check_common(B, H, max_seqlen, d, causal, scale);
  if (st == FA_OK) st = check_common(1, H, T, d, causal, scale);
  if (st != FA_OK) return st;
  if (!cu_seqlens || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return FA_ERR_INVALID_ARGUMENT;
  Strides sq, sk, sv, so;
  if (!normalise_packed(q_strides, H, T, d, &sq) || !normalise_packed(k_strides, H, T, d, &sk) ||
      !normalise_packed(v_strides, H, T, d, &sv) || !normalise_packed(o_strides, H, T, d, &so))
    return FA_ERR_INVALID_ARGUMENT;
  return fwd_impl(q, sq, k, sk, v, sv, o, so, lse, RowAxis{B, max_seqlen, cu_seqlens, T}, H, d, causal, scale,
                  stream);
}

fa_status_t fa_bwd_varlen(const void *q, const int64_t *q_strides, const void *k, const int64_t *k_strides,
                          const void *v, const int64_t *v_strides, const void *o, const int64_t *o_strides,
                          const void *dO, const int64_t *dO_strides, const float *lse, void *dq,
                          const int64_t *dq_strides, void *dk, const int64_t *dk_strides, void *dv,
                          const int64_t *dv_strides, const int *cu_seqlens, int B, int H, int T, int max_seqlen,
                          int d, int causal, float scale, void *workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
  fa_status_t st = check_common(B, H, max_seqlen, d, causal, scale);
  if (st == FA_OK) st = check_common(1, H, T, d, causal, scale);
  if (st != FA_OK) return st;
  if (!cu_seqlens || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return FA_ERR_INVALID_ARGUMENT;
  Strides s[8];
  const int64_t *in[8] = {q_strides, k_strides, v_strides, o_strides, dO_strides, dq_strides, dk_strides, dv_strides};
  for (int i = 0; i < 8; ++i)
    if (!normalise_packed(in[i], H, T, d, &s[i])) return FA_ERR_INVALID_ARGUMENT;
  return bwd_impl(q, s[0], k, s[1], v, s[2], o, s[3], dO, s[4], lse, dq, s[5], dk, s[6], dv, s[7],
                  RowAxis{B, max_seqlen, cu_seqlens, T}, H, d, causal, scale, workspace, workspace_bytes, stream);
}

fa_status_t fa_fwd_fp8(const void *q8, const void *k8, const void *v8, float q_scale, float k_scale,
                       float v_scale, void *o, float *lse, int B, int H, int N, int d, int causal, float scale,
                       cudaStream_t stream) {
  return fwd_fp8_impl(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, B, H, N, d, causal, scale, stream);
}

size_t fa_decode_workspace_bytes(int B, int H, int Nq, int Nk, int d) {
  if (check_decode(B, H, Nq, Nk, d, 0, 1.0f) != FA_OK) return 0;
  return decode_workspace(B, H, Nq, Nk, d);
}

fa_status_t fa_fwd_decode(const void *q, const int64_t *q_strides, const void *k, const int64_t *k_strides,
                          const void *v, const int64_t *v_strides, void *o, const int64_t *o_strides, float *lse,
                          const int *cache_seqlens, int B, int H, int Nq, int Nk, int d, int causal, float scale,
                          void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  return decode_impl(q, q_strides, k, k_strides, v, v_strides, o, o_strides, lse, cache_seqlens, B, H, Nq, Nk, d,
                     causal, scale, workspace, workspace_bytes, stream);
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
