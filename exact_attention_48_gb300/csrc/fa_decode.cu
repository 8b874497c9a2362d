// fa_decode.cu -- forward pass for decoding: a few new query rows per head
// against a long key/value cache.
//
// With Nq <= 8 query rows the work per key is a handful of dot products and
// AXPYs while every key costs 4*d bytes of cache traffic, so the pass is
// bound by HBM bandwidth, not by arithmetic: it runs on the CUDA cores (fp32
// FMA) with the cache streamed through shared memory by TMA, and no tensor
// core product is formed.  The keys of each head are split into chunks
// ("split-KV"); each chunk yields a partial result normalised over its own
// keys plus its logsumexp, and a second small kernel merges the partials of
// a head with the same running-max correction the tiled forward uses across
// key blocks (page "FlashAttention" (urworte.de), "Methodische Grundlagen":
// "Fortlaufende Normierung").  A persistent grid of one CTA per SM walks the
// (head, chunk) items; its producer warp keeps loading the next items'
// tiles while the consumer warps finish the current one.
//
// CTA: 8 consumer warps in two groups of 4 (group g takes the CTA's tiles
// with counter parity g, so two tiles are computed at once) and 1 producer
// warp.  Each group has its own full/empty barrier per stage: with an odd
// number of stages a stage is used by the two groups in turn, and a group
// must only ever wait for the next use of a stage that is its own (a shared
// barrier would let a group wait two phases ahead, where a parity wait
// cannot tell the phase it wants from the one before).  In a 128-key tile, warp w of a group owns keys 32*(w%4) + lane for
// the scores (lane = key: the lane reads its key row through the 128-byte
// swizzle without bank conflicts) and the same 32 keys for P*V, where each
// lane owns d/32 columns of O and receives p by shuffle.

#include <cstdint>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kDecThreads = 288;  // 8 consumer warps + 1 producer warp
constexpr int kDecConsumers = 256;
constexpr int kDecTileKeys = 128;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -INFINITY;

template <int D, int NQ>
struct DecodeLayout {
  static constexpr int kSlabs = D / 64;
  static constexpr int kSlabBytes = kDecTileKeys * 128;      // 128 rows x 64 bf16
  static constexpr int kTileBytes = kSlabs * kSlabBytes;     // K (or V) of one tile
  static constexpr int kStageBytes = 2 * kTileBytes;         // K then V
  static constexpr int kStages = D == 128 ? 3 : 6;
  static constexpr int kOffObuf = kStages * kStageBytes;     // [4][NQ][D] fp32
  static constexpr int kOffQ = kOffObuf + 4 * NQ * D * 4;    // [NQ][D] fp32, pre-scaled
  static constexpr int kOffStats = kOffQ + NQ * D * 4;       // m[4][NQ], l[4][NQ]
  static constexpr int kOffBar = kOffStats + 2 * 4 * NQ * 4; // full[2][S], empty[2][S]
  static constexpr int kOffMisc = kOffBar + 4 * kStages * 8; // abort flag
  static constexpr int kSmemBytes = kOffMisc + 16;
  static constexpr int kSmemRequest = kSmemBytes + 1024;     // 1 KB alignment slack
  static_assert(kSmemRequest <= 227 * 1024, "decode layout exceeds shared memory");
  static_assert(kOffBar % 8 == 0, "barriers need 8-byte alignment");
};

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

__device__ __forceinline__ float warp_max(float x) { return warp_max_f32(x); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Weight 2^(m - M) of a partial state with max m under the merged max M
// (0 for an empty state, m = -inf).
__device__ __forceinline__ float rescale(float m, float M) { return m == kNegInf ? 0.0f : ex2(m - M); }

// Tile c of a CTA goes to stage c % S and group c & 1.  Its use of the
// stage is the (c / S)-th; the group's own uses of that stage are every
// use (S even: a stage always serves the same group) or every other use
// (S odd: the groups alternate).  The ordinal of tile c among its group's
// uses of its stage is the phase it occupies on the group's barriers.
template <int S>
__device__ __forceinline__ uint32_t group_phase(int c) {
  const int u = c / S;
  return static_cast<uint32_t>(S % 2 == 0 ? u : u >> 1);
}

struct DecodeItem {
  int bh, b, h, split, len, t0, t1;
};

__device__ __forceinline__ DecodeItem decode_item(const DecodeParams &p, int it) {
  DecodeItem x;
  x.split = it / p.BH;
  x.bh = it - x.split * p.BH;
  x.b = x.bh / p.H;
  x.h = x.bh - x.b * p.H;
  int len = p.Nk;
  if (p.cache_len) {
    len = p.cache_len[x.b];
    len = len < 0 ? 0 : (len > p.Nk ? p.Nk : len);
  }
  x.len = len;
  const int tiles_b = (len + kDecTileKeys - 1) / kDecTileKeys;
  x.t0 = x.split * p.chunk;
  x.t1 = min(x.t0 + p.chunk, tiles_b);
  if (x.t1 < x.t0) x.t1 = x.t0;
  return x;
}

template <int D, int NQ>
__global__ void __launch_bounds__(kDecThreads, 1)
    fa_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const DecodeParams p) {
  using L = DecodeLayout<D, NQ>;
  constexpr int S = L::kStages;
  constexpr int CPL = D / 32;  // O columns per lane

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kOffBar);  // [group][stage]
  uint64_t *empty = full + 2 * S;                                     // [group][stage]
  float *obuf = reinterpret_cast<float *>(smem + L::kOffObuf);
  float *qbuf = reinterpret_cast<float *>(smem + L::kOffQ);
  float *stat_m = reinterpret_cast<float *>(smem + L::kOffStats);
  float *stat_l = stat_m + 4 * NQ;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc);
  const WaitCtl ctl{abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2 * S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);  // the 4 warps of the group
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int c = 0;
      bool ok = true;
      for (int it = blockIdx.x; ok && it < p.items; it += gridDim.x) {
        const DecodeItem x = decode_item(p, it);
        for (int t = x.t0; t < x.t1; ++t) {
          const int st = c % S;
          if (c >= S) {  // the stage's previous tile must have been released by its group
            const int cp = c - S;
            if (!(ok = mbar_wait(&empty[(cp & 1) * S + st], group_phase<S>(cp) & 1, ctl, kSiteKvEmpty))) break;
          }
          uint64_t *bar = &full[(c & 1) * S + st];
          mbar_arrive_expect_tx(bar, L::kStageBytes);
          uint8_t *dst = smem + st * L::kStageBytes;
#pragma unroll
          for (int s = 0; s < L::kSlabs; ++s) {
            tma_load_4d(dst + s * L::kSlabBytes, &tm_k, bar, s * 64, t * kDecTileKeys, x.h, x.b);
            tma_load_4d(dst + L::kTileBytes + s * L::kSlabBytes, &tm_v, bar, s * 64, t * kDecTileKeys, x.h, x.b);
          }
          ++c;
        }
      }
      // Every copy issued lands before this thread leaves, whatever the
      // other roles do (bounded waits; in a normal run they are done).
      for (int j = (c > S ? c - S : 0); j < c; ++j) mbar_drain(&full[(j & 1) * S + j % S], group_phase<S>(j) & 1);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = warp >> 2;         // group: tiles with counter parity g
  const int kq = (warp & 3) * 32;  // first key (row of the tile) of this warp
  const int r = kq + lane;         // this lane's key row for the scores
  const int tid = threadIdx.x;

  // Byte offset of this lane's O columns inside a swizzled V row.
  const int vbyte = lane * CPL * 2;
  const int vslab = vbyte >> 7, vchunk = (vbyte & 127) >> 4, vin = vbyte & 15;

  int c = 0;
  for (int it = blockIdx.x; it < p.items; it += gridDim.x) {
    const DecodeItem x = decode_item(p, it);

    // the item's query rows, fp32, scaled by scale*log2(e); rows >= Nq are 0
    for (int e = tid; e < NQ * D; e += kDecConsumers) {
      const int i = e / D, col = e - i * D;
      float v = 0.0f;
      if (i < p.Nq) v = __bfloat162float(p.q[row_offset(p.sq, x.bh, p.H, i) + col]) * p.scale_log2;
      qbuf[e] = v;
    }
    named_barrier(1, kDecConsumers);

    float m[NQ], l[NQ], o[NQ][CPL];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      m[i] = kNegInf;
      l[i] = 0.0f;
#pragma unroll
      for (int cc = 0; cc < CPL; ++cc) o[i][cc] = 0.0f;
    }
    // query i sees keys j < len, and with causal also j <= len - Nq + i
    const int vis_base = p.causal ? x.len - p.Nq : 0x3fffffff;

    for (int t = x.t0; t < x.t1; ++t) {
      const int cc_t = c + (t - x.t0);
      if ((cc_t & 1) != g) continue;
      const int st = cc_t % S;
      if (!*abort_flag) mbar_wait(&full[g * S + st], group_phase<S>(cc_t) & 1, ctl, kSiteKvFull);
      const uint8_t *sk = smem + st * L::kStageBytes;
      const uint8_t *sv = sk + L::kTileBytes;

      // ---- scores of this lane's key for every query row
      float2 acc[NQ];
#pragma unroll
      for (int i = 0; i < NQ; ++i) acc[i] = make_float2(0.0f, 0.0f);
      const uint8_t *krow = sk + r * 128;
      const int rsw = r & 7;
#pragma unroll
      for (int jj = 0; jj < D / 8; ++jj) {
        const uint4 kw =
            *reinterpret_cast<const uint4 *>(krow + (jj >> 3) * L::kSlabBytes + (((jj & 7) ^ rsw) << 4));
        const float2 k01 = bf16x2_to_float2(kw.x), k23 = bf16x2_to_float2(kw.y);
        const float2 k45 = bf16x2_to_float2(kw.z), k67 = bf16x2_to_float2(kw.w);
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
          const float4 qa = *reinterpret_cast<const float4 *>(qbuf + i * D + jj * 8);
          const float4 qb = *reinterpret_cast<const float4 *>(qbuf + i * D + jj * 8 + 4);
          acc[i] = ffma2(make_float2(qa.x, qa.y), k01, acc[i]);
          acc[i] = ffma2(make_float2(qa.z, qa.w), k23, acc[i]);
          acc[i] = ffma2(make_float2(qb.x, qb.y), k45, acc[i]);
          acc[i] = ffma2(make_float2(qb.z, qb.w), k67, acc[i]);
        }
      }
      const int j = t * kDecTileKeys + r;  // key position
      float pr[NQ];
#pragma unroll
      for (int i = 0; i < NQ; ++i) {
        const bool vis = i < p.Nq && j < x.len && j <= vis_base + i;
        const float s = vis ? acc[i].x + acc[i].y : kNegInf;
        const float mt = warp_max(s);
        const float mn = fmaxf(m[i], mt);
        if (mn == kNegInf) {  // nothing visible yet for this row
          pr[i] = 0.0f;
          continue;
        }
        if (mn > m[i]) {
          const float alpha = rescale(m[i], mn);
          l[i] *= alpha;
#pragma unroll
          for (int cc = 0; cc < CPL; ++cc) o[i][cc] *= alpha;
          m[i] = mn;
        }
        pr[i] = ex2(s - mn);  // 0 for masked keys
        l[i] += pr[i];
      }

      // ---- O += p V over the warp's 32 keys
#pragma unroll 4
      for (int k = 0; k < 32; ++k) {
        const int kr = kq + k;
        const uint8_t *vrow = sv + vslab * L::kSlabBytes + kr * 128 + ((vchunk ^ (kr & 7)) << 4) + vin;
        float vf[CPL];
        if constexpr (CPL == 4) {
          const uint2 vw = *reinterpret_cast<const uint2 *>(vrow);
          const float2 a = bf16x2_to_float2(vw.x), b2 = bf16x2_to_float2(vw.y);
          vf[0] = a.x, vf[1] = a.y, vf[2] = b2.x, vf[3] = b2.y;
        } else {
          const float2 a = bf16x2_to_float2(*reinterpret_cast<const uint32_t *>(vrow));
          vf[0] = a.x, vf[1] = a.y;
        }
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
          const float pk = __shfl_sync(0xffffffffu, pr[i], k);
#pragma unroll
          for (int cc = 0; cc < CPL; cc += 2) {
            const float2 r2 = ffma2(make_float2(pk, pk), make_float2(vf[cc], vf[cc + 1]),
                                    make_float2(o[i][cc], o[i][cc + 1]));
            o[i][cc] = r2.x;
            o[i][cc + 1] = r2.y;
          }
        }
      }
      warp_arrive(&empty[g * S + st]);
    }
    if (x.t1 > x.t0) c += x.t1 - x.t0;

    // ---- merge the 8 warps' states: 4..7 into 0..3, then 0..3 together
#pragma unroll
    for (int i = 0; i < NQ; ++i) l[i] = warp_sum(l[i]);
    if (warp >= 4) {
#pragma unroll
      for (int i = 0; i < NQ; ++i) {
#pragma unroll
        for (int cc = 0; cc < CPL; ++cc) obuf[((warp - 4) * NQ + i) * D + lane * CPL + cc] = o[i][cc];
        if (lane == 0) {
          stat_m[(warp - 4) * NQ + i] = m[i];
          stat_l[(warp - 4) * NQ + i] = l[i];
        }
      }
    }
    named_barrier(1, kDecConsumers);
    if (warp < 4) {
#pragma unroll
      for (int i = 0; i < NQ; ++i) {
        const float mb = stat_m[warp * NQ + i], lb = stat_l[warp * NQ + i];
        const float M = fmaxf(m[i], mb);
        if (M == kNegInf) continue;
        const float fa = rescale(m[i], M), fb = rescale(mb, M);
        l[i] = l[i] * fa + lb * fb;
#pragma unroll
        for (int cc = 0; cc < CPL; ++cc) o[i][cc] = o[i][cc] * fa + obuf[(warp * NQ + i) * D + lane * CPL + cc] * fb;
        m[i] = M;
      }
    }
    named_barrier(1, kDecConsumers);
    if (warp < 4) {
#pragma unroll
      for (int i = 0; i < NQ; ++i) {
#pragma unroll
        for (int cc = 0; cc < CPL; ++cc) obuf[(warp * NQ + i) * D + lane * CPL + cc] = o[i][cc];
        if (lane == 0) {
          stat_m[warp * NQ + i] = m[i];
          stat_l[warp * NQ + i] = l[i];
        }
      }
    }
    named_barrier(1, kDecConsumers);
    for (int e = tid; e < p.Nq * D; e += kDecConsumers) {
      const int i = e / D, col = e - i * D;
      float M = kNegInf;
#pragma unroll
      for (int w = 0; w < 4; ++w) M = fmaxf(M, stat_m[w * NQ + i]);
      float lsum = 0.0f, acc = 0.0f;
      if (M != kNegInf) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float f = rescale(stat_m[w * NQ + i], M);
          lsum += stat_l[w * NQ + i] * f;
          acc += obuf[(w * NQ + i) * D + col] * f;
        }
      }
      const bool any = lsum > 0.0f;
      const float out = any ? acc / lsum : 0.0f;
      const float lse2 = any ? M + log2f(lsum) : kNegInf;
      if (p.splits == 1) {
        p.o[row_offset(p.so, x.bh, p.H, i) + col] = __float2bfloat16_rn(out);
        if (col == 0) p.lse[static_cast<long long>(x.bh) * p.Nq + i] = any ? lse2 * kLn2 : kNegInf;
      } else {
        const long long part = (static_cast<long long>(x.bh) * p.splits + x.split) * p.Nq + i;
        p.part_o[part * D + col] = out;
        if (col == 0) p.part_lse[part] = lse2;
      }
    }
  }
}

// Merge the chunks' partial results of each (head, query row):
// O = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M), lse = M + log2 of the
// denominator (log2 units in the partials, natural log in the output).
template <int D>
__global__ void __launch_bounds__(D) fa_decode_combine_kernel(const DecodeParams p) {
  const int bh = blockIdx.x, col = threadIdx.x;
  for (int i = 0; i < p.Nq; ++i) {
    const long long base = static_cast<long long>(bh) * p.splits * p.Nq + i;
    float M = kNegInf;
    for (int s = 0; s < p.splits; ++s) M = fmaxf(M, p.part_lse[base + static_cast<long long>(s) * p.Nq]);
    float den = 0.0f, acc = 0.0f;
    if (M != kNegInf) {
      for (int s = 0; s < p.splits; ++s) {
        const long long part = base + static_cast<long long>(s) * p.Nq;
        const float f = rescale(p.part_lse[part], M);
        den += f;
        acc += f * p.part_o[part * D + col];
      }
    }
    const bool any = den > 0.0f;
    p.o[row_offset(p.so, bh, p.H, i) + col] = __float2bfloat16_rn(any ? acc / den : 0.0f);
    if (col == 0) p.lse[static_cast<long long>(bh) * p.Nq + i] = any ? (M + log2f(den)) * kLn2 : kNegInf;
  }
}

// ------------------------------------------------------------------
// Tensor-core decode for 2..8 query rows at d = 128.  From two rows on
// the CUDA-core products above, not HBM, set the pace; here both products
// run as tcgen05 MMAs with the 128 keys of a tile as M:
//   S^T = K Q^T      (M = 128 keys, N = 16 query rows (padded), K = d)
//   O^T += V^T P^T   (M = 128 = d, N = 16, K = 128 keys)
// so the key is the TMEM lane for the scores and d is the lane for O.  Per
// CTA: two groups of 4 row warps take alternate tiles (thread = key for the
// softmax, = d for the output), each with its own running maxima, sums and
// O^T accumulator, merged at the end of the item; warp 8 streams each
// item's query rows (into one of two buffers, ahead of time) and K and V
// by TMA; warp 9 issues the MMAs (one thread) and owns TMEM.  Each group's next
// scores are computed while it works on the current ones (two S and two P
// buffers per group), and the two groups' softmax chains overlap.

constexpr int kTcThreads = 320;    // 8 row warps, producer, MMA issuer
constexpr int kTcN = 16;
constexpr uint32_t kTcTmemCols = 128;  // per group g: S^T x 2 at 32 g (16 each), O^T at 64 + 16 g
constexpr float kTcRescale = 8.0f;     // a row's maximum moves only when exceeded by more than this (log2 units)

struct TcLayout {
  static constexpr int kStages = 3;
  static constexpr int kSlabBytes = 128 * 128;         // 128 rows x 64 bf16
  static constexpr int kTileBytes = 2 * kSlabBytes;    // K (or V) of one tile, d = 128
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kOffQ = kStages * kStageBytes;  // Q[2]: [16 rows x 128] bf16, K-major, 128-byte swizzle
  static constexpr int kQBytes = 2 * kTcN * 128;
  static constexpr int kOffP = kOffQ + 2 * kQBytes;    // P[group][2]: [16 rows x 128 keys] bf16, same layout
  static constexpr int kOffRed = kOffP + 4 * kQBytes;  // row maxima [group][2][4 warps][16], row sums [group][4][16]
  static constexpr int kOffMerge = kOffRed + (2 * 2 * 4 * kTcN + 2 * 4 * kTcN) * 4;  // group 1: m[16], l[16], O^T[128][16]
  static constexpr int kOffBar = kOffMerge + (2 * kTcN + 128 * kTcN) * 4;
  // full[S], empty[S], per group: s_full[2], s_free[2], p_ready[2], pv_done[2], o_free; q_full[2], q_empty[2], drain
  static constexpr int kNumBars = 2 * kStages + 2 * 9 + 5;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16;
  static constexpr int kSmemRequest = kSmemBytes + 1024;
  static_assert(kSmemRequest <= 227 * 1024, "tensor-core decode layout exceeds shared memory");
  static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0 && kQBytes % 1024 == 0, "swizzled operands need 1 KB alignment");
};

// Byte offset of element (r, c) in a K-major, 128-byte-swizzled bf16 tile
// of `rows` rows and 128 columns (two 64-column slabs).
__device__ __forceinline__ int sw128_off(int r, int c, int rows) {
  const int within = (c & 63) * 2;
  return (c >> 6) * rows * 128 + r * 128 + ((((within >> 4) ^ (r & 7))) << 4) + (within & 15);
}

// Tiles cc = c0 .. c0+n-1 of an item alternate between the groups: tile cc
// belongs to group cc & 1 and is that group's (cc >> 1)-th tile overall; it
// uses the group's buffer (cc >> 1) & 1, whose k-th use is phase k >> 1.
struct TcTile {
  int g, b;
  uint32_t ph;
};
__device__ __forceinline__ TcTile tc_tile(int cc) {
  const int k = cc >> 1;
  return TcTile{cc & 1, k & 1, static_cast<uint32_t>((k >> 1) & 1)};
}

template <int NQ>
__global__ void __launch_bounds__(kTcThreads, 1)
    fa_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_q, const DecodeParams p) {
  using L = TcLayout;
  constexpr int S = L::kStages;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
  uint64_t *empty = full + S;
  uint64_t *gb = empty + S;  // per group: [0,2) s_full, [2,4) s_free, [4,6) p_ready, [6,8) pv_done, 8 o_free
  uint64_t *q_full = gb + 18;  // [2]
  uint64_t *q_empty = q_full + 2;  // [2]
  uint64_t *drain = q_empty + 2;
  auto s_full = [&](int g, int b) { return gb + 9 * g + b; };
  auto s_free = [&](int g, int b) { return gb + 9 * g + 2 + b; };
  auto p_ready = [&](int g, int b) { return gb + 9 * g + 4 + b; };
  auto pv_done = [&](int g, int b) { return gb + 9 * g + 6 + b; };
  auto o_free = [&](int g) { return gb + 9 * g + 8; };
  uint8_t *sQ = smem + L::kOffQ;
  uint8_t *sP = smem + L::kOffP;
  float *red_max = reinterpret_cast<float *>(smem + L::kOffRed);  // [2][2][4][16]
  float *red_sum = red_max + 2 * 2 * 4 * kTcN;                      // [2][4][16]
  float *mrg = reinterpret_cast<float *>(smem + L::kOffMerge);      // m[16], l[16], O^T[128][16]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 4);
  const WaitCtl ctl{abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int g = 0; g < 2; ++g) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(s_full(g, b), 1);
        mbar_init(s_free(g, b), 4);
        mbar_init(p_ready(g, b), 4);
        mbar_init(pv_done(g, b), 1);
      }
      mbar_init(o_free(g), 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&q_full[b], 1);
      mbar_init(&q_empty[b], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // the P buffers start at zero: rows past Nq are never written and must
  // not bring NaNs into the (ignored) columns of O^T
  for (int e = threadIdx.x; e < 4 * L::kQBytes / 16; e += kTcThreads)
    reinterpret_cast<uint4 *>(sP)[e] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (warp == 9) {
    tmem_alloc(tmem_slot, kTcTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_q);
      int c = 0, ne = 0;
      bool ok = true;
      for (int it = blockIdx.x; ok && it < p.items; it += gridDim.x) {
        const DecodeItem x = decode_item(p, it);
        if (x.t1 <= x.t0) continue;
        // the item's query rows into Q buffer ne & 1 (rows past Nq read as zeros)
        const int qb = ne & 1;
        if (!(ok = mbar_wait(&q_empty[qb], ((ne >> 1) & 1) ^ 1, ctl, kSiteDoEmpty))) break;
        mbar_arrive_expect_tx(&q_full[qb], L::kQBytes);
#pragma unroll
        for (int s = 0; s < 2; ++s)
          tma_load_4d(smem + L::kOffQ + qb * L::kQBytes + s * kTcN * 128, &tm_q, &q_full[qb], s * 64, 0, x.h, x.b);
        ++ne;
        for (int t = x.t0; t < x.t1; ++t) {
          const int st = c % S;
          if (!(ok = mbar_wait(&empty[st], ((c / S) & 1) ^ 1, ctl, kSiteKvEmpty))) break;
          mbar_arrive_expect_tx(&full[st], L::kStageBytes);
          uint8_t *dst = smem + st * L::kStageBytes;
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            tma_load_4d(dst + s * L::kSlabBytes, &tm_k, &full[st], s * 64, t * kDecTileKeys, x.h, x.b);
            tma_load_4d(dst + L::kTileBytes + s * L::kSlabBytes, &tm_v, &full[st], s * 64, t * kDecTileKeys, x.h,
                        x.b);
          }
          ++c;
        }
      }
      // Every copy issued lands before this thread leaves, whatever the
      // other roles do (bounded waits; in a normal run they are done).
      for (int j = (c > S ? c - S : 0); j < c; ++j) mbar_drain(&full[j % S], (j / S) & 1);
      for (int j = (ne > 2 ? ne - 2 : 0); j < ne; ++j) mbar_drain(&q_full[j & 1], (j >> 1) & 1);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, kTcN, false, false);
      constexpr uint32_t kIdO = idesc_bf16(128, kTcN, true, false);
      const uint64_t dQ0 = sdesc_sw128(smem_addr(sQ), 16, 1024);
      const uint64_t dQ1 = sdesc_sw128(smem_addr(sQ + L::kQBytes), 16, 1024);
      const uint32_t aP = smem_addr(sP);
      const uint32_t aStage = smem_addr(smem);
      int c = 0, ne = 0;
      int seen0 = 0, seen1 = 0;  // items in which each group has had a tile
      bool ok = true;
      // O^T[g] += V^T P^T of global tile x; `first`: the group's first tile of the item
      auto issue_pv = [&](int x, bool first) -> bool {
        const TcTile tt = tc_tile(x);
        if (!mbar_wait(p_ready(tt.g, tt.b), tt.ph, ctl, kSitePReady)) return false;
        tc_fence_after();
        const uint64_t dv = sdesc_sw128(aStage + (x % S) * L::kStageBytes + L::kTileBytes, L::kSlabBytes, 1024);
        const uint64_t dp = sdesc_sw128(aP + (2 * tt.g + tt.b) * L::kQBytes, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + 64 + 16 * tt.g, desc_add(dv, mnmajor_step(kk)), desc_add(dp, kmajor_step(kk, kTcN)), kIdO,
                 (!first || kk > 0) ? 1u : 0u);
        tc_commit(pv_done(tt.g, tt.b));
        tc_commit(&empty[x % S]);
        return true;
      };
      for (int it = blockIdx.x; ok && it < p.items; it += gridDim.x) {
        const DecodeItem x = decode_item(p, it);
        const int n = x.t1 - x.t0;
        if (n <= 0) continue;
        const int qb = ne & 1;
        if (!(ok = mbar_wait(&q_full[qb], (ne >> 1) & 1, ctl, kSiteQFull))) break;
        const uint64_t dQ = qb ? dQ1 : dQ0;
        for (int u = 0; u <= n; ++u) {
          if (u < n) {
            const int cc = c + u;
            const TcTile tt = tc_tile(cc);
            if (!(ok = mbar_wait(&full[cc % S], (cc / S) & 1, ctl, kSiteKvFull))) break;
            if (!(ok = mbar_wait(s_free(tt.g, tt.b), tt.ph ^ 1, ctl, kSiteSFull))) break;
            tc_fence_after();
            const uint64_t dk = sdesc_sw128(aStage + (cc % S) * L::kStageBytes, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tmem + 32 * tt.g + 16 * tt.b, desc_add(dk, kmajor_step(kk, 128)),
                     desc_add(dQ, kmajor_step(kk, kTcN)), kIdS, kk > 0 ? 1u : 0u);
            tc_commit(s_full(tt.g, tt.b));
            if (u == n - 1) tc_commit(&q_empty[qb]);  // the item's last S has read its query rows
            const int seen = tt.g ? seen1 : seen0;
            if (u < 2 && seen > 0) {  // the group's O^T of its previous item must have been read
              if (!(ok = mbar_wait(o_free(tt.g), (seen - 1) & 1, ctl, kSiteMmaDone))) break;
            }
          }
          if (u > 0 && !(ok = issue_pv(c + u - 1, u - 1 < 2))) break;
        }
        if (!ok) break;
        if (n > ((c & 1) ? 1 : 0)) ++seen0;  // group g's first tile of the item is u = (c & 1) ^ g
        if (n > ((c & 1) ? 0 : 1)) ++seen1;
        c += n;
        ++ne;
      }
      // every MMA issued has completed before TMEM is released
      tc_commit(drain);
      mbar_drain(drain, 0);
    }
  } else {
    // ------------------------------------------------------------ rows
    const int g = warp >> 2;            // group
    const int tid = threadIdx.x & 127;  // key of the tile (scores), d (output)
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float csc = p.scale_log2;
    int c = 0;
    for (int it = blockIdx.x; it < p.items; it += gridDim.x) {
      const DecodeItem x = decode_item(p, it);
      const int n = x.t1 - x.t0;
      float m[NQ], lp[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        m[q] = kNegInf;
        lp[q] = 0.0f;
      }
      const int vis_base = p.causal ? x.len - p.Nq : 0x3fffffff;
      const int first_u = ((c & 1) == g) ? 0 : 1;  // this group's first tile of the item
      int last_cc = -1;
      for (int u = first_u; u < n; u += 2) {
        const int cc = c + u;
        const TcTile tt = tc_tile(cc);
        last_cc = cc;
        if (!*abort_flag) mbar_wait(s_full(g, tt.b), tt.ph, ctl, kSiteSFull);
        tc_fence_after();
        uint32_t sr[16];
        tmem_ld16(tmem + 32 * g + 16 * tt.b + lane_base, sr);
        tmem_ld_wait16(sr);
        tc_fence_before();
        warp_arrive(s_free(g, tt.b));
        const int j = (x.t0 + u) * kDecTileKeys + tid;  // this thread's key
        float t[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          const bool vis = q < p.Nq && j < x.len && j <= vis_base + q;
          t[q] = vis ? __uint_as_float(sr[q]) * csc : kNegInf;
        }
        // tile maximum of each query row over the 128 keys
        float *rm = red_max + (g * 2 + tt.b) * 4 * kTcN;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          const float w = warp_max_f32(t[q]);
          if (lane == 0) rm[(warp & 3) * kTcN + q] = w;
        }
        named_barrier(1 + g, 128);
        bool grow_any = false;
        float alpha[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          const float tm = fmaxf(fmaxf(rm[q], rm[kTcN + q]), fmaxf(rm[2 * kTcN + q], rm[3 * kTcN + q]));
          alpha[q] = 1.0f;
          if (tm > m[q] + kTcRescale || (m[q] == kNegInf && tm != kNegInf)) {
            alpha[q] = rescale(m[q], tm);
            m[q] = tm;
            grow_any = true;
          }
        }
        float pw[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          pw[q] = m[q] == kNegInf ? 0.0f : ex2(t[q] - m[q]);  // 0 for hidden keys
          lp[q] = lp[q] * alpha[q] + pw[q];
        }
        // this P buffer is free once the group's P V product two tiles back is done
        if (!*abort_flag) mbar_wait(pv_done(g, tt.b), tt.ph ^ 1, ctl, kSitePvDone);
        uint8_t *pb = sP + (2 * g + tt.b) * L::kQBytes;
#pragma unroll
        for (int q = 0; q < NQ; ++q)
          *reinterpret_cast<__nv_bfloat16 *>(pb + sw128_off(q, tid, kTcN)) = __float2bfloat16_rn(pw[q]);
        fence_proxy_async_smem();
        if (u > first_u && grow_any) {
          // O^T (lane = d) rescaled once the group's previous P V product is in
          const TcTile tp = tc_tile(cc - 2);
          if (!*abort_flag) mbar_wait(pv_done(g, tp.b), tp.ph, ctl, kSitePvDone);
          tc_fence_after();
          uint32_t o[16];
          tmem_ld16(tmem + 64 + 16 * g + lane_base, o);
          tmem_ld_wait16(o);
#pragma unroll
          for (int q = 0; q < NQ; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha[q]);
          tmem_st16(tmem + 64 + 16 * g + lane_base, o);
          tmem_st_wait();
        }
        tc_fence_before();
        warp_arrive(p_ready(g, tt.b));
      }
      // ---- the item's result: each group's O^T, then the two merged
      float o[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) o[q] = 0.0f;
      if (last_cc >= 0) {
        const TcTile tl = tc_tile(last_cc);
        if (!*abort_flag) mbar_wait(pv_done(g, tl.b), tl.ph, ctl, kSitePvDone);
        tc_fence_after();
        uint32_t orr[16];
        tmem_ld16(tmem + 64 + 16 * g + lane_base, orr);
        tmem_ld_wait16(orr);
#pragma unroll
        for (int q = 0; q < NQ; ++q) o[q] = __uint_as_float(orr[q]);
        tc_fence_before();
        warp_arrive(o_free(g));
      }
      float *rs = red_sum + g * 4 * kTcN;
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        const float w = warp_sum(lp[q]);
        if (lane == 0) rs[(warp & 3) * kTcN + q] = w;
      }
      named_barrier(1 + g, 128);
      float l[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) l[q] = rs[q] + rs[kTcN + q] + rs[2 * kTcN + q] + rs[3 * kTcN + q];
      if (g == 1) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) mrg[2 * kTcN + tid * kTcN + q] = o[q];
        if (tid == 0) {
#pragma unroll
          for (int q = 0; q < NQ; ++q) {
            mrg[q] = m[q];
            mrg[kTcN + q] = l[q];
          }
        }
      }
      named_barrier(3, 256);
      if (g == 0) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          if (q >= p.Nq) break;
          const float m1 = mrg[q], l1 = mrg[kTcN + q], o1 = mrg[2 * kTcN + tid * kTcN + q];
          const float M = fmaxf(m[q], m1);
          float lt = 0.0f, ot = 0.0f;
          if (M != kNegInf) {
            const float f0 = rescale(m[q], M), f1 = rescale(m1, M);
            lt = l[q] * f0 + l1 * f1;
            ot = (f0 > 0.0f ? o[q] * f0 : 0.0f) + (f1 > 0.0f ? o1 * f1 : 0.0f);
          }
          const bool any = lt > 0.0f;
          const float out = any ? ot / lt : 0.0f;
          const float lse2 = any ? M + log2f(lt) : kNegInf;
          if (p.splits == 1) {
            p.o[row_offset(p.so, x.bh, p.H, q) + tid] = __float2bfloat16_rn(out);
            if (tid == 0) p.lse[static_cast<long long>(x.bh) * p.Nq + q] = any ? lse2 * kLn2 : kNegInf;
          } else {
            const long long part = (static_cast<long long>(x.bh) * p.splits + x.split) * p.Nq + q;
            p.part_o[part * 128 + tid] = out;
            if (tid == 0) p.part_lse[part] = lse2;
          }
        }
      }
      named_barrier(3, 256);  // the merge area and the sums are rewritten by the next item
      if (n > 0) c += n;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcTmemCols);
  }
}

template <int D, int NQ>
cudaError_t launch_decode_t(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, int grid,
                            cudaStream_t stream) {
  using L = DecodeLayout<D, NQ>;
  auto kern = fa_decode_kernel<D, NQ>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemRequest);
  if (e != cudaSuccess) return e;
  kern<<<grid, kDecThreads, L::kSmemRequest, stream>>>(tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.splits == 1) return e;
  fa_decode_combine_kernel<D><<<p.BH, D, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int NQ>
cudaError_t launch_decode_tc(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tq,
                             const DecodeParams &p, int grid, cudaStream_t stream) {
  auto kern = fa_decode_tc_kernel<NQ>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TcLayout::kSmemRequest);
  if (e != cudaSuccess) return e;
  kern<<<grid, kTcThreads, TcLayout::kSmemRequest, stream>>>(tk, tv, tq, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.splits == 1) return e;
  fa_decode_combine_kernel<128><<<p.BH, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_d(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tq,
                            const DecodeParams &p, int grid, cudaStream_t stream) {
  if (D == 128 && p.Nq >= 2) {  // the tensor-core products
    return p.Nq <= 4 ? launch_decode_tc<4>(tk, tv, tq, p, grid, stream)
                     : launch_decode_tc<8>(tk, tv, tq, p, grid, stream);
  }
  if (p.Nq <= 1) return launch_decode_t<D, 1>(tk, tv, p, grid, stream);
  if (p.Nq <= 2) return launch_decode_t<D, 2>(tk, tv, p, grid, stream);
  if (p.Nq <= 4) return launch_decode_t<D, 4>(tk, tv, p, grid, stream);
  return launch_decode_t<D, 8>(tk, tv, p, grid, stream);
}

}  // namespace

cudaError_t launch_decode(int d, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tq,
                          const DecodeParams &p, int grid, cudaStream_t stream) {
  return d == 64 ? launch_decode_d<64>(tk, tv, tq, p, grid, stream) : launch_decode_d<128>(tk, tv, tq, p, grid, stream);
}

}  // namespace fa
