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

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

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
      if (!ok) {
        // let the copies still in flight land before the CTA exits
        for (int j = (c > S ? c - S : 0); j < c; ++j) mbar_drain(&full[(j & 1) * S + j % S], group_phase<S>(j) & 1);
      }
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

template <int D>
cudaError_t launch_decode_d(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, int grid,
                            cudaStream_t stream) {
  if (p.Nq <= 1) return launch_decode_t<D, 1>(tk, tv, p, grid, stream);
  if (p.Nq <= 2) return launch_decode_t<D, 2>(tk, tv, p, grid, stream);
  if (p.Nq <= 4) return launch_decode_t<D, 4>(tk, tv, p, grid, stream);
  return launch_decode_t<D, 8>(tk, tv, p, grid, stream);
}

}  // namespace

cudaError_t launch_decode(int d, const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, int grid,
                          cudaStream_t stream) {
  return d == 64 ? launch_decode_d<64>(tk, tv, p, grid, stream) : launch_decode_d<128>(tk, tv, p, grid, stream);
}

}  // namespace fa
