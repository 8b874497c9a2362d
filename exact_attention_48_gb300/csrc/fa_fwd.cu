// fa_fwd.cu -- forward kernel of exact attention for sm_103a.
//
// One CTA owns 128 query rows of one (batch, head) and walks the key/value
// blocks of that head (lexicon page "FlashAttention" (urworte.de), section
// "Methodische Grundlagen": block-wise processing in on-chip memory, the
// score / normalisation / weighting steps fused in one pass, and a running
// row normalisation that corrects the partial output whenever a larger
// score appears).  The grid spreads the query blocks of every head over the
// SMs (page "FlashAttention-2 (DE)", "Technische Architektur", section 2).
//
// Roles inside the CTA (256 threads):
//   warp 0      TMA producer: Q once, then K_j and V_j into a ring of stages
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into TMEM, O += P_j V_j
//   warp 2      owns the TMEM allocation
//   warps 4..7  softmax: one query row per thread, running max m and sum l
//               in registers, P_j written back as bf16 over S_j in TMEM
//               (it is the A operand of the P V product), O rescaled in TMEM
//               when m grows, final O / l and the logsumexp.
//
// TMEM columns: S_0 [0,128), S_1 [128,256), O [256, 256+d).  Two S buffers
// let the score product of block j+1 run while rows of block j are being
// normalised.  Only scores and probabilities of the current block ever
// exist, and only on chip (page "FlashAttention-2 (DE)", "Hintergrund").
//
// Scores are kept in the log2 domain: t = s * scale * log2(e).  The running
// max is only moved when a row's new block max exceeds it by more than 8
// (a factor 256 in P), so most blocks skip the O rescale; the result is the
// same because l and O always share the max they were computed with.

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kBM = 128;  // query rows per CTA
constexpr int kBN = 128;  // keys per block
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct FwdLayout {
  static constexpr int kSlabs = D / 64;  // 128-byte column slabs of a bf16 row
  static constexpr int kStages = (D == 64) ? 4 : 3;
  static constexpr uint32_t kQBytes = kBM * D * 2;
  static constexpr uint32_t kKVBytes = kBN * D * 2;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + kQBytes;
  static constexpr uint32_t kOffV = kOffK + kStages * kKVBytes;
  static constexpr uint32_t kOffBar = kOffV + kStages * kKVBytes;
  // q_full, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2], p_ready[2], pv_done[2], drain
  static constexpr int kNumBars = 1 + 4 * kStages + 6 + 1;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kBytes = kOffMisc + 16;
  static constexpr uint32_t kSmemRequest = kBytes + 1024;  // slack for 1024-byte alignment
  static_assert(kSmemRequest <= 232448, "shared memory budget");
};

constexpr uint32_t kTmemCols = 512;

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(256, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = FwdLayout<D>;
  constexpr int S = L::kStages;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
  uint64_t *q_full = bars;
  uint64_t *k_full = bars + 1;
  uint64_t *k_empty = k_full + S;
  uint64_t *v_full = k_empty + S;
  uint64_t *v_empty = v_full + S;
  uint64_t *s_full = v_empty + S;
  uint64_t *p_ready = s_full + 2;
  uint64_t *pv_done = p_ready + 2;
  uint64_t *drain = pv_done + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 4);
  const WaitCtl ctl{abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Tile order.  Causal: the heaviest query blocks (most key blocks) first,
  // across all heads.  Otherwise head-major so that CTAs running together
  // share the K/V of one head in L2.
  int bh, qblk;
  if (CAUSAL) {
    qblk = p.num_qblk - 1 - static_cast<int>(blockIdx.x) / p.BH;
    bh = static_cast<int>(blockIdx.x) % p.BH;
  } else {
    bh = static_cast<int>(blockIdx.x) / p.num_qblk;
    qblk = static_cast<int>(blockIdx.x) % p.num_qblk;
  }
  const int N = p.N;
  const int n_kv = CAUSAL ? (qblk + 1) : (N + kBN - 1) / kBN;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_ready[b], 128);
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS0 = tmem, tO = tmem + 256;

  uint8_t *sQ = smem + L::kOffQ;
  uint8_t *sK = smem + L::kOffK;
  uint8_t *sV = smem + L::kOffV;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(q_full, L::kQBytes);
#pragma unroll
      for (int s = 0; s < L::kSlabs; ++s) tma_load_3d(sQ + s * kBM * 128, &tm_q, q_full, s * 64, qblk * kBM, bh);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % S;
        const uint32_t ph = (j / S) & 1;
        if (!mbar_wait(&k_empty[st], ph ^ 1, ctl, kSiteKEmpty)) break;
        mbar_arrive_expect_tx(&k_full[st], L::kKVBytes);
#pragma unroll
        for (int s = 0; s < L::kSlabs; ++s)
          tma_load_3d(sK + st * L::kKVBytes + s * kBN * 128, &tm_k, &k_full[st], s * 64, j * kBN, bh);
        k_issued = j + 1;
        if (!mbar_wait(&v_empty[st], ph ^ 1, ctl, kSiteVEmpty)) break;
        mbar_arrive_expect_tx(&v_full[st], L::kKVBytes);
#pragma unroll
        for (int s = 0; s < L::kSlabs; ++s)
          tma_load_3d(sV + st * L::kKVBytes + s * kBN * 128, &tm_v, &v_full[st], s * 64, j * kBN, bh);
        v_issued = j + 1;
      }
      if (*abort_flag) {
        // let the copies still in flight land before the CTA exits
        mbar_drain(q_full, 0);
        for (int j = (k_issued > S ? k_issued - S : 0); j < k_issued; ++j) mbar_drain(&k_full[j % S], (j / S) & 1);
        for (int j = (v_issued > S ? v_issued - S : 0); j < v_issued; ++j) mbar_drain(&v_full[j % S], (j / S) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16(kBM, kBN, false, false);
      constexpr uint32_t kIdescO = idesc_bf16(kBM, D, false, true);
      const uint32_t aQ = smem_addr(sQ), aK = smem_addr(sK), aV = smem_addr(sV);

      // O += P_t V_t; P_t sits (bf16, two per column) over S_t in TMEM.
      auto issue_pv = [&](int t) -> bool {
        const int b = t & 1, st = t % S;
        if (!mbar_wait(&p_ready[b], (t >> 1) & 1, ctl, kSitePReady)) return false;
        if (!mbar_wait(&v_full[st], (t / S) & 1, ctl, kSiteVFull)) return false;
        tc_fence_after();
        const uint32_t vbase = aV + st * L::kKVBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // V_t is [key][d]: MN-major for this product (d contiguous).  16
          // keys = two 8-row groups of 1024 bytes; d slabs 128*128 bytes apart.
          const uint64_t bdesc = sdesc_sw128(vbase + kk * 2048, kBN * 128, 1024);
          mma_ts(tO, tS0 + b * 128 + kk * 8, bdesc, kIdescO, (t > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&v_empty[st]);
        tc_commit(&pv_done[b]);
        return true;
      };

      bool ok = mbar_wait(q_full, 0, ctl, kSiteQFull);
      tc_fence_after();
      for (int j = 0; ok && j < n_kv; ++j) {
        const int st = j % S, b = j & 1;
        if (!mbar_wait(&k_full[st], (j / S) & 1, ctl, kSiteKFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kbase = aK + st * L::kKVBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
          const uint64_t adesc = sdesc_sw128(aQ + koff, 16, 1024);
          const uint64_t bdesc = sdesc_sw128(kbase + koff, 16, 1024);
          mma_ss(tS0 + b * 128, adesc, bdesc, kIdescS, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[b]);
        tc_commit(&k_empty[st]);
        if (j > 0) ok = issue_pv(j - 1);
      }
      if (ok) issue_pv(n_kv - 1);
      tc_commit(drain);
      mbar_drain(drain, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const float c = p.scale_log2;
    const bool neg = p.neg != 0;
    float m_run = -INFINITY, l_run = 0.0f;
    bool ok = true;

    for (int j = 0; j < n_kv; ++j) {
      const int b = j & 1;
      ok = mbar_wait(&s_full[b], (j >> 1) & 1, ctl, kSiteSFull);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tS = tS0 + b * 128 + lane_base;
      uint32_t s[4][32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tmem_ld32(tS + q4 * 32, s[q4]);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tmem_ld_wait(s[q4]);

      // Masking: causal diagonal block and the ragged last key block.
      const bool need_mask = (CAUSAL && j == qblk) || ((j + 1) * kBN > N);
      int lim = kBN - 1;  // last visible column of this row
      if (need_mask) {
        lim = min(lim, N - 1 - j * kBN);
        if (CAUSAL && j == qblk) lim = min(lim, row);
        const uint32_t hide = __float_as_uint(neg ? INFINITY : -INFINITY);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (q4 * 32 + i > lim) s[q4][i] = hide;
      }

      // Block max of t = s * c (a min of s when the scale is negative).
      float mx;
      if (!neg) {
        float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            m0 = fmaxf(m0, __uint_as_float(s[q4][i]));
            m1 = fmaxf(m1, __uint_as_float(s[q4][i + 1]));
          }
        mx = fmaxf(m0, m1);
      } else {
        float m0 = INFINITY, m1 = INFINITY;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            m0 = fminf(m0, __uint_as_float(s[q4][i]));
            m1 = fminf(m1, __uint_as_float(s[q4][i + 1]));
          }
        mx = fminf(m0, m1);
      }
      const float m_cand = mx * c;
      const bool grow = m_cand > m_run + kRescaleThreshold;
      float alpha = 1.0f;
      if (grow) {
        alpha = ex2(m_run - m_cand);
        m_run = m_cand;
      }
      l_run *= alpha;
      const float neg_m = -m_run;

      // P = exp2(t - m) as bf16 pairs over the first 64 columns of S_j.
      float sum0 = 0.0f, sum1 = 0.0f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2)
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const int q4 = 2 * h + q2;
            float p0 = ex2(fmaf(__uint_as_float(s[q4][i]), c, neg_m));
            float p1 = ex2(fmaf(__uint_as_float(s[q4][i + 1]), c, neg_m));
            if (need_mask) {
              p0 = (q4 * 32 + i <= lim) ? p0 : 0.0f;
              p1 = (q4 * 32 + i + 1 <= lim) ? p1 : 0.0f;
            }
            sum0 += p0;
            sum1 += p1;
            pk[q2 * 16 + i / 2] = pack_bf16x2(p0, p1);
          }
        tmem_st32(tS + h * 32, pk);
      }
      l_run += sum0 + sum1;
      tmem_st_wait();

      // O of the previous block must be complete before it is rescaled and
      // before the next product accumulates into it.
      if (j > 0) {
        ok = mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, ctl, kSitePvDone);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        if (__any_sync(0xffffffffu, grow)) {
          tc_fence_after();
#pragma unroll 1
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t o[32];
            tmem_ld32(tO + lane_base + ch * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + lane_base + ch * 32, o);
          }
          tmem_st_wait();
        }
      }
      tc_fence_before();
      mbar_arrive(&p_ready[b]);
    }

    // Epilogue: O / l in bf16 and the natural-log logsumexp.
    if (ok) {
      const int last = n_kv - 1;
      ok = mbar_wait(&pv_done[last & 1], (last >> 1) & 1, ctl, kSitePvDone);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.0f / l_run;
      const int grow_row = qblk * kBM + row;
      const bool store = grow_row < N;
      __nv_bfloat16 *orow = p.o + (static_cast<size_t>(bh) * N + grow_row) * D;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t o[32];
        tmem_ld32(tO + lane_base + ch * 32, o);
        tmem_ld_wait(o);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
        if (store) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + ch * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if (store) p.lse[static_cast<size_t>(bh) * N + grow_row] = (m_run + log2f(l_run)) * kLn2;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_fwd_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const FwdParams &p,
                         cudaStream_t stream) {
  using L = FwdLayout<D>;
  auto kern = fa_fwd_kernel<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemRequest);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(p.BH) * static_cast<unsigned>(p.num_qblk);
  kern<<<grid, 256, L::kSmemRequest, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int d, bool causal, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const FwdParams &p, cudaStream_t stream) {
  if (d == 64) return causal ? launch_fwd_t<64, true>(tq, tk, tv, p, stream) : launch_fwd_t<64, false>(tq, tk, tv, p, stream);
  return causal ? launch_fwd_t<128, true>(tq, tk, tv, p, stream) : launch_fwd_t<128, false>(tq, tk, tv, p, stream);
}

}  // namespace fa
