// fa_fwd_fp8.cu -- FP8 (e4m3) forward for sm_103a.
//
// The page "FlashAttention-2 (DE)", section "Vergleich mit nachfolgenden
// Versionen" / "FlashAttention-3", names low-precision FP8 arithmetic as one
// of FlashAttention-3's additions.  Here both products run on the tensor
// core in its 8-bit mode (tcgen05.mma kind::f8f6f4, twice the bf16 rate):
// S = Q K^T from e4m3 Q and K, and O += P V with P rounded to e4m3 and V in
// e4m3.  What the kernel computes (the oracle writes the same definition
// out): scores from the decoded inputs times the tensor scales, in fp32;
// the running row maximum kept as an INTEGER (log2 units), so that every
// correction factor is an exact power of two and each weight, a power of
// two times 2^t, is rounded to e4m3 on a grid that does not depend on the
// order the key blocks are visited in (in e4m3's normal range); O
// normalised by the sum of the rounded weights (the weights actually
// applied); the logsumexp from the fp32 weights before rounding.
//
// Structure as in the bf16 forward: one CTA owns 256 query rows (two tiles
// of 128) of one head; warps 0..3 / 4..7 run the softmax of tile 0 / 1 (one
// row per thread), warp 8 loads Q once and K, V through a 4-stage TMA ring,
// warp 9 issues the products (one thread) and owns TMEM.  TMEM: S_0 and S_1
// (128 columns each; P is written over the first 32 columns of its S, four
// e4m3 per column, as the A operand of P V) and O_0, O_1 (128 each).
// Head dimension 128: one 128-byte swizzle row holds a whole row of Q, K or
// V.

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kD = 128;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr uint32_t kTmemCols = 512;
// The running (integer) maximum may lag a row's true maximum by up to
// kStale (log2 units) before O is rescaled; weights are 2^(t - m + 8 - kStale)
// <= 2^8, inside e4m3's range, and rescales become rare.
constexpr int kStale = 2;
constexpr int kThreads = 384;
constexpr int kWarpProducer = 8, kWarpMma = 9;
// Register split: 168 per thread at launch; the control warpgroup keeps 152
// (at 104 its issue loops spilled) and the softmax warpgroups take 176:
// 128*152 + 256*176 <= 384*168, and per SM sub-partition 32*(152 + 2*176)
// <= 16384.
constexpr uint32_t kRegsLaunch = 168, kRegsControl = 152, kRegsSoftmax = 176;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * kRegsLaunch, "register split");

struct F8Layout {
  static constexpr int kStages = 4;
  static constexpr uint32_t kQTile = kBM * kD;     // bytes: one e4m3 per element
  static constexpr uint32_t kKVBytes = kBN * kD;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + 2 * kQTile;
  static constexpr uint32_t kOffV = kOffK + kStages * kKVBytes;
  static constexpr uint32_t kOffBar = kOffV + kStages * kKVBytes;
  static constexpr int kNumBars = 1 + 4 * kStages + 6 + 1;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kBytes = kOffMisc + 16;
  static constexpr uint32_t kSmemRequest = kBytes + 1024;
  static_assert(kSmemRequest <= 232448, "shared memory budget");
};

// 2^k for an integer-valued k <= 0 (0 below the normal range, and for -inf).
__device__ __forceinline__ float exp2_int(float k) {
  return k < -126.0f ? 0.0f : __int_as_float((static_cast<int>(k) + 127) << 23);
}

struct F8SoftmaxArgs {
  uint64_t *s_full, *p_ready, *pv_done;
  uint32_t tS, tO;
  int n_kv, diag, grow0;
};

template <bool CAUSAL>
__device__ __forceinline__ void softmax_tile_f8(const F8SoftmaxArgs &a, const Fp8FwdParams &p, const WaitCtl &ctl,
                                                int bh, int warp, int lane) {
  const int wq = warp & 3;
  const int row = wq * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  const int N = p.N;
  const float c = p.scale_log2;  // scale * sq * sk * log2(e)
  const bool neg = p.neg != 0;
  const uint32_t tS = a.tS + lane_base, tO = a.tO + lane_base;
  float m_run = -INFINITY, l_run = 0.0f, lb_run = 0.0f;
  bool ok = true;

  // One key block; MASK: the causal or ragged-end mask, which only a
  // tile's last block needs.  Two copies of the body (MaskTag) keep the
  // masking instructions out of every other block (measured: 5 % faster
  // than one body with a run-time test, non-causal).
  auto block = [&](const int j, auto mask_tag) -> bool {
    const bool MASK = mask_tag;
    if (!__all_sync(0xffffffffu, mbar_wait(a.s_full, j & 1, ctl, kSiteSFull))) return false;
    tc_fence_after();
    uint32_t s[4][32];
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) tmem_ld32(tS + q4 * 32, s[q4]);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) tmem_ld_wait(s[q4]);

    int lim = kBN - 1;
    if (MASK) {
      lim = min(lim, N - 1 - j * kBN);
      if (CAUSAL && j == a.diag) lim = min(lim, row);
      const uint32_t hide = __float_as_uint(neg ? INFINITY : -INFINITY);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (q4 * 32 + i > lim) s[q4][i] = hide;
    }

    float mx;
    {
      float mq[4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float m0;
        if (!neg) {
          m0 = fmax3(__uint_as_float(s[q4][0]), __uint_as_float(s[q4][1]), __uint_as_float(s[q4][2]));
#pragma unroll
          for (int i = 3; i < 31; i += 2) m0 = fmax3(m0, __uint_as_float(s[q4][i]), __uint_as_float(s[q4][i + 1]));
          m0 = fmaxf(m0, __uint_as_float(s[q4][31]));
        } else {
          m0 = fmin3(__uint_as_float(s[q4][0]), __uint_as_float(s[q4][1]), __uint_as_float(s[q4][2]));
#pragma unroll
          for (int i = 3; i < 31; i += 2) m0 = fmin3(m0, __uint_as_float(s[q4][i]), __uint_as_float(s[q4][i + 1]));
          m0 = fminf(m0, __uint_as_float(s[q4][31]));
        }
        mq[q4] = m0;
      }
      mx = neg ? fminf(fminf(mq[0], mq[1]), fminf(mq[2], mq[3])) : fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
    }
    // Integer running maximum m, moved to ceil(block max) only when the
    // block max exceeds it by more than kStale: every weight
    // 2^(t - m + 8 - kStale) is at most 256, inside e4m3's range, and a
    // correction 2^(m_old - m_new) is exact.
    const float t_max = mx * c;
    const bool grow = t_max > m_run + static_cast<float>(kStale);
    float alpha = 1.0f;
    if (grow) {
      const float m_new = ceilf(t_max);
      alpha = exp2_int(m_run - m_new);
      m_run = m_new;
    }
    const float b0 = static_cast<float>(8 - kStale) - m_run;
    const float2 cc = make_float2(c, c), bias = make_float2(b0, b0);

    // P as e4m3, four per 32-bit column over the first 32 columns of S; the
    // fp32 sum of the unrounded P on the way (for the logsumexp).
    uint32_t pk[32];
    float2 sf = make_float2(0.f, 0.f);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      float2 sfq = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float2 x01 = ffma2(make_float2(__uint_as_float(s[q4][i]), __uint_as_float(s[q4][i + 1])), cc, bias);
        const float2 x23 =
            ffma2(make_float2(__uint_as_float(s[q4][i + 2]), __uint_as_float(s[q4][i + 3])), cc, bias);
        float p0 = ex2(x01.x), p1 = ex2(x01.y), p2 = ex2(x23.x), p3 = ex2(x23.y);
        if (MASK) {
          const int k0 = q4 * 32 + i;
          p0 = (k0 <= lim) ? p0 : 0.0f;
          p1 = (k0 + 1 <= lim) ? p1 : 0.0f;
          p2 = (k0 + 2 <= lim) ? p2 : 0.0f;
          p3 = (k0 + 3 <= lim) ? p3 : 0.0f;
        }
        pk[q4 * 8 + i / 4] = pack_e4m3x4(p0, p1, p2, p3);
        sfq = fadd2(sfq, fadd2(make_float2(p0, p1), make_float2(p2, p3)));
      }
      sf = fadd2(sf, sfq);
    }
    tmem_st32(tS, pk);
    tmem_st_wait();

    if (j > 0 && __any_sync(0xffffffffu, grow)) {
      if (!__all_sync(0xffffffffu, mbar_wait(a.pv_done, (j - 1) & 1, ctl, kSitePvDone))) return false;
      tc_fence_after();
#pragma unroll 1
      for (int ch = 0; ch < kD / 16; ++ch) {
        uint32_t o[16];
        tmem_ld16(tO + ch * 16, o);
        tmem_ld_wait16(o);
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st16(tO + ch * 16, o);
      }
      tmem_st_wait();
    }
    tc_fence_before();
    warp_arrive(a.p_ready);

    // Sum of the rounded weights (what the P V product applied): O is
    // divided by it.
    float2 sb = make_float2(0.f, 0.f);
#pragma unroll
    for (int w = 0; w < 32; ++w) {
      sb = add_e4m3x4_f32(sb, pk[w]);
    }
    l_run = l_run * alpha + (sf.x + sf.y);
    lb_run = lb_run * alpha + (sb.x + sb.y);
    return true;
  };
  for (int j = 0; j < a.n_kv; ++j) {
    const bool need_mask = (CAUSAL && j == a.diag) || ((j + 1) * kBN > N);
    if (!(need_mask ? block(j, MaskTag<true>{}) : block(j, MaskTag<false>{}))) {
      ok = false;
      break;
    }
  }


  if (ok) {
    ok = mbar_wait(a.pv_done, (a.n_kv - 1) & 1, ctl, kSitePvDone);
    ok = __all_sync(0xffffffffu, ok);
  }
  if (ok) {
    tc_fence_after();
    const float f = p.v_scale / lb_run;
    const int grow_row = a.grow0 + row;
    const bool store = grow_row < N;
    __nv_bfloat16 *orow = p.o + row_offset(p.so, bh, p.H, grow_row);
#pragma unroll 1
    for (int ch = 0; ch < kD / 32; ++ch) {
      uint32_t o[32];
      tmem_ld32(tO + ch * 32, o);
      tmem_ld_wait(o);
      uint32_t ob[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) ob[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * f, __uint_as_float(o[2 * i + 1]) * f);
      if (store) {
        uint4 *dst = reinterpret_cast<uint4 *>(orow + ch * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(ob[4 * i], ob[4 * i + 1], ob[4 * i + 2], ob[4 * i + 3]);
      }
    }
    if (store)
      p.lse[static_cast<long long>(bh) * N + grow_row] =
          (m_run - static_cast<float>(8 - kStale) + log2f(l_run)) * kLn2;
  }
}

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const Fp8FwdParams p) {
  using L = F8Layout;
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

  int bh, qb;
  if (CAUSAL) {
    qb = p.num_qblk - 1 - static_cast<int>(blockIdx.x) / p.BH;
    bh = static_cast<int>(blockIdx.x) % p.BH;
  } else {
    bh = static_cast<int>(blockIdx.x) / p.num_qblk;
    qb = static_cast<int>(blockIdx.x) % p.num_qblk;
  }
  const int bh_h = bh % p.H, bh_b = bh / p.H;
  const int nkv_all = (p.N + kBN - 1) / kBN;
  const int n0 = CAUSAL ? min(2 * qb + 1, nkv_all) : nkv_all;
  const int n1 = CAUSAL ? min(2 * qb + 2, nkv_all) : nkv_all;
  const int n_kv = n1;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_ready[t], 4);
      mbar_init(&pv_done[t], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  uint8_t *sQ = smem + L::kOffQ;
  uint8_t *sK = smem + L::kOffK;
  uint8_t *sV = smem + L::kOffV;

  if (warp >= kWarpProducer) {
    regs_decrease<kRegsControl>();
    if (warp == kWarpProducer && lane == 0) {
      // ---------------------------------------------------------- producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(q_full, 2 * L::kQTile);
#pragma unroll
      for (int t = 0; t < 2; ++t) tma_load_4d(sQ + t * L::kQTile, &tm_q, q_full, 0, qb * 2 * kBM + t * kBM, bh_h, bh_b);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % S;
        const uint32_t ph = (j / S) & 1;
        if (!mbar_wait(&k_empty[st], ph ^ 1, ctl, kSiteKEmpty)) break;
        mbar_arrive_expect_tx(&k_full[st], L::kKVBytes);
        tma_load_4d(sK + st * L::kKVBytes, &tm_k, &k_full[st], 0, j * kBN, bh_h, bh_b);
        k_issued = j + 1;
        if (!mbar_wait(&v_empty[st], ph ^ 1, ctl, kSiteVEmpty)) break;
        mbar_arrive_expect_tx(&v_full[st], L::kKVBytes);
        tma_load_4d(sV + st * L::kKVBytes, &tm_v, &v_full[st], 0, j * kBN, bh_h, bh_b);
        v_issued = j + 1;
      }
      // Every copy issued lands before this thread leaves, whatever the
      // other roles do (bounded waits; in a normal run they are done).
      mbar_drain(q_full, 0);
      for (int j = (k_issued > S ? k_issued - S : 0); j < k_issued; ++j) mbar_drain(&k_full[j % S], (j / S) & 1);
      for (int j = (v_issued > S ? v_issued - S : 0); j < v_issued; ++j) mbar_drain(&v_full[j % S], (j / S) & 1);
    } else if (warp == kWarpMma && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      // S_t = Q_t K_j^T: both K-major, 32 e4m3 (32 bytes) per K step inside
      // the 128-byte swizzle row.  O_t += P_t V_j: P from TMEM (8 columns
      // per 32 keys), V_j MN-major (d contiguous, one 128-byte atom wide),
      // 32 keys = four 1024-byte groups of 8 rows per K step.
      constexpr uint32_t kIdescS = idesc_e4m3(kBM, kBN, false, false);
      constexpr uint32_t kIdescO = idesc_e4m3(kBM, kD, false, true);
      const uint32_t aQ = smem_addr(sQ), aK = smem_addr(sK), aV = smem_addr(sV);
      const uint64_t dQ0 = sdesc_sw128(aQ, 16, 1024), dQ1 = sdesc_sw128(aQ + L::kQTile, 16, 1024);

      auto issue_s = [&](int t, int j) {
        const uint64_t bq = t ? dQ1 : dQ0, bk = sdesc_sw128(aK + (j % S) * L::kKVBytes, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kD / 32; ++kk)
          mma_ss_f8(tmem + t * 128, desc_add(bq, kk * 32), desc_add(bk, kk * 32), kIdescS, kk > 0 ? 1u : 0u);
        tc_commit(&s_full[t]);
      };
      auto issue_pv = [&](int t, int j) -> bool {
        if (!mbar_wait(&p_ready[t], j & 1, ctl, kSitePReady)) return false;
        tc_fence_after();
        const uint64_t bv = sdesc_sw128(aV + (j % S) * L::kKVBytes, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kBN / 32; ++kk)
          mma_ts_f8(tmem + 256 + t * kD, tmem + t * 128 + kk * 8, desc_add(bv, kk * 4096), kIdescO,
                    (j > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&pv_done[t]);
        return true;
      };

      bool ok = mbar_wait(q_full, 0, ctl, kSiteQFull) && mbar_wait(&k_full[0], 0, ctl, kSiteKFull);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        issue_s(1, 0);
        tc_commit(&k_empty[0]);
      }
      for (int j = 1; ok && j < n_kv; ++j) {
        const int pj = j - 1;
        if (!(ok = mbar_wait(&v_full[pj % S], (pj / S) & 1, ctl, kSiteVFull))) break;
        tc_fence_after();
        if (pj < n0 && !(ok = issue_pv(0, pj))) break;
        if (!(ok = mbar_wait(&k_full[j % S], (j / S) & 1, ctl, kSiteKFull))) break;
        tc_fence_after();
        if (j < n0) issue_s(0, j);
        if (!(ok = issue_pv(1, pj))) break;
        tc_commit(&v_empty[pj % S]);
        issue_s(1, j);
        tc_commit(&k_empty[j % S]);
      }
      if (ok) {
        const int pj = n_kv - 1;
        ok = mbar_wait(&v_full[pj % S], (pj / S) & 1, ctl, kSiteVFull);
        if (ok) {
          tc_fence_after();
          if (pj < n0) ok = issue_pv(0, pj);
          if (ok) ok = issue_pv(1, pj);
          tc_commit(&v_empty[pj % S]);
        }
      }
      tc_commit(drain);
      mbar_drain(drain, 0);
    }
  } else {
    regs_increase<kRegsSoftmax>();
    const int t = warp >> 2;
    F8SoftmaxArgs a;
    a.s_full = &s_full[t];
    a.p_ready = &p_ready[t];
    a.pv_done = &pv_done[t];
    a.tS = tmem + t * 128;
    a.tO = tmem + 256 + t * kD;
    a.n_kv = t ? n1 : n0;
    a.diag = CAUSAL ? 2 * qb + t : -1;
    a.grow0 = qb * 2 * kBM + t * kBM;
    softmax_tile_f8<CAUSAL>(a, p, ctl, bh, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool CAUSAL>
cudaError_t launch_fwd_fp8_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                             const Fp8FwdParams &p, cudaStream_t stream) {
  auto kern = fa_fwd_fp8_kernel<CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, F8Layout::kSmemRequest);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(p.BH) * static_cast<unsigned>(p.num_qblk);
  kern<<<grid, kThreads, F8Layout::kSmemRequest, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_fp8(bool causal, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const Fp8FwdParams &p, cudaStream_t stream) {
  return causal ? launch_fwd_fp8_t<true>(tq, tk, tv, p, stream) : launch_fwd_fp8_t<false>(tq, tk, tv, p, stream);
}

}  // namespace fa
