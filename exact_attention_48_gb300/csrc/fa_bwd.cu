// fa_bwd.cu -- backward kernels of exact attention for sm_103a.
//
// The backward pass does not keep the N x N probabilities of the forward
// pass; it recomputes them block by block from Q, K and the saved
// logsumexp (lexicon page "FlashAttention" (urworte.de), "Methodische
// Grundlagen", paragraph "Neuberechnung statt Speicherung").  With
// P = exp(s Q K^T - LSE) and dO given:
//     dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  D = rowsum(dO o O),
//     dK = s dS^T Q,  dQ = s dS K.
//
// Three launches on the caller's stream:
//   1. fa_bwd_pre_kernel   D = rowsum(dO o O) per query row (fp32), the
//                          saved logsumexp in log2 units, both padded to
//                          whole blocks, and a zeroed fp32 dQ accumulator.
//   2. fa_bwd_main_kernel  one CTA per (head, block of 128 keys): K_j and V_j
//                          stay in shared memory, dK_j and dV_j accumulate in
//                          TMEM over all query blocks i, and each block's
//                          dQ_i contribution is added into the fp32
//                          accumulator with vector atomics.
//   3. fa_bwd_dq_kernel    dq = bf16(s * accumulator).
//
// Main kernel roles (384 threads):
//   warp 0      TMA producer: K_j, V_j once; Q_i and dO_i into a 2-stage ring
//   warp 1      MMA issuer (one thread)
//   warp 2      owns the TMEM allocation
//   warps 4..7  one key row per thread, in two phases per query block:
//               P^T from S^T and the saved LSE, written as bf16 to TMEM (A
//               operand of dV += P^T dO) and kept in registers; then
//               dS^T = P^T o (dP^T - D) written as bf16 to shared memory
//               (operand of dK += dS^T Q and, read MN-major, of dQ = dS K);
//               final dV epilogue
//   warps 8..11 one query row per thread: drain dQ_i from TMEM into the
//               fp32 accumulator; final dK epilogue
//
// The products are computed transposed (S^T = K Q_i^T, dP^T = V dO_i^T) so
// that the key row, which owns dK/dV, is the TMEM lane.
//
// TMEM columns: S^T [0,128) (P^T as bf16 pairs over its first 64 columns),
// dP^T [128,256), dV [256,256+d), dK [256+d,256+2d).  For d = 128 that is
// all 512 columns and dQ_i reuses the dP^T columns once dS has been formed;
// for d = 64 dQ has its own columns [384,448).

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kBlk = 128;  // keys per CTA and queries per step
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ pre

template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const BwdParams p) {
  // One padded row per kTpr threads: rows q < N of every head get
  // D = rowsum(dO o O), lse * log2(e) and a zeroed dQ accumulator row; the
  // padding rows up to the next multiple of 128 get D = 0 and lse = +inf
  // (probability 0), so the main kernel reads whole blocks without checks.
  constexpr int kTpr = D / 8;  // threads per row: 8 bf16 (16 bytes) each
  constexpr int kRowsPerBlock = 256 / kTpr;
  const int Np = p.num_blk * kBlk;
  const long long prow = static_cast<long long>(blockIdx.x) * kRowsPerBlock + threadIdx.x / kTpr;
  const bool in_range = prow < static_cast<long long>(p.BH) * Np;
  const int bh = in_range ? static_cast<int>(prow / Np) : 0;
  const int q = in_range ? static_cast<int>(prow % Np) : 0;
  const bool real = in_range && q < p.N;
  const long long row = static_cast<long long>(bh) * p.N + q;
  const int part = threadIdx.x % kTpr;
  float acc = 0.0f;
  if (real) {
    const uint4 ov = reinterpret_cast<const uint4 *>(p.o + row * D)[part];
    const uint4 dv = reinterpret_cast<const uint4 *>(p.dout + row * D)[part];
    const __nv_bfloat162 *o2 = reinterpret_cast<const __nv_bfloat162 *>(&ov);
    const __nv_bfloat162 *d2 = reinterpret_cast<const __nv_bfloat162 *>(&dv);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = __bfloat1622float2(o2[i]);
      const float2 b = __bfloat1622float2(d2[i]);
      acc = fmaf(a.x, b.x, acc);
      acc = fmaf(a.y, b.y, acc);
    }
    float4 *z = reinterpret_cast<float4 *>(p.dq_acc + row * D) + 2 * part;
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = kTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (in_range && part == 0) {
    p.delta[prow] = acc;
    p.lse2[prow] = real ? p.lse[row] * kLog2e : INFINITY;
  }
}

// ------------------------------------------------------------------ dq convert

template <int D>
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const BwdParams p) {
  const long long n4 = static_cast<long long>(p.BH) * p.N * D / 4;
  const float s = p.scale;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 a = reinterpret_cast<const float4 *>(p.dq_acc)[i];
    uint2 out;
    out.x = pack_bf16x2(a.x * s, a.y * s);
    out.y = pack_bf16x2(a.z * s, a.w * s);
    reinterpret_cast<uint2 *>(p.dq)[i] = out;
  }
}

// ------------------------------------------------------------------ main

template <int D>
struct BwdLayout {
  static constexpr int kSlabs = D / 64;
  static constexpr int kStages = 2;
  static constexpr uint32_t kTile = kBlk * D * 2;  // one [128][D] bf16 tile
  static constexpr uint32_t kOffK = 0;
  static constexpr uint32_t kOffV = kOffK + kTile;
  static constexpr uint32_t kOffQ = kOffV + kTile;                 // kStages tiles
  static constexpr uint32_t kOffDO = kOffQ + kStages * kTile;      // kStages tiles
  static constexpr uint32_t kOffDS = kOffDO + kStages * kTile;     // [128 keys][128 queries] bf16
  static constexpr uint32_t kOffBar = kOffDS + kBlk * kBlk * 2;
  // kv_full, qdo_full[2], qdo_empty[2], s_full, dp_full, p_ready, ds_ready, dq_full, dq_empty,
  // acc_done, drain
  static constexpr int kNumBars = 1 + 2 * kStages + 8;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kBytes = kOffMisc + 16;
  static constexpr uint32_t kSmemRequest = kBytes + 1024;
  static_assert(kSmemRequest <= 232448, "shared memory budget");
  // TMEM columns
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  static constexpr bool kDqAliasesDP = (D == 128);
  static constexpr uint32_t kColDQ = kDqAliasesDP ? kColDP : 384;
};

constexpr uint32_t kTmemCols = 512;

// Register split over the three warpgroups: 168 per thread at launch
// (384 x 168 fits the SM); control 120, key-row warps 240, dQ drain 144:
// 128 * (120 + 240 + 144) = 384 * 168, and per SM sub-partition (one warp of
// each warpgroup) 32 * (120 + 240 + 144) <= 16384.
constexpr uint32_t kRegsLaunch = 168, kRegsControl = 120, kRegsRows = 240, kRegsDrain = 144;
static_assert(128 * (kRegsControl + kRegsRows + kRegsDrain) <= 384 * kRegsLaunch, "register split");

// Byte offset of element (row, col) in a 128-byte-swizzled tile made of
// 64-column slabs of `rows` rows (the layout the TMA loads produce).
__device__ __forceinline__ uint32_t sw128_offset(int row, int col, int rows) {
  return static_cast<uint32_t>((col >> 6) * rows * 128 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) +
                               (col & 7) * 2);
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    fa_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const BwdParams p) {
  using L = BwdLayout<D>;
  constexpr int S = L::kStages;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
  uint64_t *kv_full = bars;
  uint64_t *qdo_full = bars + 1;
  uint64_t *qdo_empty = qdo_full + S;
  uint64_t *s_full = qdo_empty + S;
  uint64_t *dp_full = s_full + 1;
  uint64_t *p_ready = dp_full + 1;
  uint64_t *ds_ready = p_ready + 1;
  uint64_t *dq_full = ds_ready + 1;
  uint64_t *dq_empty = dq_full + 1;
  uint64_t *acc_done = dq_empty + 1;
  uint64_t *drain = acc_done + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 4);
  const WaitCtl ctl{abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = p.N;
  const int nblk = p.num_blk;

  // Tile order: causal puts the key blocks with the most query blocks
  // (j small) first; otherwise the key blocks of one head run together.
  int bh, jblk;
  if (CAUSAL) {
    jblk = static_cast<int>(blockIdx.x) / p.BH;
    bh = static_cast<int>(blockIdx.x) % p.BH;
  } else {
    bh = static_cast<int>(blockIdx.x) / nblk;
    jblk = static_cast<int>(blockIdx.x) % nblk;
  }
  // Query blocks visited: causal i = j .. nblk-1; otherwise all blocks,
  // starting at j so that the CTAs of one head add into different dQ rows.
  const int n_q = CAUSAL ? (nblk - jblk) : nblk;
  auto qblock = [&](int t) { return CAUSAL ? jblk + t : (jblk + t) % nblk; };

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&qdo_full[s], 1);
      mbar_init(&qdo_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_ready, 128);
    mbar_init(ds_ready, 128);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 128);
    mbar_init(acc_done, 1);
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

  uint8_t *sK = smem + L::kOffK;
  uint8_t *sV = smem + L::kOffV;
  uint8_t *sQ = smem + L::kOffQ;
  uint8_t *sDO = smem + L::kOffDO;
  uint8_t *sDS = smem + L::kOffDS;

  if (warp < 4) {
    regs_decrease<kRegsControl>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(kv_full, 2 * L::kTile);
#pragma unroll
      for (int s = 0; s < L::kSlabs; ++s) {
        tma_load_3d(sK + s * kBlk * 128, &tm_k, kv_full, s * 64, jblk * kBlk, bh);
        tma_load_3d(sV + s * kBlk * 128, &tm_v, kv_full, s * 64, jblk * kBlk, bh);
      }
      int issued = 0;
      for (int t = 0; t < n_q; ++t) {
        const int st = t % S;
        if (!mbar_wait(&qdo_empty[st], ((t / S) & 1) ^ 1, ctl, kSiteDoEmpty)) break;
        mbar_arrive_expect_tx(&qdo_full[st], 2 * L::kTile);
        const int i = qblock(t);
#pragma unroll
        for (int s = 0; s < L::kSlabs; ++s) {
          tma_load_3d(sQ + st * L::kTile + s * kBlk * 128, &tm_q, &qdo_full[st], s * 64, i * kBlk, bh);
          tma_load_3d(sDO + st * L::kTile + s * kBlk * 128, &tm_do, &qdo_full[st], s * 64, i * kBlk, bh);
        }
        issued = t + 1;
      }
      if (*abort_flag) {
        mbar_drain(kv_full, 0);
        for (int t = (issued > S ? issued - S : 0); t < issued; ++t) mbar_drain(&qdo_full[t % S], (t / S) & 1);
      }
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t kIdescSq = idesc_bf16(kBlk, kBlk, false, false);  // S^T, dP^T
      constexpr uint32_t kIdescKB = idesc_bf16(kBlk, D, false, true);      // dV (TMEM A), dK
      constexpr uint32_t kIdescQ = idesc_bf16(kBlk, D, true, true);        // dQ
      const uint32_t aK = smem_addr(sK), aV = smem_addr(sV), aQ = smem_addr(sQ), aDO = smem_addr(sDO),
                     aDS = smem_addr(sDS);
      const uint32_t tS = tmem + L::kColS, tDP = tmem + L::kColDP, tDV = tmem + L::kColDV,
                     tDK = tmem + L::kColDK, tDQ = tmem + L::kColDQ;
      // S^T = K Q_t^T and dP^T = V dO_t^T (all operands K-major over d)
      auto issue_s = [&](int t) {
        const uint32_t q_base = aQ + (t % S) * L::kTile;
#pragma unroll 1
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kBlk * 128) + (kk & 3) * 32;
          mma_ss(tS, sdesc_sw128(aK + off, 16, 1024), sdesc_sw128(q_base + off, 16, 1024), kIdescSq, kk > 0);
        }
        tc_commit(s_full);
      };
      auto issue_dp = [&](int t) {
        const uint32_t do_base = aDO + (t % S) * L::kTile;
#pragma unroll 1
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kBlk * 128) + (kk & 3) * 32;
          mma_ss(tDP, sdesc_sw128(aV + off, 16, 1024), sdesc_sw128(do_base + off, 16, 1024), kIdescSq, kk > 0);
        }
        tc_commit(dp_full);
      };

      // Order per query block t:  dV_t, dQ_t, dK_t, S^T_{t+1}, dP^T_{t+1}.
      // The row warps form P_{t+1} while dP^T_{t+1} runs and dS_{t+1} while
      // dV_{t+1} runs; dQ_t drains while dK_t and S^T_{t+1} run.
      bool ok = mbar_wait(kv_full, 0, ctl, kSiteKvFull) && mbar_wait(&qdo_full[0], 0, ctl, kSiteDoFull);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        issue_dp(0);
      }
      for (int t = 0; ok && t < n_q; ++t) {
        const int st = t % S;
        const uint32_t q_base = aQ + st * L::kTile, do_base = aDO + st * L::kTile;
        // dV += P^T dO_t   (P^T from TMEM; dO_t is MN-major over d)
        if (!(ok = mbar_wait(p_ready, t & 1, ctl, kSitePReady))) break;
        tc_fence_after();
#pragma unroll 1
        for (int kk = 0; kk < kBlk / 16; ++kk)
          mma_ts(tDV, tS + kk * 8, sdesc_sw128(do_base + kk * 2048, kBlk * 128, 1024), kIdescKB, (t > 0 || kk > 0));
        if (!(ok = mbar_wait(ds_ready, t & 1, ctl, kSiteDsReady))) break;
        if (!L::kDqAliasesDP && t > 0 && !(ok = mbar_wait(dq_empty, (t - 1) & 1, ctl, kSiteDqEmpty))) break;
        tc_fence_after();
        // dQ_t = dS K   (dS read MN-major from the dS^T tile; K MN-major over d)
#pragma unroll 1
        for (int kk = 0; kk < kBlk / 16; ++kk)
          mma_ss(tDQ, sdesc_sw128(aDS + kk * 2048, kBlk * 128, 1024), sdesc_sw128(aK + kk * 2048, kBlk * 128, 1024),
                 kIdescQ, kk > 0);
        tc_commit(dq_full);
        // dK += dS^T Q_t   (dS^T K-major over queries; Q_t MN-major over d)
#pragma unroll 1
        for (int kk = 0; kk < kBlk / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kBlk * 128) + (kk & 3) * 32;
          mma_ss(tDK, sdesc_sw128(aDS + off, 16, 1024), sdesc_sw128(q_base + kk * 2048, kBlk * 128, 1024), kIdescKB,
                 (t > 0 || kk > 0));
        }
        tc_commit(&qdo_empty[st]);
        if (t + 1 < n_q) {
          const int nst = (t + 1) % S;
          if (!(ok = mbar_wait(&qdo_full[nst], ((t + 1) / S) & 1, ctl, kSiteDoFull))) break;
          tc_fence_after();
          issue_s(t + 1);
          if (L::kDqAliasesDP) {
            // dQ_t sits in the dP^T columns until it has been drained
            if (!(ok = mbar_wait(dq_empty, t & 1, ctl, kSiteDqEmpty))) break;
            tc_fence_after();
          }
          issue_dp(t + 1);
        }
      }
      if (ok) tc_commit(acc_done);
      tc_commit(drain);
      mbar_drain(drain, 0);
    }
  } else if (warp < 8) {
    regs_increase<kRegsRows>();
    // ------------------------------------------------------------ P^T, dS^T (one key row per thread)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // key row within the block
    const int key = jblk * kBlk + r;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + L::kColS + lane_base, tDP = tmem + L::kColDP + lane_base;
    const float c = p.scale_log2;
    const int Np = nblk * kBlk;
    const float *lse2_h = p.lse2 + static_cast<size_t>(bh) * Np;
    const float *delta_h = p.delta + static_cast<size_t>(bh) * Np;
    const uint32_t ds_row = smem_addr(sDS);
    bool ok = true;

    for (int t = 0; t < n_q; ++t) {
      const int i = qblock(t);
      // per-query statistics of this block (same for every thread: L1 broadcasts)
      const float4 *lse4 = reinterpret_cast<const float4 *>(lse2_h + i * kBlk);
      const float4 *del4 = reinterpret_cast<const float4 *>(delta_h + i * kBlk);
      const bool diag = CAUSAL && (i == jblk);
      const bool key_ok = key < N;

      // Phase 1: P^T = exp2(S^T c - lse2) -> bf16 over S^T columns [0, 64).
      ok = mbar_wait(s_full, t & 1, ctl, kSiteSFull);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t pk[64];  // P^T row, bf16 pairs, kept for phase 2
#pragma unroll
      for (int ch = 0; ch < kBlk / 32; ++ch) {
        uint32_t sv[32];
        tmem_ld32(tS + ch * 32, sv);
        tmem_ld_wait(sv);
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const int qc = ch * 32 + e;  // query column within the block
          const float4 l4 = __ldg(lse4 + qc / 4);
          const float2 x01 = ffma2(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), make_float2(c, c),
                                   make_float2(-l4.x, -l4.y));
          const float2 x23 = ffma2(make_float2(__uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3])),
                                   make_float2(c, c), make_float2(-l4.z, -l4.w));
          float pr[4] = {ex2(x01.x), ex2(x01.y), ex2(x23.x), ex2(x23.y)};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (diag) pr[u] = (qc + u >= r) ? pr[u] : 0.0f;  // key r visible to query qc+u iff r <= qc+u
            if (!key_ok) pr[u] = 0.0f;
          }
          pk[qc / 2] = pack_bf16x2(pr[0], pr[1]);
          pk[qc / 2 + 1] = pack_bf16x2(pr[2], pr[3]);
        }
        // columns [16 ch, 16 ch + 16) of S^T hold queries already read
        uint32_t part[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) part[u] = pk[ch * 16 + u];
        tmem_st16(tS + ch * 16, part);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_ready);

      // Phase 2: dS^T = P^T o (dP^T - D) -> bf16 into the swizzled dS^T tile.
      ok = mbar_wait(dp_full, t & 1, ctl, kSiteSFull);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < kBlk / 32; ++ch) {
        uint32_t dpv[32];
        tmem_ld32(tDP + ch * 32, dpv);
        tmem_ld_wait(dpv);
        uint32_t dk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const int qc = ch * 32 + e;
          const float4 d4 = __ldg(del4 + qc / 4);
          const uint32_t p01 = pk[qc / 2], p23 = pk[qc / 2 + 1];
          const float2 g01 = fadd2(make_float2(__uint_as_float(dpv[e]), __uint_as_float(dpv[e + 1])),
                                   make_float2(-d4.x, -d4.y));
          const float2 g23 = fadd2(make_float2(__uint_as_float(dpv[e + 2]), __uint_as_float(dpv[e + 3])),
                                   make_float2(-d4.z, -d4.w));
          const float2 ds01 = ffma2(make_float2(__uint_as_float(p01 << 16), __uint_as_float(p01 & 0xFFFF0000u)), g01,
                                    make_float2(0.f, 0.f));
          const float2 ds23 = ffma2(make_float2(__uint_as_float(p23 << 16), __uint_as_float(p23 & 0xFFFF0000u)), g23,
                                    make_float2(0.f, 0.f));
          dk[e / 2] = pack_bf16x2(ds01.x, ds01.y);
          dk[e / 2 + 1] = pack_bf16x2(ds23.x, ds23.y);
        }
        // dS^T row r, queries [32 ch, 32 ch + 32): four 16-byte chunks
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t addr = ds_row + sw128_offset(r, ch * 32 + u * 8, kBlk);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(dk[4 * u]), "r"(dk[4 * u + 1]),
                       "r"(dk[4 * u + 2]), "r"(dk[4 * u + 3])
                       : "memory");
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(ds_ready);
    }
    // dV epilogue
    if (ok) {
      ok = mbar_wait(acc_done, 0, ctl, kSiteMmaDone);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      __nv_bfloat16 *dst = p.dv + (static_cast<size_t>(bh) * N + key) * D;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32(tmem + L::kColDV + lane_base + ch * 32, v);
        tmem_ld_wait(v);
        if (key < N) {
          uint4 *d4 = reinterpret_cast<uint4 *>(dst + ch * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            d4[u] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * u]), __uint_as_float(v[8 * u + 1])),
                               pack_bf16x2(__uint_as_float(v[8 * u + 2]), __uint_as_float(v[8 * u + 3])),
                               pack_bf16x2(__uint_as_float(v[8 * u + 4]), __uint_as_float(v[8 * u + 5])),
                               pack_bf16x2(__uint_as_float(v[8 * u + 6]), __uint_as_float(v[8 * u + 7])));
        }
      }
    }
  } else {
    regs_decrease<kRegsDrain>();
    // ------------------------------------------------------------ dQ drain (one query row per thread)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tDQ = tmem + L::kColDQ + lane_base;
    bool ok = true;
    for (int t = 0; t < n_q; ++t) {
      ok = mbar_wait(dq_full, t & 1, ctl, kSiteDqFull);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int q = qblock(t) * kBlk + r;
      float4 *dst = reinterpret_cast<float4 *>(p.dq_acc + (static_cast<size_t>(bh) * N + q) * D);
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32(tDQ + ch * 32, v);
        tmem_ld_wait(v);
        if (q < N) {
#pragma unroll
          for (int u = 0; u < 8; ++u)
            atomicAdd(dst + ch * 8 + u, make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                                                    __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3])));
        }
      }
      tc_fence_before();
      mbar_arrive(dq_empty);
    }
    // dK epilogue (scale applied here)
    if (ok) {
      ok = mbar_wait(acc_done, 0, ctl, kSiteMmaDone);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const int key = jblk * kBlk + r;
      const float s = p.scale;
      __nv_bfloat16 *dst = p.dk + (static_cast<size_t>(bh) * N + key) * D;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32(tmem + L::kColDK + lane_base + ch * 32, v);
        tmem_ld_wait(v);
        if (key < N) {
          uint4 *d4 = reinterpret_cast<uint4 *>(dst + ch * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            d4[u] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * u]) * s, __uint_as_float(v[8 * u + 1]) * s),
                               pack_bf16x2(__uint_as_float(v[8 * u + 2]) * s, __uint_as_float(v[8 * u + 3]) * s),
                               pack_bf16x2(__uint_as_float(v[8 * u + 4]) * s, __uint_as_float(v[8 * u + 5]) * s),
                               pack_bf16x2(__uint_as_float(v[8 * u + 6]) * s, __uint_as_float(v[8 * u + 7]) * s));
        }
      }
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
cudaError_t launch_bwd_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tdo,
                         const BwdParams &p, cudaStream_t stream, cudaEvent_t ev_start, cudaEvent_t ev_stop) {
  using L = BwdLayout<D>;
  const long long rows = static_cast<long long>(p.BH) * p.N;
  const long long padded_rows = static_cast<long long>(p.BH) * p.num_blk * kBlk;
  constexpr int kRowsPerBlock = 256 / (D / 8);
  fa_bwd_pre_kernel<D>
      <<<static_cast<unsigned>((padded_rows + kRowsPerBlock - 1) / kRowsPerBlock), 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  auto kern = fa_bwd_main_kernel<D, CAUSAL>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemRequest);
  if (e != cudaSuccess) return e;
  if (ev_start && (e = cudaEventRecord(ev_start, stream)) != cudaSuccess) return e;
  kern<<<static_cast<unsigned>(p.BH) * static_cast<unsigned>(p.num_blk), 384, L::kSmemRequest, stream>>>(tq, tk, tv,
                                                                                                       tdo, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (ev_stop && (e = cudaEventRecord(ev_stop, stream)) != cudaSuccess) return e;

  const long long n4 = rows * D / 4;
  long long blocks = (n4 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  fa_bwd_dq_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(int d, bool causal, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tdo, const BwdParams &p, cudaStream_t stream, cudaEvent_t ev_start,
                       cudaEvent_t ev_stop) {
  if (d == 64)
    return causal ? launch_bwd_t<64, true>(tq, tk, tv, tdo, p, stream, ev_start, ev_stop)
                  : launch_bwd_t<64, false>(tq, tk, tv, tdo, p, stream, ev_start, ev_stop);
  return causal ? launch_bwd_t<128, true>(tq, tk, tv, tdo, p, stream, ev_start, ev_stop)
                : launch_bwd_t<128, false>(tq, tk, tv, tdo, p, stream, ev_start, ev_stop);
}

}  // namespace fa
