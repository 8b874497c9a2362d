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
// Three launches, none with atomics, so every output is bitwise
// reproducible:
//   1. fa_bwd_pre_kernel   D = rowsum(dO o O) per query row (fp32) and the
//                          saved logsumexp in log2 units, both padded to
//                          whole blocks of 128 rows.
//   2. fa_bwd_dkdv_kernel  one CTA per (head, block of 128 keys): K_j, V_j
//                          stay in shared memory, dK_j and dV_j accumulate in
//                          TMEM over the query blocks (4 products per block).
//   3. fa_bwd_dq_kernel    one CTA per (head, block of 128 queries): Q_i and
//                          dO_i stay in TMEM, dQ_i accumulates in TMEM over
//                          the key blocks (3 products per block).
// The dQ kernel reads only the inputs and the pre-kernel's statistics, so
// it runs on a side stream next to the dK/dV kernel (forked from and joined
// back to the caller's stream).  On short sequences both kernels
// give each CTA a pair of mirror blocks of one head instead of one block.
// Splitting dQ off costs two recomputed products per block pair but removes
// the fp32 reduction of dQ across key blocks through L2, which otherwise
// bounds the backward pass.
//
// Both main kernels: warp 0 TMA producer, warp 1 MMA issuer (one thread),
// warp 2 TMEM owner; the row warps from warp 4 on own one row each (key row
// in dK/dV, query row in dQ), two or four warps per row, each taking a
// slice of the row's 128 columns; they work in two phases per block: P from
// the scores, then dS from dP.

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kBlk = 128;  // rows per block, keys and queries alike
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kTmemCols = 512;
// Warps 0..3 are the control warpgroup (producer, MMA issuer, TMEM owner),
// warps 4..11 the row warps: two warpgroups that split each 128-wide row of
// scores between them (columns [0,64) and [64,128)), so that every SM
// sub-partition runs two row warps and one can issue while the other waits.
constexpr int kThreads = 384;
constexpr int kRowWarps = 8;  // row warps; each signals its barriers once (lane 0)
// The dK/dV kernel splits each key row over RG row warpgroups (RG = 2 or
// 4, a template parameter): RG = 4 gives each warp a quarter of the 128
// query columns, twice the warps per SM sub-partition to hide the latency
// of the row phases and half the work per thread (+3 % on long non-causal
// heads, measured); with few query blocks per CTA (causal) the larger CTA
// costs more than it hides (-8 % causal N = 4096), so causal keeps RG = 2.
// Per element the arithmetic is the same either way: the results are
// bitwise equal.
template <int RG>
struct KvRows {
  static constexpr int kThreads = 128 + 128 * RG;
  static constexpr int kRowWarps = 4 * RG;
  static constexpr int kCols = kBlk / RG;  // query columns per row thread
};

// ------------------------------------------------------------------ pre

template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const BwdParams p) {
  // One padded row per kTpr threads: rows q < N of every head get
  // D = rowsum(dO o O) and lse * log2(e); the padding rows up to the next
  // multiple of 128 get D = 0 and lse = +inf (probability 0), so the main
  // kernels read whole blocks without checks.  The grid strides over the
  // rows (block-uniform trip count, so every warp's shuffles see all lanes).
  constexpr int kTpr = D / 8;  // threads per row: 8 bf16 (16 bytes) each
  constexpr int kRowsPerBlock = 256 / kTpr;
  const int Np = p.num_blk * kBlk;
  const long long rows = static_cast<long long>(p.BH) * Np;
  const int part = threadIdx.x % kTpr;
  for (long long base = static_cast<long long>(blockIdx.x) * kRowsPerBlock; base < rows;
       base += static_cast<long long>(gridDim.x) * kRowsPerBlock) {
    const long long prow = base + threadIdx.x / kTpr;
    const bool in_range = prow < rows;
    const int bh = in_range ? static_cast<int>(prow / Np) : 0;
    const int q = in_range ? static_cast<int>(prow % Np) : 0;
    const SeqRange seq = seq_range(p.cu_seqlens, bh / p.H, p.N, p.T);
    const bool real = in_range && q < seq.len;
    const int trow = seq.start + q;  // the row on the tensors' row axis
    float acc = 0.0f;
    if (real) {
      const uint4 ov = reinterpret_cast<const uint4 *>(p.o + row_offset(p.so, bh, p.H, trow))[part];
      const uint4 dv = reinterpret_cast<const uint4 *>(p.dout + row_offset(p.sdo, bh, p.H, trow))[part];
      const __nv_bfloat162 *o2 = reinterpret_cast<const __nv_bfloat162 *>(&ov);
      const __nv_bfloat162 *d2 = reinterpret_cast<const __nv_bfloat162 *>(&dv);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 a = __bfloat1622float2(o2[i]);
        const float2 b = __bfloat1622float2(d2[i]);
        acc = fmaf(a.x, b.x, acc);
        acc = fmaf(a.y, b.y, acc);
      }
    }
#pragma unroll
    for (int off = kTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (in_range && part == 0) {
      p.delta[prow] = acc;
      p.lse2[prow] = real ? p.lse[(bh / p.H) * p.lse_b + (bh % p.H) * p.lse_h + trow] * kLog2e : INFINITY;
    }
  }
}

// ------------------------------------------------------------------ shared pieces

// One row of a TMEM accumulator (lane = row, D fp32 columns), times `mul`,
// into a bf16 row of global memory.
template <int D>
__device__ __forceinline__ void store_acc_row(uint32_t taddr, __nv_bfloat16 *dst, bool store, float mul) {
#pragma unroll 1
  for (int ch = 0; ch < D / 32; ++ch) {
    uint32_t v[32];
    tmem_ld32(taddr + ch * 32, v);
    tmem_ld_wait(v);
    if (store) {
      uint4 *d4 = reinterpret_cast<uint4 *>(dst + ch * 32);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        d4[u] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * u]) * mul, __uint_as_float(v[8 * u + 1]) * mul),
                           pack_bf16x2(__uint_as_float(v[8 * u + 2]) * mul, __uint_as_float(v[8 * u + 3]) * mul),
                           pack_bf16x2(__uint_as_float(v[8 * u + 4]) * mul, __uint_as_float(v[8 * u + 5]) * mul),
                           pack_bf16x2(__uint_as_float(v[8 * u + 6]) * mul, __uint_as_float(v[8 * u + 7]) * mul));
    }
  }
}

template <int D>
struct BwdLayout {
  static constexpr int kSlabs = D / 64;
  static constexpr int kStages = 2;
  static constexpr uint32_t kTile = kBlk * D * 2;  // one [128][D] bf16 tile
  // Both kernels hold two resident tiles (K, V or Q, dO), a 2-stage ring of
  // two tiles (Q, dO or K, V) and one [128][128] bf16 dS tile.
  static constexpr uint32_t kOffRes0 = 0;
  static constexpr uint32_t kOffRes1 = kOffRes0 + kTile;
  static constexpr uint32_t kOffRing0 = kOffRes1 + kTile;             // kStages tiles
  static constexpr uint32_t kOffRing1 = kOffRing0 + kStages * kTile;  // kStages tiles
  // per ring stage, the query block's row statistics: lse*log2(e) [128]
  // then D [128] (fp32), loaded with Q and dO
  static constexpr uint32_t kStatBytes = 2 * kBlk * 4;
  static constexpr uint32_t kOffStats = kOffRing1 + kStages * kTile;
  static constexpr uint32_t kOffBar = kOffStats + kStages * kStatBytes;
  static constexpr int kNumBars = 16;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kBytes = kOffMisc + 16;
  static constexpr uint32_t kSmemRequest = kBytes + 1024;
  static_assert(kSmemRequest <= 232448, "shared memory budget");
};

// ------------------------------------------------------------------ dK, dV

// TMEM columns: S^T [0,128) (P^T of queries [64h, 64h+64) as bf16 pairs
// over columns [64h, 64h+32), h = 0, 1: each half writes over scores it has
// already read), dP^T [128,256) (dS^T the same way over columns
// [128+64h, 128+64h+32)), dV [256,256+D), dK [256+D,256+2D).  The products
// are formed transposed (S^T = K Q^T, dP^T = V dO^T) so the key row, which
// owns dK and dV, is the TMEM lane; P^T and dS^T are then the TMEM A
// operands of dV += P^T dO and dK += dS^T Q, and never touch shared memory.
// MMA order per query block t:
//   dV(t), S^T(t+1), dK(t), dP^T(t+1)
// so P^T(t+1) is formed while dK(t) and dP^T(t+1) run, and dS^T(t+1) while
// dV(t+1) and S^T(t+2) run.  Each product that overwrites a TMEM region
// comes after the one that reads it (the tensor core runs them in order).
template <int D, bool CAUSAL, bool VARLEN, int RG, bool PAIRS>
__global__ void __launch_bounds__(KvRows<RG>::kThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const BwdParams p) {
  using L = BwdLayout<D>;
  constexpr int S = L::kStages;
  constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  constexpr int kKvCols = KvRows<RG>::kCols;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
  uint64_t *kv_full = bars;
  uint64_t *qdo_full = bars + 1;       // [S]
  uint64_t *qdo_empty = qdo_full + S;  // [S]
  uint64_t *s_full = qdo_empty + S;
  uint64_t *dp_full = s_full + 1;
  uint64_t *p_ready = dp_full + 1;
  uint64_t *ds_ready = p_ready + 1;
  uint64_t *acc_done = ds_ready + 1;
  uint64_t *drain = acc_done + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 4);
  const WaitCtl ctl{abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nblk = p.num_blk;  // blocks of the longest sequence (the padding of the row statistics)

  // Tile order.  With pairs (short sequences): a CTA takes two key blocks of
  // one head, j and its mirror nb-1-j (one block when they coincide); causal,
  // they see nb + 1 query blocks together whatever j is, so every CTA has
  // the same work; the second block's start overlaps the first one's end,
  // and the CTAs of a head run together.  Causal otherwise: one key block
  // per CTA, the blocks with the most query blocks (j small) first, across
  // all heads -- or head by head when the heaviest block is short against
  // each SM's share of the work, so that the blocks running together share
  // their Q and dO in L2.  Non-causal: the key blocks of one head run
  // together.
  constexpr bool pairs = PAIRS;
  int bh, j0;
  if (pairs) {
    bh = static_cast<int>(blockIdx.x) / ((nblk + 1) / 2);
    j0 = static_cast<int>(blockIdx.x) % ((nblk + 1) / 2);
  } else if (CAUSAL && !p.head_major) {
    j0 = static_cast<int>(blockIdx.x) / p.BH;
    bh = static_cast<int>(blockIdx.x) % p.BH;
  } else {
    bh = static_cast<int>(blockIdx.x) / nblk;
    j0 = static_cast<int>(blockIdx.x) % nblk;
  }
  // The block's sequence; a block past its end (packed mode) has no work.
  const SeqRange seq = VARLEN ? seq_range(p.cu_seqlens, bh / p.H, p.N, p.T) : SeqRange{0, p.N};
  const int N = seq.len, row0 = seq.start;
  const int nb = (N + kBlk - 1) / kBlk;  // blocks of this sequence
  if (VARLEN && (pairs ? 2 * j0 >= nb : j0 >= nb)) return;
  const int tma_h = bh % p.H, tma_b = VARLEN ? 0 : bh / p.H;
  const int n_items = (pairs && nb - 1 - j0 != j0) ? 2 : 1;
  // Key block of item `it`, and the query blocks it visits: causal
  // i = j .. nb-1; otherwise all of them.
  auto item_j = [&](int it) { return it == 0 ? j0 : nb - 1 - j0; };
  auto item_nq = [&](int it) { return CAUSAL ? nb - item_j(it) : nb; };

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&qdo_full[s], 1);
      mbar_init(&qdo_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_ready, KvRows<RG>::kRowWarps);
    mbar_init(ds_ready, KvRows<RG>::kRowWarps);
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

  uint8_t *sK = smem + L::kOffRes0;
  uint8_t *sV = smem + L::kOffRes1;
  uint8_t *sQ = smem + L::kOffRing0;
  uint8_t *sDO = smem + L::kOffRing1;
  uint8_t *sStats = smem + L::kOffStats;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      // (block counters run over both items: ring stages and barrier
      // phases carry on from the first item to the second)
      int issued = 0, kv_issued = 0;
      bool pok = true;
      for (int it = 0; pok && it < n_items; ++it) {
        const int jb = item_j(it), nq = item_nq(it), ib = CAUSAL ? jb : 0;
        // K and V of the second item replace the first's once every
        // product of the first is complete
        if (it > 0 && !(pok = mbar_wait(acc_done, (it - 1) & 1, ctl, kSiteKvEmpty))) break;
        mbar_arrive_expect_tx(kv_full, 2 * L::kTile);
#pragma unroll
        for (int s = 0; s < L::kSlabs; ++s) {
          tma_load_4d(sK + s * kBlk * 128, &tm_k, kv_full, s * 64, row0 + jb * kBlk, tma_h, tma_b);
          tma_load_4d(sV + s * kBlk * 128, &tm_v, kv_full, s * 64, row0 + jb * kBlk, tma_h, tma_b);
        }
        kv_issued = it + 1;
        for (int t = 0; t < nq; ++t) {
          const int g = issued, st = g % S;
          if (!(pok = mbar_wait(&qdo_empty[st], ((g / S) & 1) ^ 1, ctl, kSiteDoEmpty))) break;
          mbar_arrive_expect_tx(&qdo_full[st], 2 * L::kTile + L::kStatBytes);
          const int i = ib + t;
#pragma unroll
          for (int s = 0; s < L::kSlabs; ++s) {
            tma_load_4d(sQ + st * L::kTile + s * kBlk * 128, &tm_q, &qdo_full[st], s * 64, row0 + i * kBlk, tma_h,
                        tma_b);
            tma_load_4d(sDO + st * L::kTile + s * kBlk * 128, &tm_do, &qdo_full[st], s * 64, row0 + i * kBlk, tma_h,
                        tma_b);
          }
          const size_t srow = static_cast<size_t>(bh) * nblk * kBlk + static_cast<size_t>(i) * kBlk;
          bulk_load(sStats + st * L::kStatBytes, p.lse2 + srow, kBlk * 4, &qdo_full[st]);
          bulk_load(sStats + st * L::kStatBytes + kBlk * 4, p.delta + srow, kBlk * 4, &qdo_full[st]);
          issued = g + 1;
        }
      }
      // Every copy issued lands before this thread leaves, whatever the
      // other roles do (bounded waits; in a normal run they are done).
      // A K/V load is issued only after the previous one was consumed, so
      // the last one's phase covers both.
      if (kv_issued > 0) mbar_drain(kv_full, (kv_issued - 1) & 1);
      for (int t = (issued > S ? issued - S : 0); t < issued; ++t) mbar_drain(&qdo_full[t % S], (t / S) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescSq = idesc_bf16(kBlk, kBlk, false, false);  // S^T, dP^T
      constexpr uint32_t kIdescKV = idesc_bf16(kBlk, D, false, true);      // dV (TMEM A), dK
      const uint32_t aK = smem_addr(sK), aV = smem_addr(sV), aQ = smem_addr(sQ), aDO = smem_addr(sDO);
      const uint32_t tS = tmem + kColS, tDP = tmem + kColDP, tDV = tmem + kColDV, tDK = tmem + kColDK;

      // Descriptors: fixed tiles once, ring tiles per stage; every MMA adds
      // a compile-time step offset (all issue loops are unrolled).
      const uint64_t dK = sdesc_sw128(aK, 16, 1024), dV = sdesc_sw128(aV, 16, 1024);
      auto q_kmaj = [&](int t) { return sdesc_sw128(aQ + (t % S) * L::kTile, 16, 1024); };
      auto q_mn = [&](int t) { return sdesc_sw128(aQ + (t % S) * L::kTile, kBlk * 128, 1024); };
      auto do_kmaj = [&](int t) { return sdesc_sw128(aDO + (t % S) * L::kTile, 16, 1024); };
      auto do_mn = [&](int t) { return sdesc_sw128(aDO + (t % S) * L::kTile, kBlk * 128, 1024); };

      // S^T(t) = K Q_t^T and dP^T(t) = V dO_t^T (all operands K-major over d)
      auto issue_dp = [&](int t) {
        const uint64_t bdo = do_kmaj(t);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tDP, desc_add(dV, kmajor_step(kk, kBlk)), desc_add(bdo, kmajor_step(kk, kBlk)), kIdescSq, kk > 0);
        tc_commit(dp_full);
      };
      auto issue_s = [&](int t) {
        const uint64_t bq = q_kmaj(t);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tS, desc_add(dK, kmajor_step(kk, kBlk)), desc_add(bq, kmajor_step(kk, kBlk)), kIdescSq, kk > 0);
        tc_commit(s_full);
      };

      // g: block counter over both items (ring stage g % S, phases g & 1)
      bool ok = true;
      for (int it = 0, g0 = 0; ok && it < n_items; g0 += item_nq(it), ++it) {
        const int nq = item_nq(it);
        // (the second item's first S^T, dP^T overwrite columns the first
        // item's last dV, dK read: issued after them, they run after them)
        ok = mbar_wait(kv_full, it & 1, ctl, kSiteKvFull) && mbar_wait(&qdo_full[g0 % S], (g0 / S) & 1, ctl, kSiteDoFull);
        if (!ok) break;
        tc_fence_after();
        issue_s(g0);
        issue_dp(g0);
        for (int t = 0; ok && t < nq; ++t) {
          const int g = g0 + t;
          const bool more = t + 1 < nq;
          // dV += P^T dO_t   (P^T from TMEM; dO_t is MN-major over d).  The
          // item's first dV overwrites the accumulator: its rows arrive on
          // p_ready only after storing the previous item's dV and dK.
          if (!(ok = mbar_wait(p_ready, g & 1, ctl, kSitePReady))) break;
          tc_fence_after();
          {
            const uint64_t bdo = do_mn(g);
#pragma unroll
            for (int kk = 0; kk < kBlk / 16; ++kk)  // P^T of queries [c g, c g + c) sits at columns c g.. (c = kKvCols)
              mma_ts(tDV, tS + (kk / (kKvCols / 16)) * kKvCols + (kk % (kKvCols / 16)) * 8,
                     desc_add(bdo, mnmajor_step(kk)), kIdescKV, (t > 0 || kk > 0));
          }
          // S^T(t+1): the rows have read S^T(t) (p_ready) and dV(t), issued
          // first, reads P^T(t) before S^T(t+1) overwrites it
          if (more) {
            if (!(ok = mbar_wait(&qdo_full[(g + 1) % S], ((g + 1) / S) & 1, ctl, kSiteDoFull))) break;
            tc_fence_after();
            issue_s(g + 1);
          }
          // dK += dS^T Q_t (dS^T from TMEM over the dP^T columns; Q_t MN-major
          // over d), then dP^T(t+1) over them once dK(t) has read them
          if (!(ok = mbar_wait(ds_ready, g & 1, ctl, kSiteDsReady))) break;
          tc_fence_after();
          {
            const uint64_t bq = q_mn(g);
#pragma unroll
            for (int kk = 0; kk < kBlk / 16; ++kk)  // dS^T of queries [c g, c g + c) sits at columns 128 + c g..
              mma_ts(tDK, tDP + (kk / (kKvCols / 16)) * kKvCols + (kk % (kKvCols / 16)) * 8,
                     desc_add(bq, mnmajor_step(kk)), kIdescKV, (t > 0 || kk > 0));
          }
          tc_commit(&qdo_empty[g % S]);
          if (more) issue_dp(g + 1);
        }
        // the item's dV, dK are complete (the rows store them), and K, V
        // are free for the next item (the producer waits on this too)
        if (ok) tc_commit(acc_done);
      }
      tc_commit(drain);
      mbar_drain(drain, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ key rows
    const int grp = (warp >> 2) - 1;  // query columns [kKvCols grp, kKvCols (grp + 1))
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // key row within the block
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + kColS + lane_base, tDP = tmem + kColDP + lane_base;
    const float c = p.scale_log2;
    const int c0 = grp * kKvCols;  // first query column of this quarter
    bool ok = true;

    for (int it = 0, g0 = 0; ok && it < n_items; g0 += item_nq(it), ++it) {
      const int jblk = item_j(it), n_q = item_nq(it), i0 = CAUSAL ? jblk : 0;
      const int key = jblk * kBlk + r;
      const bool key_ok = key < N;
      for (int t = 0; t < n_q; ++t) {
        const int i = i0 + t, g = g0 + t;  // g: block counter over both items
        // per-query statistics of this block, in shared memory with Q and dO
        // (same address in every thread: broadcast reads)
        const float *stats = reinterpret_cast<const float *>(sStats + (g % S) * L::kStatBytes);
        const float4 *lse4 = reinterpret_cast<const float4 *>(stats + c0);
        const float4 *del4 = reinterpret_cast<const float4 *>(stats + kBlk + c0);
        const bool diag = CAUSAL && (i == jblk);

        // Phase 1: P^T = exp2(S^T c - lse2) -> bf16 over S^T columns [c0, c0 + kKvCols / 2).
        // (The stage's copies are complete once S^T(t) is; the rows wait on
        // them too so that the statistics' copy is visible to their loads.
        // The stage cannot be refilled before ds_ready(t).)
        ok = mbar_wait(s_full, g & 1, ctl, kSiteSFull) &&
             mbar_wait(&qdo_full[g % S], (g / S) & 1, ctl, kSiteDoFull);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // P^T of this quarter row in fp32 pairs (kept for phase 2) and as bf16
        // pairs in TMEM.  Key rows past N (zero rows of K, so S = 0) get a
        // finite P that only reaches their own dV, dK rows, which are not
        // stored: no mask needed.
        constexpr int kCh = kKvCols / 32;  // 32-column chunks per row thread
        float2 pf[kKvCols / 2];
        {
          uint32_t sva[kCh][32];
#pragma unroll
          for (int ch = 0; ch < kCh; ++ch) tmem_ld32(tS + c0 + ch * 32, sva[ch]);
#pragma unroll
          for (int ch = 0; ch < kCh; ++ch) tmem_ld_wait(sva[ch]);
#pragma unroll
          for (int ch = 0; ch < kCh; ++ch) {
            const uint32_t(&sv)[32] = sva[ch];
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const int qh = ch * 32 + e;  // query column within this thread's columns
              const float4 l4 = lse4[qh / 4];
              const float2 x01 = ffma2(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                       make_float2(c, c), make_float2(-l4.x, -l4.y));
              const float2 x23 = ffma2(make_float2(__uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3])),
                                       make_float2(c, c), make_float2(-l4.z, -l4.w));
              float pr[4] = {ex2(x01.x), ex2(x01.y), ex2(x23.x), ex2(x23.y)};
              if (diag) {
#pragma unroll
                for (int u = 0; u < 4; ++u) pr[u] = (c0 + qh + u >= r) ? pr[u] : 0.0f;  // key r visible to query q iff r <= q
              }
              pf[qh / 2] = make_float2(pr[0], pr[1]);
              pf[qh / 2 + 1] = make_float2(pr[2], pr[3]);
              pk[e / 2] = pack_bf16x2(pr[0], pr[1]);
              pk[e / 2 + 1] = pack_bf16x2(pr[2], pr[3]);
            }
            tmem_st16(tS + c0 + ch * 16, pk);  // over scores of this thread's columns, already read
          }
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(p_ready);

        // Phase 2: dS^T = P^T o (dP^T - D) -> bf16 pairs over this quarter's
        // own, already read, dP^T columns.
        ok = mbar_wait(dp_full, g & 1, ctl, kSiteSFull);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        {
          uint32_t dpa[kCh][32];
#pragma unroll
          for (int ch = 0; ch < kCh; ++ch) tmem_ld32(tDP + c0 + ch * 32, dpa[ch]);
#pragma unroll
          for (int ch = 0; ch < kCh; ++ch) tmem_ld_wait(dpa[ch]);
#pragma unroll
          for (int ch = 0; ch < kCh; ++ch) {
            const uint32_t(&dpv)[32] = dpa[ch];
            uint32_t dk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const int qh = ch * 32 + e;
              const float4 d4 = del4[qh / 4];
              const float2 g01 = fadd2(make_float2(__uint_as_float(dpv[e]), __uint_as_float(dpv[e + 1])),
                                       make_float2(-d4.x, -d4.y));
              const float2 g23 = fadd2(make_float2(__uint_as_float(dpv[e + 2]), __uint_as_float(dpv[e + 3])),
                                       make_float2(-d4.z, -d4.w));
              const float2 ds01 = fmul2(pf[qh / 2], g01);
              const float2 ds23 = fmul2(pf[qh / 2 + 1], g23);
              dk[e / 2] = pack_bf16x2(ds01.x, ds01.y);
              dk[e / 2 + 1] = pack_bf16x2(ds23.x, ds23.y);
            }
            tmem_st16(tDP + c0 + ch * 16, dk);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(ds_ready);
      }
      // epilogues: the first half of the row groups writes dV, the second dK
      // (scale applied here), each group a D / (RG / 2) column slice
      if (ok) {
        ok = mbar_wait(acc_done, it & 1, ctl, kSiteMmaDone);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) {
        tc_fence_after();
        constexpr int kW = D / (RG / 2);  // columns per group
        const int col = (grp % (RG / 2)) * kW;
        if (grp < RG / 2)
          store_acc_row<kW>(tmem + kColDV + lane_base + col, p.dv + row_offset(p.sdv, bh, p.H, row0 + key) + col,
                            key_ok, 1.0f);
        else
          store_acc_row<kW>(tmem + kColDK + lane_base + col, p.dk + row_offset(p.sdk, bh, p.H, row0 + key) + col,
                            key_ok, p.scale);
      }
    }  // items
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ dQ

template <int D>
struct DqLayout {
  static constexpr int kSlabs = D / 64;
  static constexpr int kKStages = 4, kVStages = 3;
  static constexpr uint32_t kTile = kBlk * D * 2;  // one [128][D] bf16 tile
  // K in a 4-stage ring, V in a 3-stage ring.  Q, dO and dS live in TMEM
  // (the A operands of S = Q K^T, dP = dO V^T and dQ = dS K), which leaves
  // the shared memory to the rings.
  static constexpr uint32_t kOffK = 0;
  static constexpr uint32_t kOffV = kOffK + kKStages * kTile;
  static constexpr uint32_t kOffBar = kOffV + kVStages * kTile;
  static constexpr int kNumBars = 24;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kBytes = kOffMisc + 16;
  static constexpr uint32_t kSmemRequest = kBytes + 1024;
  static_assert(kSmemRequest <= 232448, "shared memory budget");
};

// TMEM columns: S [0,128) (lane = query row), dP [128,256) (dS of keys
// [64h, 64h+64) as bf16 pairs over columns [128+64h, 128+64h+32), written by
// the rows over dP they have already read), dQ [256,256+D), dO
// [384, 384+D/2) and Q [448, 448+D/2) as bf16 pairs (copied in once by the
// rows).  Every product then reads only its B operand from shared memory.
// MMA order per key block j:  S(j+1), dQ(j), dP(j+1)
// so the rows form P(j+1) while dQ(j) and dP(j+1) run and dS(j+1) while
// S(j+2) runs; dP(j+1) overwrites dS(j) after dQ(j) has read it (the tensor
// core runs the products in order).  K(j) is read by S(j) and, last, by
// dQ(j); the third K stage lets K(j+2) load while dQ(j) still holds K(j).
template <int D, bool CAUSAL, bool VARLEN, bool PAIRS>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const BwdParams p) {
  using L = DqLayout<D>;
  constexpr int SK = L::kKStages, SV = L::kVStages;
  constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDO = 384, kColQ = 448;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
  uint64_t *do_ready = bars;          // Q and dO written to TMEM by the rows
  // kv_full[g % SK]: K and V of key block g have both landed (V in its own
  // ring, stage g % SV): one wait for the MMA thread per block
  uint64_t *kv_full = do_ready + 1;   // [SK]
  uint64_t *k_empty = kv_full + SK;   // [SK]
  uint64_t *v_empty = k_empty + SK;   // [SV]
  uint64_t *s_full = v_empty + SV;
  uint64_t *dp_full = s_full + 1;
  uint64_t *s_free = dp_full + 1;
  uint64_t *ds_ready = s_free + 1;
  uint64_t *dq_done = ds_ready + 1;
  uint64_t *drain = dq_done + 1;
  static_assert(1 + 2 * SK + SV + 6 <= L::kNumBars, "barrier slots");
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 4);
  const WaitCtl ctl{abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nblk = p.num_blk;  // blocks of the longest sequence (the padding of the row statistics)

  // Tile order.  With pairs (short sequences): a CTA takes the query blocks
  // nb-1-i and i of one head (one block when they coincide; causal, they see
  // nb + 1 key blocks together); the CTAs of a head run together.  Causal
  // otherwise: the query blocks with the most key blocks (i large) first,
  // across all heads or head by head (as the dK/dV kernel).  Non-causal: the
  // query blocks of one head run together.
  constexpr bool pairs = PAIRS;
  int bh, i0;  // i0: the first item's query block (pairs: its mirror's index)
  if (pairs) {
    bh = static_cast<int>(blockIdx.x) / ((nblk + 1) / 2);
    i0 = static_cast<int>(blockIdx.x) % ((nblk + 1) / 2);
  } else if (CAUSAL && !p.head_major) {
    i0 = nblk - 1 - static_cast<int>(blockIdx.x) / p.BH;
    bh = static_cast<int>(blockIdx.x) % p.BH;
  } else if (CAUSAL) {  // head by head, heaviest query blocks first
    bh = static_cast<int>(blockIdx.x) / nblk;
    i0 = nblk - 1 - static_cast<int>(blockIdx.x) % nblk;
  } else {
    bh = static_cast<int>(blockIdx.x) / nblk;
    i0 = static_cast<int>(blockIdx.x) % nblk;
  }
  // The block's sequence; a block past its end (packed mode) has no work.
  const SeqRange seq = VARLEN ? seq_range(p.cu_seqlens, bh / p.H, p.N, p.T) : SeqRange{0, p.N};
  const int N = seq.len, row0 = seq.start;
  const int nb = (N + kBlk - 1) / kBlk;  // blocks of this sequence
  if (VARLEN && (pairs ? 2 * i0 >= nb : i0 >= nb)) return;
  const int tma_h = bh % p.H, tma_b = VARLEN ? 0 : bh / p.H;
  const int n_items = (pairs && nb - 1 - i0 != i0) ? 2 : 1;
  // Query block of item `it` (pairs: the heavier one first) and the key
  // blocks 0 .. n_kv-1 it visits.
  auto item_i = [&](int it) { return pairs ? (it == 0 ? nb - 1 - i0 : i0) : i0; };
  auto item_nkv = [&](int it) { return CAUSAL ? item_i(it) + 1 : nb; };

  if (threadIdx.x == 0) {
    mbar_init(do_ready, kRowWarps);
    for (int s = 0; s < SK; ++s) {
      mbar_init(&kv_full[s], 2);  // the K and the V producer lane
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(s_free, kRowWarps);
    mbar_init(ds_ready, kRowWarps);
    mbar_init(dq_done, 1);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producers
    if (lane == 0) {
      // the K ring
      tma_prefetch_desc(&tm_k);
      // (the ring runs over both items' key blocks: stage g % SK)
      int issued = 0;
      bool pok = true;
      for (int it = 0; pok && it < n_items; ++it)
        for (int j = 0; j < item_nkv(it); ++j) {
          const int g = issued, st = g % SK;
          if (!(pok = mbar_wait(&k_empty[st], ((g / SK) & 1) ^ 1, ctl, kSiteKEmpty))) break;
          mbar_arrive_expect_tx(&kv_full[st], L::kTile);
#pragma unroll
          for (int s = 0; s < L::kSlabs; ++s)
            tma_load_4d(sK + st * L::kTile + s * kBlk * 128, &tm_k, &kv_full[st], s * 64, row0 + j * kBlk, tma_h,
                        tma_b);
          issued = g + 1;
        }
      for (int j = (issued > SK ? issued - SK : 0); j < issued; ++j) mbar_drain(&kv_full[j % SK], (j / SK) & 1);
    } else if (lane == 1) {
      // the V ring
      tma_prefetch_desc(&tm_v);
      int issued = 0;
      bool pok = true;
      for (int it = 0; pok && it < n_items; ++it)
        for (int j = 0; j < item_nkv(it); ++j) {
          const int g = issued, st = g % SV;
          if (!(pok = mbar_wait(&v_empty[st], ((g / SV) & 1) ^ 1, ctl, kSiteVEmpty))) break;
          mbar_arrive_expect_tx(&kv_full[g % SK], L::kTile);
#pragma unroll
          for (int s = 0; s < L::kSlabs; ++s)
            tma_load_4d(sV + st * L::kTile + s * kBlk * 128, &tm_v, &kv_full[g % SK], s * 64, row0 + j * kBlk, tma_h,
                        tma_b);
          issued = g + 1;
        }
      for (int j = (issued > SV ? issued - SV : 0); j < issued; ++j) mbar_drain(&kv_full[j % SK], (j / SK) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16(kBlk, kBlk, false, false);  // S, dP
      constexpr uint32_t kIdescQ = idesc_bf16(kBlk, D, false, true);      // dQ
      const uint32_t aK = smem_addr(sK), aV = smem_addr(sV);
      const uint32_t tS = tmem + kColS, tDP = tmem + kColDP, tDQ = tmem + kColDQ, tDO = tmem + kColDO,
                     tQ = tmem + kColQ;

      // Descriptors: fixed tiles once, ring tiles per stage; every MMA adds
      // a compile-time step offset (all issue loops are unrolled).
      auto k_kmaj = [&](int j) { return sdesc_sw128(aK + (j % SK) * L::kTile, 16, 1024); };
      auto k_mn = [&](int j) { return sdesc_sw128(aK + (j % SK) * L::kTile, kBlk * 128, 1024); };
      auto v_kmaj = [&](int j) { return sdesc_sw128(aV + (j % SV) * L::kTile, 16, 1024); };

      // S(j) = Q K_j^T (Q from TMEM, K_j K-major over d)
      auto issue_s = [&](int j) {
        const uint64_t bk = k_kmaj(j);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ts(tS, tQ + kk * 8, desc_add(bk, kmajor_step(kk, kBlk)), kIdescS, kk > 0);
        tc_commit(s_full);
      };
      // one K step of dP(j) = dO V_j^T (dO from TMEM, V_j K-major over d)
      auto dp_step = [&](uint64_t bv, int kk) {
        mma_ts(tDP, tDO + kk * 8, desc_add(bv, kmajor_step(kk, kBlk)), kIdescS, kk > 0);
      };

      // g: key-block counter over both items (ring stages, barrier phases)
      bool ok = true;
      for (int it = 0, g0 = 0; ok && it < n_items; g0 += item_nkv(it), ++it) {
        const int n_kv = item_nkv(it);
        // the item's Q and dO in TMEM (written by the rows once the previous
        // item's products were complete and its dQ was read out)
        ok = mbar_wait(&kv_full[g0 % SK], (g0 / SK) & 1, ctl, kSiteKvFull) &&
             mbar_wait(do_ready, it & 1, ctl, kSiteDoFull);
        if (!ok) break;
        tc_fence_after();
        issue_s(g0);
        {
          const uint64_t bv = v_kmaj(g0);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) dp_step(bv, kk);
        }
        tc_commit(dp_full);
        tc_commit(&v_empty[g0 % SV]);
        for (int j = 0; ok && j < n_kv; ++j) {
          const int g = g0 + j;
          const bool more = j + 1 < n_kv;
          if (more) {
            // S(j+1) once the rows have read S(j)
            if (!(ok = mbar_wait(&kv_full[(g + 1) % SK], ((g + 1) / SK) & 1, ctl, kSiteKvFull))) break;
            if (!(ok = mbar_wait(s_free, g & 1, ctl, kSiteSFull))) break;
            tc_fence_after();
            issue_s(g + 1);
          }
          // dQ += dS K_j (dS from TMEM over the dP columns; K_j MN-major over
          // d) once the rows have written dS(j), then dP(j+1) over it
          if (!(ok = mbar_wait(ds_ready, g & 1, ctl, kSiteDsReady))) break;
          tc_fence_after();
          {
            const uint64_t bk = k_mn(g);
#pragma unroll
            for (int kk = 0; kk < kBlk / 16; ++kk)  // dS of keys [64h, 64h+64) sits at columns 128 + 64h..
              mma_ts(tDQ, tDP + (kk >> 2) * 64 + (kk & 3) * 8, desc_add(bk, mnmajor_step(kk)), kIdescQ,
                     (j > 0 || kk > 0));
          }
          tc_commit(&k_empty[g % SK]);
          if (more) {
            const uint64_t bv = v_kmaj(g + 1);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) dp_step(bv, kk);
            tc_commit(dp_full);
            tc_commit(&v_empty[(g + 1) % SV]);
          }
        }
        // the item's dQ is complete, and its Q, dO columns are free
        if (ok) tc_commit(dq_done);
      }
      tc_commit(drain);
      mbar_drain(drain, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ query rows
    const int half = (warp >> 2) - 1;  // key columns [64 half, 64 half + 64)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // query row within the block
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + kColS + lane_base, tDP = tmem + kColDP + lane_base;
    const float c = p.scale_log2;
    const int c0 = half * 64;  // first key column of this half
    bool ok = true;

    for (int it = 0, g0 = 0; ok && it < n_items; g0 += item_nkv(it), ++it) {
      const int iblk = item_i(it), n_kv = item_nkv(it);
      const int qrow = iblk * kBlk + r;
      const size_t srow = static_cast<size_t>(bh) * nblk * kBlk + qrow;
      const float lse2 = p.lse2[srow];  // +inf on padding rows: P = 0
      const float dlt = p.delta[srow];
      const float2 cc = make_float2(c, c), nl = make_float2(-lse2, -lse2), nd = make_float2(-dlt, -dlt);

      // Q and dO rows -> TMEM (bf16 pairs over D/2 columns each): the A
      // operands of S and dP.  The two halves share the 64-element pieces.
      // (A second item overwrites the first's once its products are complete:
      // these rows have waited for dq_done and stored its dQ.)
      {
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const uint4 *src = reinterpret_cast<const uint4 *>(m ? p.dout + row_offset(p.sdo, bh, p.H, row0 + qrow)
                                                               : p.q + row_offset(p.sq, bh, p.H, row0 + qrow));
          const uint32_t col = m ? kColDO : kColQ;
#pragma unroll
          for (int hh = 0; hh < D / 64; ++hh) {
            if (((hh + m) & 1) != half) continue;
            uint32_t v[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const uint4 x = qrow < N ? src[hh * 8 + u] : make_uint4(0, 0, 0, 0);
              v[4 * u] = x.x;
              v[4 * u + 1] = x.y;
              v[4 * u + 2] = x.z;
              v[4 * u + 3] = x.w;
            }
            tmem_st32(tmem + col + lane_base + hh * 32, v);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(do_ready);
      }

      for (int j = 0; j < n_kv; ++j) {
        const int gb = g0 + j;  // key-block counter over both items
        const bool diag = CAUSAL && (j == iblk);
        // packed mode: keys past the sequence are the next sequence's rows and
        // must get P = 0 (batched mode: they are zero rows of K and V, whose
        // dS K adds nothing)
        const int klim = N - 1 - j * kBlk;  // last key column of this block inside the sequence
        const bool kmask = VARLEN && klim < kBlk - 1;
        // Phase 1: P = exp2(S c - lse2) for this half of the keys, kept as bf16 pairs.
        ok = mbar_wait(s_full, gb & 1, ctl, kSiteSFull);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float2 pf[32];  // P of this half row (fp32 pairs), kept for phase 2
        uint32_t sva[2][32];
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) tmem_ld32(tS + c0 + ch * 32, sva[ch]);
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) tmem_ld_wait(sva[ch]);
        tc_fence_before();
        warp_arrive(s_free);  // S is in registers: the next S may overwrite it
        // (two copies, the mask flag fixed at compile time: the blocks that
        // need no mask carry no masking instructions; with one body and a
        // run-time test the causal kernel ran its ALU pipe at twice the
        // non-causal one's rate)
        auto form_p = [&](auto mask_tag) {
          const bool masked = mask_tag;
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            const uint32_t(&sv)[32] = sva[ch];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 x = ffma2(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), cc, nl);
              float p0 = ex2(x.x), p1 = ex2(x.y);
              if (masked) {  // key kc visible to query r iff kc <= r (causal) and kc < N
                const int lim = diag ? min(r, klim) : klim;
                p0 = (c0 + ch * 32 + e <= lim) ? p0 : 0.0f;
                p1 = (c0 + ch * 32 + e + 1 <= lim) ? p1 : 0.0f;
              }
              pf[ch * 16 + e / 2] = make_float2(p0, p1);
            }
          }
        };
        if (diag || kmask)
          form_p(MaskTag<true>{});
        else
          form_p(MaskTag<false>{});

        // Phase 2: dS = P o (dP - D) -> bf16 pairs over this half's own,
        // already read, dP columns (dQ(j-1) has read dS(j-1) from there: it
        // ran before dP(j)).
        ok = mbar_wait(dp_full, gb & 1, ctl, kSiteSFull);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t dpa[2][32];
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) tmem_ld32(tDP + c0 + ch * 32, dpa[ch]);
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) tmem_ld_wait(dpa[ch]);
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const uint32_t(&dpv)[32] = dpa[ch];
          uint32_t dsv[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 g = fadd2(make_float2(__uint_as_float(dpv[e]), __uint_as_float(dpv[e + 1])), nd);
            const float2 ds = fmul2(pf[ch * 16 + e / 2], g);
            dsv[e / 2] = pack_bf16x2(ds.x, ds.y);
          }
          tmem_st16(tDP + c0 + ch * 16, dsv);
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(ds_ready);
      }
      // dQ epilogue (the scale applied here): each half writes D/2 columns
      if (ok) {
        ok = mbar_wait(dq_done, it & 1, ctl, kSiteMmaDone);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) {
        tc_fence_after();
        store_acc_row<D / 2>(tmem + kColDQ + lane_base + half * (D / 2),
                             p.dq + row_offset(p.sdq, bh, p.H, row0 + qrow) + half * (D / 2), qrow < N, p.scale);
      }
    }  // items
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <typename Kern>
cudaError_t launch_main(Kern kern, unsigned grid, int threads, uint32_t smem, const CUtensorMap &tq,
                        const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tdo, const BwdParams &p,
                        cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, threads, smem, stream>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError();
}

// A side stream and two events per host thread and device, for running the
// dQ kernel next to the dK/dV kernel (created on first use, kept until the
// process ends).
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

cudaError_t side_stream(SideStream **out) {
  constexpr int kMaxDevices = 64;
  thread_local SideStream res[kMaxDevices];
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  SideStream &r = res[dev];
  if (!r.stream) {
    if ((e = cudaEventCreateWithFlags(&r.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&r.join, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&r.stream, cudaStreamNonBlocking)) != cudaSuccess) return e;
  }
  *out = &r;
  return cudaSuccess;
}

template <int D, bool CAUSAL, bool VARLEN>
cudaError_t launch_bwd_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tdo,
                         const BwdParams &p, cudaStream_t stream, const cudaEvent_t *ev, bool concurrent) {
  using L = BwdLayout<D>;
  const long long padded_rows = static_cast<long long>(p.BH) * p.num_blk * kBlk;
  constexpr int kRowsPerBlock = 256 / (D / 8);
  const long long pre_blocks = (padded_rows + kRowsPerBlock - 1) / kRowsPerBlock;
  constexpr long long kPreGridMax = 152LL * 8 * 64;  // grid-stride beyond this
  fa_bwd_pre_kernel<D>
      <<<static_cast<unsigned>(pre_blocks < kPreGridMax ? pre_blocks : kPreGridMax), 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // one CTA per block, or (pairs) per pair of mirror blocks
  const unsigned grid_kv = static_cast<unsigned>(p.BH) *
                           static_cast<unsigned>(p.pairs_kv ? (p.num_blk + 1) / 2 : p.num_blk);
  const unsigned grid_q = static_cast<unsigned>(p.BH) *
                          static_cast<unsigned>(p.pairs_q ? (p.num_blk + 1) / 2 : p.num_blk);
  // (long non-causal heads: four row groups; causal: two, see KvRows)
  constexpr int RG = CAUSAL ? 2 : 4;
  // the schedule is a template parameter: the one-block kernels carry no
  // loop over items (measured 3-4 % faster than a run-time flag)
  const auto kern_kv = p.pairs_kv ? fa_bwd_dkdv_kernel<D, CAUSAL, VARLEN, RG, true>
                                  : fa_bwd_dkdv_kernel<D, CAUSAL, VARLEN, RG, false>;
  const auto kern_q = p.pairs_q ? fa_bwd_dq_kernel<D, CAUSAL, VARLEN, true> : fa_bwd_dq_kernel<D, CAUSAL, VARLEN, false>;
  if (concurrent && !ev) {
    // The dQ kernel reads only the inputs and the pre-kernel's statistics,
    // so it runs on a side stream next to the dK/dV kernel: each grid is
    // 13.5 waves of one CTA per SM at the bench shape, and the two
    // together leave fewer SMs idle in a last wave than one after the
    // other.  The caller's stream waits for both before anything after.
    SideStream *side = nullptr;
    if ((e = side_stream(&side)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(side->fork, stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(side->stream, side->fork, 0)) != cudaSuccess) return e;
    e = launch_main(kern_kv, grid_kv, KvRows<RG>::kThreads, L::kSmemRequest, tq,
                    tk, tv, tdo, p, stream);
    if (e != cudaSuccess) return e;
    e = launch_main(kern_q, grid_q, kThreads, DqLayout<D>::kSmemRequest, tq, tk, tv, tdo,
                    p, side->stream);
    if (e != cudaSuccess) return e;
    if ((e = cudaEventRecord(side->join, side->stream)) != cudaSuccess) return e;
    return cudaStreamWaitEvent(stream, side->join, 0);
  }
  if (ev && (e = cudaEventRecord(ev[0], stream)) != cudaSuccess) return e;
  e = launch_main(kern_kv, grid_kv, KvRows<RG>::kThreads, L::kSmemRequest, tq, tk,
                  tv, tdo, p, stream);
  if (e != cudaSuccess) return e;
  if (ev && (e = cudaEventRecord(ev[1], stream)) != cudaSuccess) return e;
  e = launch_main(kern_q, grid_q, kThreads, DqLayout<D>::kSmemRequest, tq, tk, tv, tdo,
                  p, stream);
  if (e != cudaSuccess) return e;
  if (ev && (e = cudaEventRecord(ev[2], stream)) != cudaSuccess) return e;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd(int d, bool causal, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tdo, const BwdParams &p, cudaStream_t stream, const cudaEvent_t *ev,
                       bool concurrent) {
  // (the packed-sequence mode is a template parameter: the batched kernels
  // carry none of its per-block work)
  const bool v = p.cu_seqlens != nullptr;
  if (d == 64) {
    if (causal)
      return v ? launch_bwd_t<64, true, true>(tq, tk, tv, tdo, p, stream, ev, concurrent)
               : launch_bwd_t<64, true, false>(tq, tk, tv, tdo, p, stream, ev, concurrent);
    return v ? launch_bwd_t<64, false, true>(tq, tk, tv, tdo, p, stream, ev, concurrent)
             : launch_bwd_t<64, false, false>(tq, tk, tv, tdo, p, stream, ev, concurrent);
  }
  if (causal)
    return v ? launch_bwd_t<128, true, true>(tq, tk, tv, tdo, p, stream, ev, concurrent)
             : launch_bwd_t<128, true, false>(tq, tk, tv, tdo, p, stream, ev, concurrent);
  return v ? launch_bwd_t<128, false, true>(tq, tk, tv, tdo, p, stream, ev, concurrent)
           : launch_bwd_t<128, false, false>(tq, tk, tv, tdo, p, stream, ev, concurrent);
}

}  // namespace fa
