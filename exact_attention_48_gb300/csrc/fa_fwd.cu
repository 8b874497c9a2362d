// fa_fwd.cu -- forward kernel of exact attention for sm_103a.
//
// One CTA owns 256 query rows (two tiles of 128) of one (batch, head) and
// walks the key/value blocks of that head (lexicon page "FlashAttention"
// (urworte.de), section "Methodische Grundlagen": block-wise processing in
// on-chip memory, the score / normalisation / weighting steps fused in one
// pass, and a running row normalisation that corrects the partial output
// whenever a larger score appears).  The grid spreads the query blocks of
// every head over the SMs (page "FlashAttention-2 (DE)", "Technische
// Architektur", section 2).  Short batched sequences run a persistent grid
// instead: one CTA per SM takes such 256-row tiles in turn and overlaps each
// tile's start with the previous tile's end.
//
// Roles inside the CTA (384 threads, three warpgroups):
//   warps 0..3   softmax of tile 0, warps 4..7 softmax of tile 1: one query
//                row per thread, running max m and sum l in registers, P
//                written back as bf16 over S in TMEM (it is the A operand of
//                the P V product), O rescaled in TMEM when m grows, final
//                O / l and the logsumexp.
//   warp 8       TMA producer: both Q tiles once, then K_j and V_j into a
//                ring of stages
//   warp 9       MMA issuer (one thread): S_t = Q_t K_j^T into TMEM and
//                O_t += P_t V_j for both tiles t, interleaved so that the
//                tensor core works on one tile while the other is
//                normalised; the warp also owns the TMEM allocation.
//   warps 10, 11 idle (they complete the third warpgroup).
//
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256, 256+w),
// O_1 [256+w, 256+2w) with w = d, except at d = 64 where w = 80: there the
// P V product also multiplies P by a slab of ones placed after V in shared
// memory, and O's columns 64..79 receive the sum of the bf16 weights it
// applied (the divisor of O), which the softmax warps then need not add up
// element by element.  Only scores and probabilities of the current block
// ever exist, and only on chip (page "FlashAttention-2 (DE)", "Hintergrund").
//
// Scores are kept in the log2 domain: t = s * scale * log2(e).  The running
// max is only moved when a row's new block max exceeds it by more than 8
// (a factor 256 in P), so most blocks skip the O rescale; the result is the
// same because l and O always share the max they were computed with.

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kBM = 128;  // query rows per tile (two tiles per CTA)
constexpr int kBN = 128;  // keys per block
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr uint32_t kTmemCols = 512;

// QB: buffers of the two Q tiles (2 in the persistent d = 64 kernel, which
// loads the next 256 rows' Q while it still works on the current ones; at
// d = 128 a second 64 KB buffer does not fit beside the K/V ring).
template <int D, int QB>
struct FwdLayout {
  static constexpr int kSlabs = D / 64;  // 128-byte column slabs of a bf16 row
  // K/V ring stages (three beside the persistent kernel's second Q buffer:
  // measured as fast as four there)
  static constexpr int kStages = (D == 64) ? (QB == 2 ? 3 : 4) : 2;
  static constexpr int kQBufs = QB;
  static constexpr uint32_t kQTile = kBM * D * 2;
  static constexpr uint32_t kKVBytes = kBN * D * 2;
  static constexpr uint32_t kOffQ = 0;  // QB buffers of two tiles
  static constexpr uint32_t kOffK = kOffQ + QB * 2 * kQTile;
  static constexpr uint32_t kOffV = kOffK + kStages * kKVBytes;
  // d = 64: one 128-key slab of bf16 ones, the extra 16 columns of V in P V
  static constexpr uint32_t kOnesBytes = (D == 64) ? kBN * 128 : 0;
  static constexpr uint32_t kOffOnes = kOffV + kStages * kKVBytes;
  static constexpr uint32_t kOffBar = kOffOnes + kOnesBytes;
  // q_full[QB], q_empty[QB], k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2], p_ready[2],
  // pv_done[2], drain
  static constexpr int kNumBars = 2 * QB + 4 * kStages + 6 + 1;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kBytes = kOffMisc + 16;
  static constexpr uint32_t kSmemRequest = kBytes + 1024;  // slack for 1024-byte alignment
  static_assert(kSmemRequest <= 232448, "shared memory budget");
};

constexpr int kThreads = 384;
constexpr int kWarpProducer = 8, kWarpMma = 9;
// Register split: 168 per thread at launch (384 x 168 fits the SM); the
// control warpgroup gives registers back and the two softmax warpgroups take
// them: at d = 128 104 and 200, at d = 64 152 and 176 (the MMA issuer's
// unrolled d = 64 loops spill at 104; without the spills the d = 64 kernels
// run 4 % faster, while the d = 128 ones are 1-2 % faster with the softmax
// at 200).  The persistent d = 64 kernel carries its tile loop's state
// through the softmax and gives it 184 (136 for control): 2-3 % faster than
// 152 and 176, where its softmax spilled.  128*control + 256*softmax <=
// 384*168, and per SM sub-partition (one warp of each warpgroup)
// 32*(control + 2*softmax) <= 16384.
constexpr uint32_t kRegsLaunch = 168;
template <int D, bool PERSIST>
constexpr uint32_t kRegsControl = (D == 64) ? (PERSIST ? 136 : 152) : 104;
template <int D, bool PERSIST>
constexpr uint32_t kRegsSoftmax = (D == 64) ? (PERSIST ? 184 : 176) : 200;
template <int D, bool PERSIST>
constexpr bool kRegSplitFits = 128 * kRegsControl<D, PERSIST> + 256 * kRegsSoftmax<D, PERSIST> <= kThreads * kRegsLaunch &&
                               32 * (kRegsControl<D, PERSIST> + 2 * kRegsSoftmax<D, PERSIST>) <= 16384;
static_assert(kRegSplitFits<64, false> && kRegSplitFits<64, true> && kRegSplitFits<128, false> &&
                  kRegSplitFits<128, true>,
              "register split");

// Buffers of a CTA's two Q tiles (see FwdLayout).
template <int D, bool PERSIST>
constexpr int kQBufs = (PERSIST && D == 64) ? 2 : 1;

// Columns of O in TMEM: d, plus 16 at d = 64 where the product also forms
// the sum of the weights it applied.
template <int D>
constexpr int kOW = (D == 64) ? D + 16 : D;

struct SoftmaxArgs {
  uint64_t *s_full, *p_ready, *pv_done;
  uint32_t tS, tO;  // TMEM columns of this tile's S and O (lane base added inside)
  int n_kv;         // key blocks this tile visits
  int diag;         // causal: index of the diagonal key block, else -1
  int grow0;        // first query row of the tile (within its sequence)
  int N;            // rows of this tile's sequence
  int row0;         // first row of the sequence on the tensors' row axis
  int cb0;          // blocks this tile's barriers completed for earlier tiles (their phase base)
};

// Online softmax of one 128-row tile: one query row per thread.  Returns
// false if a wait gave up.
template <int D, bool CAUSAL, bool VARLEN>
__device__ __forceinline__ bool softmax_tile(const SoftmaxArgs &a, const FwdParams &p, const WaitCtl &ctl, int bh,
                                             int warp, int lane) {
  const int wq = warp & 3;
  const int row = wq * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  // batched: the length from the kernel parameters (a constant operand;
  // measurably faster in this loop than a register copy)
  const int N = VARLEN ? a.N : p.N;
  const float c = p.scale_log2;
  const bool neg = p.neg != 0;
  const uint32_t tS = a.tS + lane_base, tO = a.tO + lane_base;
  float m_run = -INFINITY, l_run = 0.0f, lb_run = 0.0f;
  bool ok = true;

  // One key block.  `mask` (a run-time flag, or a compile-time one) says
  // whether the block needs the causal or ragged-end mask, which only a
  // tile's last block can.  With the flag known at compile time, two copies
  // of the body keep the masking instructions out of every other block.
  // Measured: the causal kernels with one body and a run-time test ran
  // their ALU pipe at 41 % against 23 % without a mask, and the two copies
  // made them 8-18 % faster (and the d = 64 kernels 5 %); only the
  // batched non-causal d = 128 kernel was 2 % faster with the one body.
  auto block = [&](const int j, auto mask) -> bool {
    const bool MASK = mask;
    if (!__all_sync(0xffffffffu, mbar_wait(a.s_full, (a.cb0 + j) & 1, ctl, kSiteSFull))) return false;
    tc_fence_after();
    uint32_t s[4][32];
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) tmem_ld32(tS + q4 * 32, s[q4]);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) tmem_ld_wait(s[q4]);

    // Masking: causal diagonal block and the ragged last key block.
    int lim = kBN - 1;  // last visible column of this row
    if (MASK) {
      lim = min(lim, N - 1 - j * kBN);
      if (j == a.diag) lim = min(lim, row);
      const uint32_t hide = __float_as_uint(neg ? INFINITY : -INFINITY);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (q4 * 32 + i > lim) s[q4][i] = hide;
    }

    // Block max of t = s * c (a min of s when the scale is negative).
    // (one partial per 32-column quarter keeps the dependency chains short)
    float mx;
    if (!neg) {
      float mq[4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float m0 = fmax3(__uint_as_float(s[q4][0]), __uint_as_float(s[q4][1]), __uint_as_float(s[q4][2]));
#pragma unroll
        for (int i = 3; i < 31; i += 2) m0 = fmax3(m0, __uint_as_float(s[q4][i]), __uint_as_float(s[q4][i + 1]));
        mq[q4] = fmaxf(m0, __uint_as_float(s[q4][31]));
      }
      mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
    } else {
      float mq[4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float m0 = fmin3(__uint_as_float(s[q4][0]), __uint_as_float(s[q4][1]), __uint_as_float(s[q4][2]));
#pragma unroll
        for (int i = 3; i < 31; i += 2) m0 = fmin3(m0, __uint_as_float(s[q4][i]), __uint_as_float(s[q4][i + 1]));
        mq[q4] = fminf(m0, __uint_as_float(s[q4][31]));
      }
      mx = fminf(fminf(mq[0], mq[1]), fminf(mq[2], mq[3]));
    }
    const float m_cand = mx * c;
    const bool grow = m_cand > m_run + kRescaleThreshold;
    float alpha = 1.0f;
    if (grow) {
      alpha = ex2(m_run - m_cand);
      m_run = m_cand;
    }
    const float2 cc = make_float2(c, c), nm = make_float2(-m_run, -m_run);

    // P = exp2(t - m) as bf16 pairs over the first 64 columns of S (the A
    // operand of the P V product), one quarter (32 keys -> 16 columns) at a
    // time.  The sum of the fp32 P (for the logsumexp) is taken on the way;
    // the sum of the bf16 P (for O) waits until the MMA warp has been
    // released (below), off the path that the tensor core waits on.
    uint32_t pk[4][16];
    float2 sf = make_float2(0.f, 0.f);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      float2 sfq = make_float2(0.f, 0.f);  // per-quarter partial sum
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float2 x = ffma2(make_float2(__uint_as_float(s[q4][i]), __uint_as_float(s[q4][i + 1])), cc, nm);
        float p0 = ex2(x.x), p1 = ex2(x.y);
        if (MASK) {
          p0 = (q4 * 32 + i <= lim) ? p0 : 0.0f;
          p1 = (q4 * 32 + i + 1 <= lim) ? p1 : 0.0f;
        }
        pk[q4][i / 2] = pack_bf16x2(p0, p1);
        sfq = fadd2(sfq, make_float2(p0, p1));
      }
      tmem_st16(tS + q4 * 16, pk[q4]);
      sf = fadd2(sf, sfq);
    }
    tmem_st_wait();

    // A row whose max moved rescales O, which needs the previous product
    // complete (it is: S of this block was issued after it, and S is
    // complete; the wait only makes that explicit).  Rows that keep their
    // max leave O alone, and the next product simply accumulates into it.
    if (j > 0 && __any_sync(0xffffffffu, grow)) {
      if (!__all_sync(0xffffffffu, mbar_wait(a.pv_done, (a.cb0 + j - 1) & 1, ctl, kSitePvDone))) return false;
      {
        tc_fence_after();
#pragma unroll 1
        for (int ch = 0; ch < kOW<D> / 16; ++ch) {  // 16 columns at a time: P stays in registers meanwhile
          uint32_t o[16];
          tmem_ld16(tO + ch * 16, o);
          tmem_ld_wait16(o);
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st16(tO + ch * 16, o);
        }
        tmem_st_wait();
      }
    }
    tc_fence_before();
    warp_arrive(a.p_ready);

    // Sum of the bf16 P the P V product used: O is divided by it, so that
    // the weights applied to V add up to one.  (At d = 64 the product forms
    // it itself, in O's extra columns.)
    l_run = l_run * alpha + (sf.x + sf.y);
    if constexpr (D != 64) {
      float2 sb = make_float2(0.f, 0.f);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float2 sbq = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 16; ++i) sbq = add_bf16x2_f32(sbq, pk[q4][i]);
        sb = fadd2(sb, sbq);
      }
      lb_run = lb_run * alpha + (sb.x + sb.y);
    }
    return true;
  };
  constexpr bool kTwoBodies = !(D == 128 && !CAUSAL && !VARLEN);
  for (int j = 0; j < a.n_kv; ++j) {
    const bool need_mask = (j == a.diag) || ((j + 1) * kBN > N);
    bool cont;
    if constexpr (kTwoBodies)
      cont = need_mask ? block(j, MaskTag<true>{}) : block(j, MaskTag<false>{});
    else
      cont = block(j, need_mask);
    if (!cont) {
      ok = false;
      break;
    }
  }

  // Epilogue: O / l in bf16 and the natural-log logsumexp.
  if (ok) {
    ok = mbar_wait(a.pv_done, (a.cb0 + a.n_kv - 1) & 1, ctl, kSitePvDone);
    ok = __all_sync(0xffffffffu, ok);
  }
  if (ok) {
    tc_fence_after();
    float lb = lb_run;
    if constexpr (D == 64) {
      uint32_t r16[16];
      tmem_ld16(tO + D, r16);
      tmem_ld_wait16(r16);
      lb = __uint_as_float(r16[0]);
    }
    const float inv_l = 1.0f / lb;
    const int grow_row = a.grow0 + row;
    const bool store = grow_row < N;
    __nv_bfloat16 *orow = p.o + row_offset(p.so, bh, p.H, a.row0 + grow_row);
#pragma unroll 1
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t o[32];
      tmem_ld32(tO + ch * 32, o);
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
    if (store)
      p.lse[(bh / p.H) * p.lse_b + (bh % p.H) * p.lse_h + a.row0 + grow_row] = (m_run + log2f(l_run)) * kLn2;
  }
  return ok;
}

// One 256-row block of query rows of one (batch, head): what a CTA works on.
struct FwdTile {
  int bh, qb;      // (batch, head) index and 256-row block
  int row0, N;     // the sequence's first row on the row axis, its length
  int bh_h, bh_b;  // TMA coordinates of the head
  int n0, n1;      // key blocks of its tiles 0 and 1 (n0 <= n1)
  bool empty;      // packed mode: the block lies past its sequence's end
};

// Tile order.  Causal: the heaviest 256-row blocks (most key blocks) first,
// across all heads.  Otherwise head-major so that CTAs running together
// share the K/V of one head in L2.
template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ FwdTile fwd_tile(const FwdParams &p, int x) {
  FwdTile t;
  if (CAUSAL) {
    t.qb = p.num_qblk - 1 - x / p.BH;
    t.bh = x % p.BH;
  } else {
    t.bh = x / p.num_qblk;
    t.qb = x % p.num_qblk;
  }
  const SeqRange seq = VARLEN ? seq_range(p.cu_seqlens, t.bh / p.H, p.N, p.T) : SeqRange{0, p.N};
  t.empty = VARLEN && t.qb * 2 * kBM >= seq.len;
  t.row0 = seq.start;
  t.N = seq.len;
  t.bh_h = t.bh % p.H;
  t.bh_b = VARLEN ? 0 : t.bh / p.H;
  const int nkv_all = (t.N + kBN - 1) / kBN;
  t.n0 = CAUSAL ? min(2 * t.qb + 1, nkv_all) : nkv_all;
  t.n1 = CAUSAL ? min(2 * t.qb + 2, nkv_all) : nkv_all;
  return t;
}

// PERSIST: one CTA per SM walks the tiles (its turn r = 0, 1, ... takes
// tile r * gridDim.x + blockIdx.x, mirrored in odd turns when causal);
// otherwise one CTA per tile.  At d = 64 the persistent kernel keeps two Q
// buffers, so the next tile's Q arrives while the current tile is worked
// on, and its first scores are formed while the softmax warps still write
// the current tile's output: the load latency, pipeline fill and epilogue
// that a CTA of its own pays per tile overlap the neighbouring tiles' work.
// At d = 128 (one Q buffer) the next tile's Q loads once the current tile's
// last scores are complete, while its last P V products and its epilogue
// run.  The K/V ring and every barrier's phase run on across tiles.
template <int D, bool CAUSAL, bool VARLEN, bool PERSIST>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  static_assert(!(PERSIST && VARLEN), "the packed mode launches one CTA per tile");
  constexpr int QB = kQBufs<D, PERSIST>;
  using L = FwdLayout<D, QB>;
  constexpr int S = L::kStages;
  // tiles a CTA takes at most (the persistent loop ends on the tile count)
  constexpr int kTurns = PERSIST ? 0x7fffffff : 1;
  const int num_tiles = p.BH * p.num_qblk;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
  uint64_t *q_full = bars;          // [QB]
  uint64_t *q_empty = q_full + QB;  // [QB]
  uint64_t *k_full = q_empty + QB;
  uint64_t *k_empty = k_full + S;
  uint64_t *v_full = k_empty + S;
  uint64_t *v_empty = v_full + S;
  uint64_t *s_full = v_empty + S;   // [2 tiles]
  uint64_t *p_ready = s_full + 2;   // [2 tiles]
  uint64_t *pv_done = p_ready + 2;  // [2 tiles]
  uint64_t *drain = pv_done + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 4);
  const WaitCtl ctl{abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // A CTA of its own takes its tile here (and has no work if the tile lies
  // past its sequence's end, packed mode); persistent CTAs take theirs in
  // each role's tile loop.
  FwdTile own{};
  if constexpr (!PERSIST) {
    own = fwd_tile<CAUSAL, VARLEN>(p, static_cast<int>(blockIdx.x));
    if (own.empty) return;
  }
  // Persistent CTAs take tile r * G + c in turn r (G CTAs, c = blockIdx);
  // causal tiles come heaviest first, and odd turns run c backwards so that
  // each CTA's heavy and light tiles even out.
  auto tile_index = [&](int r) -> int {
    const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    return r * G + ((CAUSAL && (r & 1)) ? G - 1 - c : c);
  };
  auto tile_at = [&](int x) -> FwdTile {
    if constexpr (PERSIST)
      return fwd_tile<CAUSAL, VARLEN>(p, x);
    else
      return own;
  };

  if (threadIdx.x == 0) {
    for (int b = 0; b < QB; ++b) {
      mbar_init(&q_full[b], 1);
      mbar_init(&q_empty[b], 1);
    }
    for (int s = 0; s < S; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_ready[t], 4);  // one arrival per softmax warp of the tile
      mbar_init(&pv_done[t], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if constexpr (D == 64) {  // the ones slab (every bf16 1.0, so its swizzle does not matter)
    uint4 *ones = reinterpret_cast<uint4 *>(smem + L::kOffOnes);
    for (int i = static_cast<int>(threadIdx.x); i < static_cast<int>(L::kOnesBytes / 16); i += kThreads)
      ones[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    fence_proxy_async_smem();
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
    regs_decrease<kRegsControl<D, PERSIST>>();
    if (warp == kWarpProducer && lane == 0) {
      // ---------------------------------------------------------- producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int g = 0;  // K/V blocks loaded so far, over all tiles (ring position)
      int q_issued = 0, k_issued = 0, v_issued = 0;
      bool run = true;
      for (int r = 0; run && r < kTurns; ++r) {
        const int x = tile_index(r);
        if (PERSIST && x >= num_tiles) break;
        const FwdTile tl = tile_at(x);
        const int qbuf = r % QB;
        if (!mbar_wait(&q_empty[qbuf], ((r / QB) & 1) ^ 1, ctl, kSiteQEmpty)) break;
        mbar_arrive_expect_tx(&q_full[qbuf], 2 * L::kQTile);
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int s = 0; s < L::kSlabs; ++s)
            tma_load_4d(sQ + (qbuf * 2 + t) * L::kQTile + s * kBM * 128, &tm_q, &q_full[qbuf], s * 64,
                        tl.row0 + tl.qb * 2 * kBM + t * kBM, tl.bh_h, tl.bh_b);
        q_issued = r + 1;
        for (int j = 0; j < tl.n1; ++j, ++g) {
          const int st = g % S;
          const uint32_t ph = (g / S) & 1;
          if (!mbar_wait(&k_empty[st], ph ^ 1, ctl, kSiteKEmpty)) {
            run = false;
            break;
          }
          mbar_arrive_expect_tx(&k_full[st], L::kKVBytes);
#pragma unroll
          for (int s = 0; s < L::kSlabs; ++s)
            tma_load_4d(sK + st * L::kKVBytes + s * kBN * 128, &tm_k, &k_full[st], s * 64, tl.row0 + j * kBN,
                        tl.bh_h, tl.bh_b);
          k_issued = g + 1;
#ifdef FA_TEST_SKIP_FIRST_V_LOAD
          // Test builds only: the first V block is never loaded, so the MMA
          // thread's wait for it runs out and the bounded-wait path is taken.
          if (g == 0) continue;
#endif
          if (!mbar_wait(&v_empty[st], ph ^ 1, ctl, kSiteVEmpty)) {
            run = false;
            break;
          }
          mbar_arrive_expect_tx(&v_full[st], L::kKVBytes);
#pragma unroll
          for (int s = 0; s < L::kSlabs; ++s)
            tma_load_4d(sV + st * L::kKVBytes + s * kBN * 128, &tm_v, &v_full[st], s * 64, tl.row0 + j * kBN,
                        tl.bh_h, tl.bh_b);
          v_issued = g + 1;
        }
      }
      // Every copy issued lands before this thread leaves, whatever the
      // other roles do: after a timeout elsewhere in the CTA nobody else
      // waits for them.  (Bounded waits; in a normal run they are done.)
      for (int i = (q_issued > QB ? q_issued - QB : 0); i < q_issued; ++i) mbar_drain(&q_full[i % QB], (i / QB) & 1);
      for (int i = (k_issued > S ? k_issued - S : 0); i < k_issued; ++i) mbar_drain(&k_full[i % S], (i / S) & 1);
      for (int i = (v_issued > S ? v_issued - S : 0); i < v_issued; ++i) mbar_drain(&v_full[i % S], (i / S) & 1);
    } else if (warp == kWarpMma && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t kIdescS = idesc_bf16(kBM, kBN, false, false);
      constexpr uint32_t kIdescO = idesc_bf16(kBM, kOW<D>, false, true);
      const uint32_t aQ = smem_addr(sQ), aK = smem_addr(sK), aV = smem_addr(sV);
      // TMEM columns of tile t: S at t*128, O at 256 + t*kOW<D>
      int g = 0;           // ring position of the current tile's first K/V block
      int c0 = 0, c1 = 0;  // blocks tiles 0 and 1 finished in earlier tiles (barrier phases)
      bool ok = true;
      for (int r = 0; ok && r < kTurns; ++r) {
        const int x = tile_index(r);
        if (PERSIST && x >= num_tiles) break;
        const FwdTile tl = tile_at(x);
        const int n0 = tl.n0, n_kv = tl.n1;
        const int qbuf = r % QB;

        // Descriptors: the Q tiles once, K/V per stage; every MMA adds a
        // compile-time step offset (the issue loops are unrolled).
        const uint64_t dQ0 = sdesc_sw128(aQ + qbuf * 2 * L::kQTile, 16, 1024),
                       dQ1 = sdesc_sw128(aQ + (qbuf * 2 + 1) * L::kQTile, 16, 1024);

        // S_t = Q_t K_j^T (both operands K-major over d)
        auto issue_s = [&](int t, int j) {
          const uint64_t bq = t ? dQ1 : dQ0, bk = sdesc_sw128(aK + ((g + j) % S) * L::kKVBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + t * 128, desc_add(bq, kmajor_step(kk, kBM)), desc_add(bk, kmajor_step(kk, kBN)), kIdescS,
                   kk > 0 ? 1u : 0u);
          tc_commit(&s_full[t]);
        };
        // O_t += P_t V_j; P_t sits (bf16, two per column) over S_t in TMEM
        // and V_j is [key][d]: MN-major for this product (d contiguous); 16
        // keys = two 8-row groups of 1024 bytes, d slabs 128*128 bytes apart.
        // The tile's first product overwrites O: the softmax warps have
        // read the previous tile's O before they release this P.
        auto issue_pv = [&](int t, int j) -> bool {
          if (!mbar_wait(&p_ready[t], ((t ? c1 : c0) + j) & 1, ctl, kSitePReady)) return false;
          tc_fence_after();
          const uint32_t aVj = aV + ((g + j) % S) * L::kKVBytes;
          // (d = 64: the slab after V's one column slab is the ones slab)
          const uint64_t bv = sdesc_sw128(aVj, D == 64 ? smem_addr(smem + L::kOffOnes) - aVj : kBN * 128, 1024);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts(tmem + 256 + t * kOW<D>, tmem + t * 128 + kk * 8, desc_add(bv, mnmajor_step(kk)), kIdescO,
                   (j > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&pv_done[t]);
          return true;
        };
        auto kv_wait = [&](uint64_t *full, int j, int site) {
          return mbar_wait(&full[(g + j) % S], ((g + j) / S) & 1, ctl, site);
        };

        ok = mbar_wait(&q_full[qbuf], (r / QB) & 1, ctl, kSiteQFull) && kv_wait(k_full, 0, kSiteKFull);
        if (ok) {
          tc_fence_after();
          issue_s(0, 0);
          issue_s(1, 0);
          tc_commit(&k_empty[g % S]);
        }
        for (int j = 1; ok && j < n_kv; ++j) {
          const int pj = j - 1;
          if (!(ok = kv_wait(v_full, pj, kSiteVFull))) break;
          tc_fence_after();
          if (pj < n0 && !(ok = issue_pv(0, pj))) break;
          if (!(ok = kv_wait(k_full, j, kSiteKFull))) break;
          tc_fence_after();
          if (j < n0) issue_s(0, j);
          if (!(ok = issue_pv(1, pj))) break;
          tc_commit(&v_empty[(g + pj) % S]);
          issue_s(1, j);
          tc_commit(&k_empty[(g + j) % S]);
        }
        if (ok) {
          tc_commit(&q_empty[qbuf]);  // every product that reads this Q buffer is issued
          const int pj = n_kv - 1;
          ok = kv_wait(v_full, pj, kSiteVFull);
          if (ok) {
            tc_fence_after();
            if (pj < n0) ok = issue_pv(0, pj);
            if (ok) ok = issue_pv(1, pj);
            tc_commit(&v_empty[(g + pj) % S]);
          }
        }
        g += n_kv;
        c0 += n0;
        c1 += n_kv;
      }
      tc_commit(drain);
      mbar_drain(drain, 0);
    }
  } else {
    regs_increase<kRegsSoftmax<D, PERSIST>>();
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;
    int cb = 0;  // blocks this tile's barriers completed in earlier tiles
    for (int r = 0; r < kTurns; ++r) {
      const int x = tile_index(r);
      if (PERSIST && x >= num_tiles) break;
      const FwdTile tl = tile_at(x);
      SoftmaxArgs a;
      a.s_full = &s_full[t];
      a.p_ready = &p_ready[t];
      a.pv_done = &pv_done[t];
      a.tS = tmem + t * 128;
      a.tO = tmem + 256 + t * kOW<D>;
      a.n_kv = t ? tl.n1 : tl.n0;
      a.diag = CAUSAL ? 2 * tl.qb + t : -1;
      a.grow0 = tl.qb * 2 * kBM + t * kBM;
      a.N = tl.N;
      a.row0 = tl.row0;
      a.cb0 = cb;
      if (!softmax_tile<D, CAUSAL, VARLEN>(a, p, ctl, tl.bh, warp, lane)) break;
      cb += a.n_kv;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool CAUSAL, bool VARLEN, bool PERSIST>
cudaError_t launch_fwd_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const FwdParams &p,
                         cudaStream_t stream) {
  using L = FwdLayout<D, kQBufs<D, PERSIST>>;
  auto kern = fa_fwd_kernel<D, CAUSAL, VARLEN, PERSIST>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemRequest);
  if (e != cudaSuccess) return e;
  const unsigned tiles = static_cast<unsigned>(p.BH) * static_cast<unsigned>(p.num_qblk);
  const unsigned ctas = static_cast<unsigned>(p.persist_ctas);
  const unsigned grid = (PERSIST && ctas < tiles) ? ctas : tiles;
  kern<<<grid, kThreads, L::kSmemRequest, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int d, bool causal, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const FwdParams &p, cudaStream_t stream) {
  // (the packed-sequence mode and the persistent grid are template
  // parameters: the other kernels carry none of their per-tile work)
  const bool v = p.cu_seqlens != nullptr, pers = p.persist_ctas > 0 && !v;
  if (d == 64) {
    if (v) return causal ? launch_fwd_t<64, true, true, false>(tq, tk, tv, p, stream)
                         : launch_fwd_t<64, false, true, false>(tq, tk, tv, p, stream);
    if (causal) return pers ? launch_fwd_t<64, true, false, true>(tq, tk, tv, p, stream)
                            : launch_fwd_t<64, true, false, false>(tq, tk, tv, p, stream);
    return pers ? launch_fwd_t<64, false, false, true>(tq, tk, tv, p, stream)
                : launch_fwd_t<64, false, false, false>(tq, tk, tv, p, stream);
  }
  if (v) return causal ? launch_fwd_t<128, true, true, false>(tq, tk, tv, p, stream)
                       : launch_fwd_t<128, false, true, false>(tq, tk, tv, p, stream);
  if (causal) return pers ? launch_fwd_t<128, true, false, true>(tq, tk, tv, p, stream)
                          : launch_fwd_t<128, true, false, false>(tq, tk, tv, p, stream);
  return pers ? launch_fwd_t<128, false, false, true>(tq, tk, tv, p, stream)
              : launch_fwd_t<128, false, false, false>(tq, tk, tv, p, stream);
}

}  // namespace fa
