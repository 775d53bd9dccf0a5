// attn_fwd.cu — fused attention forward for sm_103a: O = softmax(s Q K^T) V and
// the per-row natural-log log-sum-exp of the scaled scores.
//
// Follows the forward definition of "ops(8)：self-attention 的 CUDA 实现及优化
// (下) - 深度分析" (§2.1: S = QK^T/sqrt(d_k), P = softmax(S), O = PV; §1.3: the
// forward also returns the softmax statistics the backward needs), computed
// the way "FlashAttention Triton实现中的内存访问模式优化与寄存器分配策略"
// describes in §2.2 (the query tile stays on chip while the loop walks the
// key/value tiles, with a running row maximum and row sum) and §4.2 (the
// division by the row sum happens once, after the loop).
//
// One CTA (384 threads) per SM, persistent over work items; an item is two
// consecutive 128-row Q tiles of one (sequence, head).  The producer claims
// items from a per-call counter (head-major, longest first within a head; see
// attn_common.cuh) and hands each to the other roles through a 2-slot ring, so
// the CTAs running at any moment share a few heads' K and V in L2:
//   warps 0-3, 4-7  softmax warpgroup w owns Q tile w: thread r holds query
//                   row r (TMEM lane r)
//   warp 8          TMA producer and work claimer: the two Q tiles once per
//                   item, K and V tiles into rings of their own
//   warp 9          MMA issuer: S_w = Q_w K^T and O_w += P_w V
// Tensor memory: S_0, S_1 at columns [0,128), [128,256), O_0, O_1 after them.
// P is written back into the S columns as bf16 pairs and read from there by
// the O += P V product (A operand in tensor memory), so it never touches
// shared memory.  The two warpgroups alternate: while one computes its P, the
// tensor core runs the other tile's MMAs.  The running maximum is only moved
// (and O rescaled) when it grows by more than 2^8, so most tiles skip it.
// The kernels built for a block mask (kMask) visit only the kv tiles the mask
// keeps, in the order MaskOrder describes, with the producer publishing each
// tile's step flags to the MMA issuer.
#include <cuda_bf16.h>

#include <climits>

#include "attn_common.cuh"
#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

// Softmax warpgroups 0 and 1; warpgroup 2 holds the TMA warp (8) and the MMA
// warp (9), warps 10-11 idle.  Launched with 168 registers a thread; warpgroup 2
// drops to 128, which lets the two softmax warpgroups rise to 184
// (2 x 184 + 128 <= 3 x 168).
constexpr int kFwdThreads = 384;
constexpr uint32_t kRegsCtl = 128;
constexpr uint32_t kRegsSoftmax = 184;
static_assert(2 * kRegsSoftmax + kRegsCtl <= 3 * 168, "register split");
constexpr int kPanelBytes = kTile * 128;  // [128 rows][64] bf16

// P = 2^(S*scale*log2e - m) for the 128 scores of a row (thread = row): the
// row sum and the bf16 pairs of keys 0-63 (pk0) and 64-127 (pk1).  The
// arguments and the sum use packed FP32 pairs (two scores per instruction).
__device__ __forceinline__ float softmax_exp(const uint32_t (&sr)[4][32], float scale_log2,
                                             float m_use, uint32_t (&pk0)[32],
                                             uint32_t (&pk1)[32]) {
  const uint64_t sc2 = f2(scale_log2, scale_log2), nm2 = f2(-m_use, -m_use);
  uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};  // four independent chains of pair sums
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const uint64_t x2 = fma2(f2(__uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1])), sc2, nm2);
      const float p0 = ex2(f2_lo(x2)), p1 = ex2(f2_hi(x2));
      rs2[(e >> 1) & 3] = add2(rs2[(e >> 1) & 3], f2(p0, p1));
      if (c < 2) pk0[c * 16 + e / 2] = pack_bf16(p0, p1);
      else pk1[(c - 2) * 16 + e / 2] = pack_bf16(p0, p1);
    }
  }
  const uint64_t s4 = add2(add2(rs2[0], rs2[1]), add2(rs2[2], rs2[3]));
  return f2_lo(s4) + f2_hi(s4);
}

constexpr int kMaxSmem = 232448;

template <int DQK, int DV>
struct FwdCfg {
  static constexpr int kQPanels = DQK / 64;
  static constexpr int kVPanels = DV / 64;
  static constexpr int kQTileBytes = kQPanels * kPanelBytes;  // one 128-row Q tile
  static constexpr int kQBytes = 2 * kQTileBytes;             // the item's two Q tiles
  static constexpr int kKBytes = kQPanels * kPanelBytes;
  static constexpr int kVBytes = kVPanels * kPanelBytes;
  static constexpr int kBarBytes = 512;
  // the dynamic shared memory window starts 1024-byte aligned (checked at run time)
  static constexpr int kFixed = kQBytes + kBarBytes;
  // K and V have rings of their own: S(t) needs only a K slot, so it can be
  // issued while V of the previous tile is still being read by O += P V.
  static constexpr int kPairsFit = (kMaxSmem - kFixed) / (kKBytes + kVBytes);
  static constexpr int kKStages = kPairsFit >= 4 ? 4 : (kPairsFit >= 2 ? kPairsFit : 2);
  static constexpr int kVStagesFit = (kMaxSmem - kFixed - kKStages * kKBytes) / kVBytes;
  static constexpr int kVStages = kVStagesFit > kKStages ? kKStages : kVStagesFit;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kQBytes;
  static constexpr int kOffV = kOffK + kKStages * kKBytes;
  static constexpr int kOffBar = kOffV + kVStages * kVBytes;
  static constexpr int kSmemBytes = kOffBar + kBarBytes;
  // Tensor memory: S of Q tile w at [128w, 128w+128) (P, bf16 pairs, over its
  // first 64 columns), O of Q tile w at [256 + w*DV, 256 + (w+1)*DV).
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTmemS = 0;
  static constexpr uint32_t kTmemO = 256;
  static_assert(kVStages >= 1, "shared memory too small");
  static_assert(kKStages <= 4 && kVStages <= 4, "barrier arrays hold 4 stages");
  static_assert(kSmemBytes <= kMaxSmem, "shared memory budget");
  static_assert(kTmemO + 2 * DV <= kTmemCols, "tensor memory budget");
};

struct FwdBars {
  uint64_t item_full[2], item_empty[2];  // work items handed from the producer to the other roles
  uint64_t q_full, q_empty;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int item_slot[2];
  // block mask only, written by the producer before the matching arrive:
  int q_none;       // 1: the item loads no kv tile (with q_full)
  int kv_flags[4];  // per K stage (with k_full): kKvUse0 | kKvUse1 | kKvFirst0 | ...
};
static_assert(sizeof(FwdBars) <= 512, "barrier block size");

// kv_flags bits: which Q tiles use the stage's kv tile, whether it is a Q
// tile's first or last in the visiting order, and whether it is the item's
// last loaded kv tile.
constexpr int kKvUse0 = 1, kKvUse1 = 2, kKvFirst0 = 4, kKvLast0 = 8, kKvFirst1 = 16,
              kKvLast1 = 32, kKvItemLast = 64;

// kv-tile ranges [lo_w, hi_w] of the two Q tiles of an item (the band's tiles;
// lo0 <= lo1 and hi0 <= hi1, and the two ranges leave no gap between them).
// A Q tile that lies wholly past the sequence end can get an empty band (its
// rows see no key); it then runs its last tile anyway — its rows are never
// stored — so that every Q tile takes part in at least one step.
__device__ __forceinline__ void kv_ranges(const SeqShape& sh, const Item& it, int& lo0, int& hi0,
                                          int& lo1, int& hi1) {
  const int nk = cdiv(it.Lk, kTile);
  hi0 = last_kvtile(sh, it, 2 * it.tile, nk);
  lo0 = min(first_kvtile(sh, it, 2 * it.tile), hi0);
  hi1 = last_kvtile(sh, it, 2 * it.tile + 1, nk);
  lo1 = min(first_kvtile(sh, it, 2 * it.tile + 1), hi1);
}

// Whether Q tile w (0, 1) of the item uses kv tile j: j lies in the tile's
// band range [lo, hi] and the block mask keeps the pair.  With a block mask
// (kMask) a Q tile wholly past the sequence end uses no kv tile at all.
template <bool kMask>
__device__ __forceinline__ bool kv_used(const SeqShape& sh, const Item& it, int w, int j, int lo,
                                        int hi) {
  if (j < lo || j > hi) return false;
  if constexpr (!kMask) return true;
  const int qt = 2 * it.tile + w;
  return qt * kTile < it.Lq && tile_on(sh, it, qt, j);
}

// The order in which a block-masked item visits its kv tiles: first those
// both Q tiles keep (ascending), then alternately one that only Q tile 0
// keeps and one that only Q tile 1 keeps (each ascending).  Consecutive steps
// then belong to different Q tiles, so each softmax warpgroup overlaps the
// other tile's MMAs, as in the dense kernel; the online softmax does not
// depend on the order of the kv tiles.
struct MaskOrder {
  int phase, c0, c1, turn;  // phase 0: tiles both keep; c0 / c1: scan positions
};

// The next kv tile in MaskOrder, or hi1 + 1 when none is left; `who` gets
// the Q tiles that use it (bit 0: tile 0, bit 1: tile 1).
__device__ __forceinline__ int mask_order_next(MaskOrder& o, const SeqShape& sh, const Item& it,
                                               int lo0, int hi0, int lo1, int hi1, int& who) {
  const int end = hi1 + 1;
  if (o.phase == 0) {
    while (o.c0 < end && !(kv_used<true>(sh, it, 0, o.c0, lo0, hi0) &&
                           kv_used<true>(sh, it, 1, o.c0, lo1, hi1)))
      ++o.c0;
    who = 3;
    if (o.c0 < end) return o.c0++;
    o.phase = 1;
    o.c0 = o.c1 = lo0;
  }
  for (int k = 0; k < 2; ++k) {  // this turn's Q tile; the other once that one has no tile left
    const int w = o.turn ^ k;
    int c = w ? o.c1 : o.c0;
    while (c < end && !(kv_used<true>(sh, it, w, c, w ? lo1 : lo0, w ? hi1 : hi0) &&
                        !kv_used<true>(sh, it, w ^ 1, c, w ? lo0 : lo1, w ? hi0 : hi1)))
      ++c;
    if (w) o.c1 = c + 1; else o.c0 = c + 1;
    if (c < end) {
      o.turn = w ^ 1;
      who = 1 << w;
      return c;
    }
  }
  return end;
}

// kMask: built with block-mask support (sh.blk non-null); the kernels without
// it carry none of the mask's walks.  kLeft: the band has a left edge (a
// window's left bound, sh.wl >= 0); without one the kernel sees wl = -1 as a
// constant and its left-edge tests fold away.
template <int DQK, int DV, typename Tables, bool kMask, bool kLeft>
__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ out,
                    float* __restrict__ lse, const int64_t o_row_stride,
                    const int64_t lse_head_stride, const int64_t lse_seq_stride,
                    const float scale_log2, int* status, int* claim, const SeqShape sh_in,
                    const __grid_constant__ Tables tb) {
  using C = FwdCfg<DQK, DV>;
  SeqShape sh = sh_in;
  if constexpr (!kLeft) sh.wl = -1;
  extern __shared__ __align__(1024) uint8_t smem[];
  // Every CTA counts out on claim[1] once it will claim no more items; the
  // last one leaves both counters at zero for the next call that uses them.
  auto count_out = [&]() {
    __threadfence();  // this CTA's claims are ordered before its count-out
    if (atomicAdd(&claim[1], 1) == (int)gridDim.x - 1) {
      atomicExch(&claim[0], 0);
      atomicExch(&claim[1], 0);
    }
  };
  if (smem_u32(smem) & 1023u) {  // the swizzled panels need a 1024-byte aligned window
    if (threadIdx.x == 0) {
      atomicCAS(status, 0, kStatusInternal);
      count_out();
    }
    return;
  }
  FwdBars* bars = reinterpret_cast<FwdBars*>(smem + C::kOffBar);
  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  const uint32_t sK = smem_u32(smem + C::kOffK);
  const uint32_t sV = smem_u32(smem + C::kOffV);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  Abort ab{&bars->abort_flag, status};

  if (threadIdx.x == 0) {
    bars->abort_flag = 0;
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_u32(&bars->item_full[k]), 1);
      mbar_init(smem_u32(&bars->item_empty[k]), 1 + 8);  // MMA thread + softmax warps
    }
    mbar_init(smem_u32(&bars->q_full), 1);
    mbar_init(smem_u32(&bars->q_empty), 1);
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(smem_u32(&bars->k_full[s]), 1);
      mbar_init(smem_u32(&bars->k_empty[s]), 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(smem_u32(&bars->v_full[s]), 1);
      mbar_init(smem_u32(&bars->v_empty[s]), 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(smem_u32(&bars->s_full[w]), 1);
      mbar_init(smem_u32(&bars->p_full[w]), 4);
      mbar_init(smem_u32(&bars->o_done[w]), 1);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(&bars->tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp >= 8) {
   regs_dec<kRegsCtl>();
   if (warp == 8 && lane == 0) {
    // ------------------------------------------------------------ producer
    {
      uint32_t kv_it = 0, item_iter = 0, q_issued = 0, k_issued = 0;
      bool ok = true;
      // claim the next work item (items are taken in order by all CTAs) and
      // hand it to the MMA issuer and the softmax warps through a 2-slot ring
      auto claim_next = [&]() -> int {
        const uint32_t slot = item_iter & 1;
        if (!mbar_wait(smem_u32(&bars->item_empty[slot]), ((item_iter >> 1) & 1) ^ 1, ab)) {
          ok = false;
          return sh.n_items;
        }
        const int item = atomicAdd(claim, 1);
        bars->item_slot[slot] = item;
        mbar_arrive(smem_u32(&bars->item_full[slot]));
        return item;
      };
      for (int item = claim_next(); ok && item < sh.n_items; ++item_iter, item = claim_next()) {
        const Item it = decode_item(sh, tb, item, true);
        int lo0, hi0, lo1, hi1;
        kv_ranges(sh, it, lo0, hi0, lo1, hi1);
        // block mask: how many kv tiles each Q tile uses and how many load
        int tot0 = 0, tot1 = 0, nload = 0;
        if constexpr (kMask) {
          for (int j = lo0; j <= hi1; ++j) {
            const bool a0 = kv_used<kMask>(sh, it, 0, j, lo0, hi0);
            const bool a1 = kv_used<kMask>(sh, it, 1, j, lo1, hi1);
            tot0 += a0 ? 1 : 0;
            tot1 += a1 ? 1 : 0;
            nload += (a0 || a1) ? 1 : 0;
          }
        }
        if (!(ok = mbar_wait(smem_u32(&bars->q_empty), (item_iter & 1) ^ 1, ab))) break;
        if constexpr (kMask) bars->q_none = nload == 0 ? 1 : 0;
        const uint32_t qf = smem_u32(&bars->q_full);
        mbar_arrive_expect_tx(qf, C::kQBytes);
        q_issued = item_iter + 1;
        for (int w = 0; w < 2; ++w)
          for (int pnl = 0; pnl < C::kQPanels; ++pnl)
            tma_load_3d(sQ + w * C::kQTileBytes + pnl * kPanelBytes, &tm_q, qf, pnl * 64, it.head,
                        it.row0 + it.tile * kFwdRows + w * kTile);
        const int krow0 = key_row0(sh, it);
        // every kv tile either Q tile uses: lo0 .. hi1, or MaskOrder's tiles
        MaskOrder ord{0, lo0, lo0, 0};
        int who = 3, k0 = 0, k1 = 0, r = 0;
        for (int j = kMask ? mask_order_next(ord, sh, it, lo0, hi0, lo1, hi1, who) : lo0; j <= hi1;
             j = kMask ? mask_order_next(ord, sh, it, lo0, hi0, lo1, hi1, who) : j + 1) {
          // (never true without a mask — the band ranges leave no gap — but
          // the kernel without one issues its loads measurably faster with it)
          if (!kMask && !kv_used<kMask>(sh, it, 0, j, lo0, hi0) &&
              !kv_used<kMask>(sh, it, 1, j, lo1, hi1))
            continue;
          const uint32_t sk = kv_it % C::kKStages, sv = kv_it % C::kVStages;
          if (!(ok = mbar_wait(smem_u32(&bars->k_empty[sk]), ((kv_it / C::kKStages) & 1) ^ 1, ab)))
            break;
          if constexpr (kMask) {  // the MMA issuer's step flags for this kv tile
            int f = who;
            if ((who & 1) && k0 == 0) f |= kKvFirst0;
            if ((who & 1) && k0 + 1 == tot0) f |= kKvLast0;
            if ((who & 2) && k1 == 0) f |= kKvFirst1;
            if ((who & 2) && k1 + 1 == tot1) f |= kKvLast1;
            if (r + 1 == nload) f |= kKvItemLast;
            k0 += who & 1;
            k1 += (who >> 1) & 1;
            ++r;
            bars->kv_flags[sk] = f;
          }
          const uint32_t kf = smem_u32(&bars->k_full[sk]);
          mbar_arrive_expect_tx(kf, C::kKBytes);
          for (int pnl = 0; pnl < C::kQPanels; ++pnl)
            tma_load_3d(sK + sk * C::kKBytes + pnl * kPanelBytes, &tm_k, kf, pnl * 64, it.head,
                        krow0 + j * kTile);
          k_issued = kv_it + 1;
          if (!(ok = mbar_wait(smem_u32(&bars->v_empty[sv]), ((kv_it / C::kVStages) & 1) ^ 1, ab)))
            break;
          const uint32_t vf = smem_u32(&bars->v_full[sv]);
          mbar_arrive_expect_tx(vf, C::kVBytes);
          for (int pnl = 0; pnl < C::kVPanels; ++pnl)
            tma_load_3d(sV + sv * C::kVBytes + pnl * kPanelBytes, &tm_v, vf, pnl * 64, it.head,
                        krow0 + j * kTile);
          ++kv_it;
        }
      }
      count_out();
      if (!ok) {
        // let every copy already issued land before the CTA's memory is released
        for (uint32_t t = k_issued > (uint32_t)C::kKStages ? k_issued - C::kKStages : 0;
             t < k_issued; ++t)
          mbar_wait_drain(smem_u32(&bars->k_full[t % C::kKStages]), (t / C::kKStages) & 1);
        for (uint32_t t = kv_it > (uint32_t)C::kVStages ? kv_it - C::kVStages : 0; t < kv_it; ++t)
          mbar_wait_drain(smem_u32(&bars->v_full[t % C::kVStages]), (t / C::kVStages) & 1);
        if (q_issued > 0) mbar_wait_drain(smem_u32(&bars->q_full), (q_issued - 1) & 1);
      }
    }
   } else if (warp == 9 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    // Order per kv tile j:  PV_0(j), S_0(j+1), PV_1(j), S_1(j+1) — while one
    // softmax warpgroup works on its S, the tensor core runs the other's MMAs.
    {
      constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idO = idesc_bf16(128, DV, false, true);
      uint32_t kv_it = 0, item_iter = 0, cnt0 = 0, cnt1 = 0;
      bool ok = true;
      const uint64_t bQ0 = kmajor_base(sQ), bQ1 = kmajor_base(sQ + C::kQTileBytes);
      auto W = [&](uint64_t& bar, uint32_t parity) -> bool {
        if (!mbar_wait(smem_u32(&bar), parity, ab)) return false;
        tc_fence_after();
        return true;
      };
      // descriptors of ring slot 0; slot s adds s * (slot bytes >> 4) to the
      // start-address field (no carry: shared addresses stay below 2^18)
      const uint64_t bK_0 = kmajor_base(sK), bV_0 = mnmajor_base(sV, 128);
      auto mma_S = [&](uint64_t bQ, uint32_t tS, uint64_t& sfull, uint32_t t) {
        const uint64_t bK = bK_0 + (uint64_t)((t % C::kKStages) * (C::kKBytes >> 4));
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk)
          mma_bf16(tS, bQ + kmajor_step(kk, 128), bK + kmajor_step(kk, 128), idS,
                   kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(&sfull));
      };
      auto mma_PV = [&](uint32_t tS, uint32_t tO, uint32_t t, bool first) {  // A = P from TMEM
        const uint64_t bV = bV_0 + (uint64_t)((t % C::kVStages) * (C::kVBytes >> 4));
        mma_bf16_ts(tO, tS, bV, idO, first ? 0u : 1u);
#pragma unroll
        for (int kk = 1; kk < kTile / 16; ++kk)
          mma_bf16_ts(tO, tS + kk * 8, bV + mnmajor_step(kk), idO, 1u);
      };
      const uint32_t tS0 = tmem + C::kTmemS, tS1 = tmem + C::kTmemS + 128;
      const uint32_t tO0 = tmem + C::kTmemO, tO1 = tmem + C::kTmemO + DV;
      // one Q tile's step at kv tile j (ring index t): when j is in its range,
      // wait for its P and do O += P V (first / last of the range flagged);
      // then S of kv tile j+1 when that is in its range
      auto step = [&](uint32_t tS, uint32_t tO, uint64_t bQ, uint64_t& pfull, uint64_t& sfull,
                      uint64_t& odone, uint32_t& cnt, bool pv, bool first, bool last,
                      bool s_next, uint32_t t) -> bool {
        if (pv) {
          if (!W(pfull, cnt & 1)) return false;
          mma_PV(tS, tO, t, first);
          if (last) mma_commit(smem_u32(&odone));
          ++cnt;
        }
        if (s_next) mma_S(bQ, tS, sfull, t + 1);
        return true;
      };
      auto flag = [&](const int& v) { return *static_cast<const volatile int*>(&v); };
      auto read_next = [&]() -> int {
        const uint32_t slot = item_iter & 1;
        if (!mbar_wait(smem_u32(&bars->item_full[slot]), (item_iter >> 1) & 1, ab)) {
          ok = false;
          return sh.n_items;
        }
        const int item = *static_cast<volatile int*>(&bars->item_slot[slot]);
        mbar_arrive(smem_u32(&bars->item_empty[slot]));
        return item;
      };
      for (int item = read_next(); ok && item < sh.n_items; ++item_iter, item = read_next()) {
        const Item it = decode_item(sh, tb, item, true);
        int lo0, hi0, lo1, hi1;
        kv_ranges(sh, it, lo0, hi0, lo1, hi1);
        if (!(ok = W(bars->q_full, item_iter & 1))) break;
        if constexpr (kMask) {
          // block mask: the kv tiles come in MaskOrder; the producer's flags
          // (read after the waits that publish them) say which Q tiles use
          // each, its place among each Q tile's tiles, and the item's end
          if (flag(bars->q_none)) {  // the mask drops every tile pair of the item
            mma_commit(smem_u32(&bars->q_empty));
            continue;
          }
          uint32_t t = kv_it;
          if (!(ok = W(bars->k_full[t % C::kKStages], (t / C::kKStages) & 1))) break;
          int f = flag(bars->kv_flags[t % C::kKStages]);
          if (f & kKvUse0) mma_S(bQ0, tS0, bars->s_full[0], t);
          if (f & kKvUse1) mma_S(bQ1, tS1, bars->s_full[1], t);
          mma_commit(smem_u32(&bars->k_empty[t % C::kKStages]));
          if (f & kKvItemLast) mma_commit(smem_u32(&bars->q_empty));
          for (;; ++t) {
            const bool next = !(f & kKvItemLast);
            if (!(ok = W(bars->v_full[t % C::kVStages], (t / C::kVStages) & 1))) break;
            int fn = 0;  // flags of the next kv tile
            if (next) {
              if (!(ok = W(bars->k_full[(t + 1) % C::kKStages], ((t + 1) / C::kKStages) & 1)))
                break;
              fn = flag(bars->kv_flags[(t + 1) % C::kKStages]);
            }
            if (!(ok = step(tS0, tO0, bQ0, bars->p_full[0], bars->s_full[0], bars->o_done[0], cnt0,
                            f & kKvUse0, f & kKvFirst0, f & kKvLast0, fn & kKvUse0, t)))
              break;
            if (!(ok = step(tS1, tO1, bQ1, bars->p_full[1], bars->s_full[1], bars->o_done[1], cnt1,
                            f & kKvUse1, f & kKvFirst1, f & kKvLast1, fn & kKvUse1, t)))
              break;
            mma_commit(smem_u32(&bars->v_empty[t % C::kVStages]));
            if (!next) break;
            mma_commit(smem_u32(&bars->k_empty[(t + 1) % C::kKStages]));
            if (fn & kKvItemLast) mma_commit(smem_u32(&bars->q_empty));  // after the last S
            f = fn;
          }
          if (!ok) break;
          kv_it = t + 1;
        } else {
          // without a block mask the kv tiles are lo0 .. hi1 (the two band
          // ranges leave no gap); Q tile w uses those in [lo_w, hi_w].  (This
          // form of the loop, a kv-tile cursor beside the step count and
          // range tests for the flags, issues faster than one that derives
          // the flags from the step count.)
          auto u0 = [&](int jj) { return jj >= lo0 && jj <= hi0; };
          auto u1 = [&](int jj) { return jj >= lo1 && jj <= hi1; };
          const int n = hi1 - lo0 + 1;
          int j = lo0;
          // S of the first kv tile (tile 1 joins later when its band starts later)
          if (!(ok = W(bars->k_full[kv_it % C::kKStages], (kv_it / C::kKStages) & 1))) break;
          if (u0(j)) mma_S(bQ0, tS0, bars->s_full[0], kv_it);
          if (u1(j)) mma_S(bQ1, tS1, bars->s_full[1], kv_it);
          mma_commit(smem_u32(&bars->k_empty[kv_it % C::kKStages]));
          if (n == 1) mma_commit(smem_u32(&bars->q_empty));
          for (int r = 0; ok && r < n; ++r) {
            const uint32_t t = kv_it + r;
            const bool next = r + 1 < n;
            const int jn = next ? j + 1 : hi1 + 1;
            if (!(ok = W(bars->v_full[t % C::kVStages], (t / C::kVStages) & 1))) break;
            if (next && !(ok = W(bars->k_full[(t + 1) % C::kKStages], ((t + 1) / C::kKStages) & 1)))
              break;
            if (!(ok = step(tS0, tO0, bQ0, bars->p_full[0], bars->s_full[0], bars->o_done[0], cnt0,
                            u0(j), j == lo0, j == hi0, next && u0(jn), t)))
              break;
            if (!(ok = step(tS1, tO1, bQ1, bars->p_full[1], bars->s_full[1], bars->o_done[1], cnt1,
                            u1(j), j == lo1, j == hi1, next && u1(jn), t)))
              break;
            mma_commit(smem_u32(&bars->v_empty[t % C::kVStages]));
            if (next) {
              mma_commit(smem_u32(&bars->k_empty[(t + 1) % C::kKStages]));
              if (r + 2 == n) mma_commit(smem_u32(&bars->q_empty));  // after the last S
            }
            j = jn;
          }
          if (!ok) break;
          kv_it += n;
        }
      }
      if (!ok) {
        mma_commit(smem_u32(&bars->drain));
        mbar_wait_drain(smem_u32(&bars->drain), 0);
      }
    }
   }
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int w = warp >> 2;                 // Q tile of this warpgroup
    const int r = (warp & 3) * 32 + lane;    // query row within the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::kTmemS + w * 128;
    const uint32_t tO = tmem + lane_base + C::kTmemO + w * DV;
    uint32_t cnt = 0, items_done = 0, n_read = 0;
    bool ok = true;
    auto read_next = [&]() -> int {
      const uint32_t slot = n_read & 1;
      if (!mbar_wait_warp(smem_u32(&bars->item_full[slot]), (n_read >> 1) & 1, ab)) {
        ok = false;
        return sh.n_items;
      }
      const int item = *static_cast<volatile int*>(&bars->item_slot[slot]);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->item_empty[slot]));
      ++n_read;
      return item;
    };
    for (int item = read_next(); ok && item < sh.n_items; item = read_next()) {
      const Item it = decode_item(sh, tb, item, true);
      int lo0, hi0, lo1, hi1;
      kv_ranges(sh, it, lo0, hi0, lo1, hi1);
      const int jlo = w ? lo1 : lo0, jhi = w ? hi1 : hi0;
      const int qt = 2 * it.tile + w;           // q-tile index within the sequence
      const int qidx = qt * kTile + r;
      float m = -INFINITY, l = 0.f;
      bool started = false;  // this Q tile has had a kv tile
      // kv tiles jlo .. jhi in order; with a block mask MaskOrder's subsequence
      // for this Q tile (first the tiles both Q tiles keep, then its own),
      // found 32 tiles at a time: each lane reads one mask byte, ballots
      // gather them (sweep 0: both keep, sweep 1: only this one)
      int sweep = 0, c0 = jlo - 32;
      uint32_t bits = 0;
      auto next_j = [&]() -> int {
        while (bits == 0) {
          c0 += 32;
          if (c0 > jhi) {
            if (sweep == 1) return INT_MAX;
            sweep = 1;
            c0 = jlo;
          }
          const int jj = c0 + lane;
          const uint32_t mine = __ballot_sync(0xffffffffu, kv_used<kMask>(sh, it, w, jj, jlo, jhi));
          const uint32_t other = __ballot_sync(
              0xffffffffu, kv_used<kMask>(sh, it, w ^ 1, jj, w ? lo0 : lo1, w ? hi0 : hi1));
          bits = sweep == 0 ? (mine & other) : (mine & ~other);
        }
        const int b = __ffs(bits) - 1;
        bits &= bits - 1;
        return c0 + b;
      };
      for (int j = kMask ? next_j() : jlo; j <= jhi; j = kMask ? next_j() : j + 1) {
        if (!(ok = mbar_wait_warp(smem_u32(&bars->s_full[w]), cnt & 1, ab))) break;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
        tmem_ld_wait();
        const int kbase = j * kTile;
        // some row of the tile does not see all of its keys: the band's right
        // edge (first row) or left edge (last row) crosses it, or it is ragged
        const bool need_mask =
            (sh.wr >= 0 && kbase + kTile - 1 > qt * kTile + band_off(sh, it) + sh.wr) ||
            (sh.wl >= 0 && kbase < qt * kTile + kTile - 1 + band_off(sh, it) - sh.wl) ||
            (kbase + kTile > it.Lk);
        // row maximum over 8 independent chains (a single chain is latency-bound)
        float mx[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mx[u] = -INFINITY;
        if (need_mask) {  // edge or ragged tile: keys outside the row's band -> -inf
          // this row's visible keys, relative to the tile: [klo, khi)
          const int klo = sh.wl >= 0 ? qidx + band_off(sh, it) - sh.wl - kbase : INT_MIN / 2;
          const int khi =
              min(it.Lk, sh.wr >= 0 ? qidx + band_off(sh, it) + sh.wr + 1 : it.Lk) - kbase;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float x = (c * 32 + e >= klo && c * 32 + e < khi) ? __uint_as_float(sr[c][e])
                                                                      : -INFINITY;
              sr[c][e] = __float_as_uint(x);
              mx[e & 7] = fmaxf(mx[e & 7], x);
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int e = 0; e < 32; e += 2)
              mx[(e >> 1) & 7] = max3(mx[(e >> 1) & 7], __uint_as_float(sr[c][e]),
                                      __uint_as_float(sr[c][e + 1]));
          }
        }
        const float rowmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                   fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        // all PV products of this warpgroup issued before this S are complete
        // (tensor-core work completes in issue order), so O is stable here
        const float m_new = fmaxf(m, rowmax * scale_log2);
        // a row that has seen no key yet (its band starts in a later tile of
        // the Q tile's range) keeps m = -inf; its P row is exp2(-inf) = 0
        const bool none = need_mask && m_new == -INFINITY;  // unmasked tiles show every key
        const bool resc = !none && (m_new - m) > 8.0f;  // also true on a row's first keys
        const float m_use = none ? 0.f : (resc ? m_new : m);
        const float alpha = resc ? ex2(m - m_use) : 1.0f;
        uint32_t pk0[32], pk1[32];  // P as bf16 pairs: keys 0-63, 64-127
        const float rowsum = softmax_exp(sr, scale_log2, m_use, pk0, pk1);
        if ((kMask ? started : j > jlo) && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
          for (int c = 0; c < DV / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tO + c * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st32(tO + c * 32, ov);
          }
        }
        l = l * alpha + rowsum;
        m = none ? -INFINITY : m_use;
        // P (bf16 pairs) over the S columns just read: A operand of O += P V
        tmem_st32(tS, pk0);
        tmem_st32(tS + 32, pk1);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[w]));
        started = true;
        ++cnt;
      }
      if (!ok) break;
      const bool valid = qidx < it.Lq;
      __nv_bfloat16* orow =
          out + (int64_t)(it.row0 + qidx) * o_row_stride + (int64_t)it.head * DV;
      auto lse_at = [&]() {
        return (int64_t)it.head * lse_head_stride +
               (sh.varlen ? (int64_t)it.row0 : (int64_t)it.seq * lse_seq_stride) + qidx;
      };
      if (kMask && !started) {
        // the block mask drops every kv tile of this Q tile: its rows see no
        // key (empty sums): O = 0, LSE = -inf
        if (valid) {
#pragma unroll 1
          for (int c = 0; c < DV / 8; ++c)
            *reinterpret_cast<uint4*>(orow + c * 8) = make_uint4(0u, 0u, 0u, 0u);
          if (lse != nullptr) lse[lse_at()] = -INFINITY;
        }
        continue;
      }
      // epilogue: O / l and the log-sum-exp (under a block mask a row can have
      // seen no key: l = 0, O = 0 and LSE = -inf)
      if (!(ok = mbar_wait_warp(smem_u32(&bars->o_done[w]), items_done & 1, ab))) break;
      ++items_done;
      tc_fence_after();
      const bool no_key = kMask && !(l > 0.f);
      const float inv_l = no_key ? 0.f : 1.0f / l;
      // O rows 32-byte aligned (base and row stride)
      const bool st32 = ((reinterpret_cast<uintptr_t>(out) | (uintptr_t)(o_row_stride * 2)) & 31u) == 0;
#pragma unroll 1
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tO + c * 32, ov);
        tmem_ld_wait();
        if (valid) {
          uint32_t pw[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pw[e] = pack_bf16(__uint_as_float(ov[2 * e]) * inv_l, __uint_as_float(ov[2 * e + 1]) * inv_l);
          if (st32) {  // 32-byte stores: half the requests of 16-byte ones
            st_global_v8(orow + c * 32, pw[0], pw[1], pw[2], pw[3], pw[4], pw[5], pw[6], pw[7]);
            st_global_v8(orow + c * 32 + 16, pw[8], pw[9], pw[10], pw[11], pw[12], pw[13], pw[14],
                         pw[15]);
          } else {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              *reinterpret_cast<uint4*>(orow + c * 32 + q4 * 8) =
                  make_uint4(pw[4 * q4], pw[4 * q4 + 1], pw[4 * q4 + 2], pw[4 * q4 + 3]);
          }
        }
      }
      tc_fence_before();
      if (lse != nullptr && valid)
        lse[lse_at()] = no_key ? -INFINITY : (m + log2f(l)) * 0.69314718055994530942f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int DQK, int DV, bool kMask, bool kLeft>
cudaError_t launch_kernel(const FwdLaunch& L) {
  using C = FwdCfg<DQK, DV>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.grid);
  cfg.blockDim = dim3(kFwdThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = L.stream;
  if (L.tables) {
    auto* k = attn_fwd_kernel<DQK, DV, VarlenTables, kMask, kLeft>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, k, L.tm_q, L.tm_k, L.tm_v,
                              reinterpret_cast<__nv_bfloat16*>(L.o), L.lse, L.o_row_stride,
                              L.lse_head_stride, L.lse_seq_stride, L.scale_log2, L.status, L.claim,
                              L.sh, *L.tables);
  }
  auto* k = attn_fwd_kernel<DQK, DV, NoTables, kMask, kLeft>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, k, L.tm_q, L.tm_k, L.tm_v, reinterpret_cast<__nv_bfloat16*>(L.o),
                            L.lse, L.o_row_stride, L.lse_head_stride, L.lse_seq_stride,
                            L.scale_log2, L.status, L.claim, L.sh, NoTables{});
}

template <int DQK, int DV>
cudaError_t launch_typed(const FwdLaunch& L) {
  const bool mask = L.sh.blk != nullptr, left = L.sh.wl >= 0;
  if (mask) return left ? launch_kernel<DQK, DV, true, true>(L) : launch_kernel<DQK, DV, true, false>(L);
  return left ? launch_kernel<DQK, DV, false, true>(L) : launch_kernel<DQK, DV, false, false>(L);
}

}  // namespace

// Sticky status word of the forward kernels on each device (a bounded wait
// that gave up writes its code here; attn_fwd_status reads and clears it).
__device__ int g_fwd_status = 0;

// Work-item counters of the forward: a pair (items claimed, CTAs done) per
// call in flight, taken round-robin, so up to kFwdClaimSlots calls may
// overlap on different streams.  A kernel leaves its pair at zero.
__device__ int g_fwd_claim[2 * kFwdClaimSlots];

int* fwd_claim_ptr(int slot) {
  void* p = nullptr;
  if (slot < 0 || slot >= kFwdClaimSlots) return nullptr;
  if (cudaGetSymbolAddress(&p, g_fwd_claim) != cudaSuccess) return nullptr;
  return static_cast<int*>(p) + 2 * slot;
}

int* fwd_status_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_fwd_status) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

int fwd_smem_bytes(int dqk, int dv) {
  if (dqk == 64 && dv == 64) return FwdCfg<64, 64>::kSmemBytes;
  if (dqk == 128 && dv == 128) return FwdCfg<128, 128>::kSmemBytes;
  if (dqk == 192 && dv == 128) return FwdCfg<192, 128>::kSmemBytes;
  return -1;
}

cudaError_t launch_fwd(const FwdLaunch& L, int dqk, int dv) {
  if (dqk == 64 && dv == 64) return launch_typed<64, 64>(L);
  if (dqk == 128 && dv == 128) return launch_typed<128, 128>(L);
  if (dqk == 192 && dv == 128) return launch_typed<192, 128>(L);
  return cudaErrorInvalidValue;
}

}  // namespace attn
