// attn_bwd_pair.cu — the backward main kernel on CTA pairs (tcgen05 cta_group::2)
// for dqk = dv = 128, as "深度学习反向传播优化：2-CTA MMA模式与内存访问优化" §2.1-2.2
// describes it: two CTAs on neighbouring SMs issue their products as one MMA of
// M = 256 rows with the B operand split between their shared memories, and the
// dQ product contracts over both CTAs' keys after the CTAs exchange halves of
// dS through distributed shared memory — so each dQ tile receives one fp32
// contribution per PAIR of key tiles (half the global atomics of the one-CTA
// kernel, §3.1).
//
// A work item is (sequence, head, pair p): CTA c of the cluster owns key tile
// j_c = 2p + c (K_jc, V_jc in its shared memory, dK_jc and dV_jc in its tensor
// memory) and the pair walks the query tiles i of the pair's band:
//   S^T  = K Q_i^T      M = 256 keys (128 per CTA), N = 128 queries: CTA c
//                       supplies queries [64c, 64c + 64) of Q_i (all d)
//   P^T  = exp2(S^T s log2e - LSE2_i)          per CTA, as in the one-CTA kernel
//   dP^T = V dO_i^T     as S^T, with dO_i
//   dV  += P^T dO_i     A = P^T (tensor memory), B = dO_i[:, 64c .. 64c+63] from CTA c
//   dS^T = P^T ⊙ (dP^T - D_i)  into tensor memory (A of dK) and into the dQ
//                       operand: the panel of queries [64g, 64g+64) goes to CTA g
//   dK  += dS^T Q_i     A = dS^T (tensor memory), B = Q_i[:, 64c .. 64c+63]
//   dQ_i = dS K         M = 128 queries (64 per CTA), K = 256 keys of both tiles,
//                       N = 128: CTA c holds dS[keys of j0 | j1][its 64 queries]
//                       and K_j0, K_j1 columns [64c, 64c+64)
// Each CTA adds its 64 rows of dQ_i to the fp32 accumulator (ordered by pair in
// deterministic mode, one semaphore per tile half).
//
// Roles (512 threads per CTA, as in the one-CTA kernel):
//   warps 0-7   P / dS warpgroups (thread = key row = TMEM lane), both CTAs
//   warps 8-11  dQ drain + atomics, dK / dV epilogue, both CTAs
//   warp 12     producer: the leader claims work items and hands them to the
//               peer; each CTA loads its own operand halves, completing on the
//               leader's barriers (TMA .cta_group::2)
//   warp 13     MMA issuer (leader only); tensor memory of both CTAs
// Barriers that gate pair MMAs live in the leader and receive arrivals from
// both CTAs; MMA completions are multicast to the same barrier in both CTAs.
//
// Tensor memory (512 columns, per CTA): S^T [0,128) with P^T packed in place;
// dP^T [128,256) with dS^T packed in place; dQ (64 columns) [128,192) once dK
// has read dS^T; dV [256,384); dK [384,512).
// Shared memory: K, V of the own tile (64 KB), the dQ operands (K halves and
// dS halves, 64 KB), one slot each of the S / dP operand halves of Q and dO
// (32 KB), two slots each of the dK / dV operand halves (64 KB) and of the
// per-row statistics: 226.5 KB.
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kPanel = kTile * 128;  // [128 rows][64] bf16, 128-byte swizzle
constexpr int kHalfPanel = 64 * 128;  // [64 rows][64]
constexpr int kThreads = 512;
constexpr int kTmaWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kMaxSmem = 232448;
constexpr uint16_t kBoth = 3;  // multicast mask: both CTAs of the pair

// Registers after the split (launched with 512 x 128): P/dS 112, dQ 144 (a
// thread drains 64 dQ values), control 144 (the MMA issuer keeps the
// operand descriptors of both CTAs' buffers live).
constexpr uint32_t kRegsCompute = 112, kRegsDq = 144, kRegsCtl = 144;
static_assert(2 * kRegsCompute + kRegsDq + kRegsCtl <= 4 * 128, "register split");
// setmaxnreg.dec may only lower and setmaxnreg.inc only raise the count a
// warpgroup holds (128 at launch)
static_assert(kRegsCompute <= 128 && kRegsDq >= 128 && kRegsCtl >= 128, "setmaxnreg direction");

struct Cfg {
  static constexpr int kOffK = 0;                         // own K: 2 panels
  static constexpr int kOffV = kOffK + 2 * kPanel;        // own V: 2 panels
  static constexpr int kOffKdq = kOffV + 2 * kPanel;      // K_j0, K_j1 columns [64c, 64c+64)
  static constexpr int kOffdSq = kOffKdq + 2 * kPanel;    // dS[keys j0 | j1][queries 64c..]
  static constexpr int kOffQs = kOffdSq + 2 * kPanel;     // Q rows 64c.., d halves 0 and 1
  static constexpr int kOffdOp = kOffQs + 2 * kHalfPanel; // dO rows 64c.., dv halves
  static constexpr int kOffQk = kOffdOp + 2 * kHalfPanel; // 2 slots: Q[:, 64c..64c+63]
  static constexpr int kOffdOv = kOffQk + 2 * kPanel;     // 2 slots: dO[:, 64c..]
  static constexpr int kOffStat = kOffdOv + 2 * kPanel;   // 2 slots: -LSE2, -D (128 each)
  static constexpr int kStatBytes = 2 * kTile * 4;
  static constexpr int kOffBar = kOffStat + 2 * kStatBytes;
  static constexpr int kBarBytes = 512;
  static constexpr int kSmemBytes = kOffBar + kBarBytes;
  static_assert(kSmemBytes <= kMaxSmem, "shared memory budget");
  static constexpr uint32_t kTmemS = 0, kTmemdP = 128, kTmemdQ = 128, kTmemdV = 256,
                            kTmemdK = 384, kTmemCols = 512;
  // transaction bytes of the pair (both CTAs) per barrier phase
  static constexpr uint32_t kKvTx = 2 * 6 * kPanel;
  static constexpr uint32_t kHalfTx = 2 * 2 * kHalfPanel;  // Qs or dOp
  static constexpr uint32_t kSlotTx = 2 * kPanel;          // Qk or dOv
};

struct Bars {
  uint64_t item_full[2], item_empty[2];
  uint64_t kv_full, kv_done, acc_free;
  uint64_t qs_full, qs_empty, dop_full, dop_empty;
  uint64_t qk_full[2], qk_empty[2], dov_full[2], dov_empty[2];
  uint64_t stat_full[2], stat_empty[2];
  uint64_t s_full, p_full, dp_full, ds_half[2], ds_free, dq_full, dq_free;
  uint64_t drain;
  int item_slot[2];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= Cfg::kBarBytes, "barrier block size");

// Optional phase trace of the first cluster (compiled in only with
// -DATTN_TRACE): the first thread of each role stores (clock64 << 8 | event)
// for q-tile steps [ATTN_TRACE_FROM, ATTN_TRACE_FROM + 8), 64 records per
// thread, indexed by (CTA, thread).  Clocks are per SM: compare events of one
// CTA only.
#ifdef ATTN_TRACE
#ifndef ATTN_TRACE_FROM
#define ATTN_TRACE_FROM 40
#endif
constexpr int kTraceCap = 64;
#define PAIR_TRACE_DECL int tr_n = 0
#define PAIR_TRACE(ev, step)                                                                 \
  do {                                                                                       \
    if (a.trace != nullptr && blockIdx.x < 2 && (uint32_t)(step) >= ATTN_TRACE_FROM &&      \
        (uint32_t)(step) < ATTN_TRACE_FROM + 8 && tr_n < kTraceCap)                          \
      a.trace[(blockIdx.x * kThreads + threadIdx.x) * kTraceCap + tr_n++] =                  \
          ((unsigned long long)clock64() << 8) | (unsigned)(ev);                             \
  } while (0)
#else
#define PAIR_TRACE_DECL \
  do {                  \
  } while (0)
#define PAIR_TRACE(ev, step) \
  do {                       \
  } while (0)
#endif

struct PairArgs {
#ifdef ATTN_TRACE
  unsigned long long* trace;
#endif
  int sem_bias;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int64_t dk_row_stride, dv_row_stride;
  float scale, scale_log2;
  int deterministic;
  BwdWorkspace ws;
  SeqShape sh;
};

// TMEM column of the packed bf16 operand (P^T, dS^T) for K-step kk (16 queries):
// the queries of warpgroup g are packed into the first 32 of its 64 columns.
__device__ __forceinline__ uint32_t pk_col(int kk) { return (kk >> 2) * 64 + (kk & 3) * 8; }

// Pair items: per (sequence, head), ceil(key tiles / 2) pairs, taken in
// ascending pair order (descending in deterministic mode); the item's
// `tile` is the pair index p (key tiles 2p, 2p + 1).
template <typename Tables>
__device__ __forceinline__ Item decode_pair(const SeqShape& sh, const Tables& tb, int item);

template <>
__device__ __forceinline__ Item decode_pair<NoTables>(const SeqShape& sh, const NoTables&,
                                                      int item) {
  const int np = cdiv(sh.nk_tiles, 2);
  Item it;
  const int bh = item / np;
  const int rank = item - bh * np;
  it.tile = sh.descending ? np - 1 - rank : rank;
  it.seq = bh / sh.H;
  it.head = bh - it.seq * sh.H;
  it.Lq = sh.Tq;
  it.Lk = sh.Tk;
  it.row0 = it.seq * sh.Tq;
  it.krow0 = it.seq * sh.Tk;
  it.band_off = sh.band_off;
  it.tile_base = it.seq * sh.nq_tiles;
  return it;
}

template <>
__device__ __forceinline__ Item decode_pair<VarlenTables>(const SeqShape& sh,
                                                          const VarlenTables& tb, int item) {
  int lo = 0, hi = sh.nseq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tb.item_start[mid] <= item) lo = mid; else hi = mid - 1;
  }
  Item it;
  it.seq = tb.order[lo];
  const int local = item - tb.item_start[lo];
  it.row0 = tb.cu[it.seq];
  it.krow0 = tb.cuk[it.seq];
  it.Lq = tb.cu[it.seq + 1] - it.row0;
  it.Lk = tb.cuk[it.seq + 1] - it.krow0;
  it.band_off = it.Lk - it.Lq;
  const int np = cdiv(it.Lk, 2 * kTile);
  it.head = local / np;
  const int rank = local - it.head * np;
  it.tile = sh.descending ? np - 1 - rank : rank;
  it.tile_base = tb.tile_start[it.seq];
  return it;
}

// Query tiles of the pair's band: those of key tile 2p through those of 2p + 1.
__device__ __forceinline__ void pair_band(const SeqShape& sh, const Item& it, int& i0, int& i1) {
  const int nq = cdiv(it.Lq, kTile);
  Item t = it;
  t.tile = 2 * it.tile;
  i0 = first_qtile(sh, t, t.tile);
  t.tile = 2 * it.tile + 1;
  i1 = last_qtile(sh, t, t.tile, nq) + 1;
}

template <typename Tables>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_bwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_q64,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_do64, const PairArgs a,
                         const __grid_constant__ Tables tb) {
  using C = Cfg;
  extern __shared__ __align__(1024) uint8_t smem[];
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kOffBar);
  const uint32_t rank = cluster_rank();  // 0: leader
  const bool leader = rank == 0;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const SeqShape& sh = a.sh;
  Abort ab{&bars->abort_flag, a.ws.header};
  PAIR_TRACE_DECL;
  const bool misaligned = (smem_u32(smem) & 1023u) != 0;
  if (threadIdx.x == 0) {
    bars->abort_flag = misaligned ? 1 : 0;
    if (misaligned) atomicCAS(a.ws.header, 0, kStatusInternal);
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_u32(&bars->item_full[k]), 1);
      mbar_init(smem_u32(&bars->item_empty[k]), 2 * (8 + 4) + 1 + 1);  // P, dQ; MMA; peer producer
      mbar_init(smem_u32(&bars->qk_full[k]), 1);
      mbar_init(smem_u32(&bars->qk_empty[k]), 1);
      mbar_init(smem_u32(&bars->dov_full[k]), 1);
      mbar_init(smem_u32(&bars->dov_empty[k]), 1);
      mbar_init(smem_u32(&bars->stat_full[k]), 1);
      mbar_init(smem_u32(&bars->stat_empty[k]), 8);
      mbar_init(smem_u32(&bars->ds_half[k]), 16);
    }
    mbar_init(smem_u32(&bars->kv_full), 1);
    mbar_init(smem_u32(&bars->kv_done), 1);
    mbar_init(smem_u32(&bars->acc_free), 8);
    mbar_init(smem_u32(&bars->qs_full), 1);
    mbar_init(smem_u32(&bars->qs_empty), 1);
    mbar_init(smem_u32(&bars->dop_full), 1);
    mbar_init(smem_u32(&bars->dop_empty), 1);
    mbar_init(smem_u32(&bars->s_full), 1);
    mbar_init(smem_u32(&bars->p_full), 16);
    mbar_init(smem_u32(&bars->dp_full), 1);
    mbar_init(smem_u32(&bars->ds_free), 1);
    mbar_init(smem_u32(&bars->dq_full), 1);
    mbar_init(smem_u32(&bars->dq_free), 8);
    mbar_init(smem_u32(&bars->drain), 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(smem_u32(&bars->tmem_base), C::kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == kTmaWarp && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_q64);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_do);
    prefetch_tmap(&tm_do64);
  }
  tc_fence_before();
  cluster_sync();  // both CTAs: barriers initialised, tensor memory allocated
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // the leader's copy of a barrier, as a cluster address
  auto L = [&](uint64_t& bar) { return mapa_shared(smem_u32(&bar), 0); };

  if (warp >= 12) {
    regs_inc<kRegsCtl>();
    if (warp == kTmaWarp && lane == 0 && !misaligned) {
      // ============================================= producer (both CTAs)
      uint32_t q_it = 0;
      bool ok = true;
      const uint32_t sK = smem_u32(smem + C::kOffK), sV = smem_u32(smem + C::kOffV);
      const uint32_t sKdq = smem_u32(smem + C::kOffKdq);
      const uint32_t sQs = smem_u32(smem + C::kOffQs), sdOp = smem_u32(smem + C::kOffdOp);
      const uint32_t sQk = smem_u32(smem + C::kOffQk), sdOv = smem_u32(smem + C::kOffdOv);
      const uint32_t sStat = smem_u32(smem + C::kOffStat);
      for (uint32_t k = 0;; ++k) {
        const uint32_t slot = k & 1;
        int item;
        if (leader) {
          if (!(ok = mbar_wait_cluster(smem_u32(&bars->item_empty[slot]), ((k >> 1) & 1) ^ 1, ab)))
            break;
          item = ld_acquire_gpu(a.ws.header) != 0 ? sh.n_items : atomicAdd(&a.ws.header[1], 1);
          bars->item_slot[slot] = item;
          const uint32_t peer_slot = mapa_shared(smem_u32(&bars->item_slot[slot]), 1);
          asm volatile("st.shared::cluster.b32 [%0], %1;" ::"r"(peer_slot), "r"(item) : "memory");
          mbar_arrive_cluster(mapa_shared(smem_u32(&bars->item_full[slot]), 0));
          mbar_arrive_cluster(mapa_shared(smem_u32(&bars->item_full[slot]), 1));
        } else {
          if (!(ok = mbar_wait_cluster(smem_u32(&bars->item_full[slot]), (k >> 1) & 1, ab))) break;
          item = *static_cast<volatile int*>(&bars->item_slot[slot]);
          mbar_arrive_cluster(L(bars->item_empty[slot]));
        }
        if (item >= sh.n_items) break;
        const Item it = decode_pair(sh, tb, item);
        const int j0 = 2 * it.tile, jc = j0 + (int)rank;
        const int kbase = key_row0(sh, it);
        // own K, V and the dQ operand's K halves (previous item's MMAs done with them)
        if (!(ok = mbar_wait(smem_u32(&bars->kv_done), (k & 1) ^ 1, ab))) break;
        if (leader) mbar_arrive_expect_tx(smem_u32(&bars->kv_full), C::kKvTx);
        const uint32_t kvb = L(bars->kv_full);
        for (int p = 0; p < 2; ++p) {
          tma_load_3d_pair(sK + p * kPanel, &tm_k, kvb, p * 64, it.head, kbase + jc * kTile);
          tma_load_3d_pair(sV + p * kPanel, &tm_v, kvb, p * 64, it.head, kbase + jc * kTile);
        }
        for (int t = 0; t < 2; ++t)
          tma_load_3d_pair(sKdq + t * kPanel, &tm_k, kvb, (int)rank * 64, it.head,
                           kbase + (j0 + t) * kTile);
        int i0, i1;
        pair_band(sh, it, i0, i1);
        for (int i = i0; i < i1; ++i, ++q_it) {
          const uint32_t u = q_it, st = u & 1, par1 = u & 1, par2 = (u >> 1) & 1;
          const int qrow = it.row0 + i * kTile;
          const int64_t g = (int64_t)(it.tile_base + i) * sh.H + it.head;
          // in the order the MMAs free the slots: dV (dO halves), S (Q rows),
          // dK (Q halves), dP (dO rows)
          if (!(ok = mbar_wait(smem_u32(&bars->dov_empty[st]), par2 ^ 1, ab))) break;
          PAIR_TRACE(50, u);
          if (leader) mbar_arrive_expect_tx(smem_u32(&bars->dov_full[st]), C::kSlotTx);
          tma_load_3d_pair(sdOv + st * kPanel, &tm_do, L(bars->dov_full[st]), (int)rank * 64,
                           it.head, qrow);
          if (!(ok = mbar_wait(smem_u32(&bars->qs_empty), par1 ^ 1, ab))) break;
          PAIR_TRACE(51, u);
          if (leader) mbar_arrive_expect_tx(smem_u32(&bars->qs_full), C::kHalfTx);
          for (int p = 0; p < 2; ++p)
            tma_load_3d_pair(sQs + p * kHalfPanel, &tm_q64, L(bars->qs_full), p * 64, it.head,
                             qrow + (int)rank * 64);
          if (!(ok = mbar_wait(smem_u32(&bars->stat_empty[st]), par2 ^ 1, ab))) break;
          {
            const uint32_t sb = smem_u32(&bars->stat_full[st]);
            mbar_arrive_expect_tx(sb, C::kStatBytes);
            bulk_load(sStat + st * C::kStatBytes, a.ws.nlse2 + g * kTile, kTile * 4, sb);
            bulk_load(sStat + st * C::kStatBytes + kTile * 4, a.ws.ndsum + g * kTile, kTile * 4, sb);
          }
          if (!(ok = mbar_wait(smem_u32(&bars->qk_empty[st]), par2 ^ 1, ab))) break;
          PAIR_TRACE(53, u);
          if (leader) mbar_arrive_expect_tx(smem_u32(&bars->qk_full[st]), C::kSlotTx);
          tma_load_3d_pair(sQk + st * kPanel, &tm_q, L(bars->qk_full[st]), (int)rank * 64,
                           it.head, qrow);
          if (!(ok = mbar_wait(smem_u32(&bars->dop_empty), par1 ^ 1, ab))) break;
          PAIR_TRACE(54, u);
          if (leader) mbar_arrive_expect_tx(smem_u32(&bars->dop_full), C::kHalfTx);
          for (int p = 0; p < 2; ++p)
            tma_load_3d_pair(sdOp + p * kHalfPanel, &tm_do64, L(bars->dop_full), p * 64, it.head,
                             qrow + (int)rank * 64);
        }
        if (!ok) break;
      }
      if (!ok) {
        // copies already issued complete on the leader's barriers, which this
        // CTA cannot wait on: give them time to land before the pair leaves
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 2000000ull) {
        }
      }
    } else if (warp == kMmaWarp && lane == 0 && leader && !misaligned) {
      // ============================================= MMA issuer (leader)
      constexpr uint32_t idS = idesc_bf16(256, 128, false, false);  // S^T, dP^T
      constexpr uint32_t idV = idesc_bf16(256, 128, false, true);   // dV += P^T dO
      constexpr uint32_t idK = idesc_bf16(256, 128, false, true);   // dK += dS^T Q
      constexpr uint32_t idQ = idesc_bf16(128, 128, true, true);    // dQ = dS K
      const uint64_t bK = kmajor_base(smem_u32(smem + C::kOffK));
      const uint64_t bV = kmajor_base(smem_u32(smem + C::kOffV));
      const uint64_t bKdq = mnmajor_base(smem_u32(smem + C::kOffKdq), 128);
      const uint64_t bdSq = mnmajor_base(smem_u32(smem + C::kOffdSq), 128);
      const uint64_t bQs = kmajor_base(smem_u32(smem + C::kOffQs));
      const uint64_t bdOp = kmajor_base(smem_u32(smem + C::kOffdOp));
      const uint32_t tS = tmem + C::kTmemS, tdP = tmem + C::kTmemdP, tdQ = tmem + C::kTmemdQ;
      const uint32_t tdV = tmem + C::kTmemdV, tdK = tmem + C::kTmemdK;
      uint32_t q_it = 0, gi = 0;
      bool ok = true;
      auto W = [&](uint64_t& bar, uint32_t parity) -> bool {
        if (!mbar_wait_cluster(smem_u32(&bar), parity, ab)) return false;
        tc_fence_after();
        return true;
      };
      auto commit = [&](uint64_t& bar) { mma_commit_pair(smem_u32(&bar), kBoth); };
      auto mma_S = [&]() {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_pair(tS, bK + kmajor_step(kk, 128), bQs + kmajor_step(kk, 64), idS,
                        kk > 0 ? 1u : 0u);
        commit(bars->s_full);
        commit(bars->qs_empty);
      };
      auto mma_dP = [&]() {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_pair(tdP, bV + kmajor_step(kk, 128), bdOp + kmajor_step(kk, 64), idS,
                        kk > 0 ? 1u : 0u);
        commit(bars->dp_full);
        commit(bars->dop_empty);
      };
      auto mma_dV = [&](uint32_t st, bool first) {
        const uint64_t b = mnmajor_base(smem_u32(smem + C::kOffdOv + st * kPanel), 128);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_pair_ts(tdV, tS + pk_col(kk), b + mnmajor_step(kk), idV,
                           (first && kk == 0) ? 0u : 1u);
        commit(bars->dov_empty[st]);
      };
      // dK += dS^T Q in two halves: K steps {0,1,4,5} read the dS^T columns the
      // P / dS warps finish first, {2,3,6,7} the rest
      auto mma_dK = [&](uint32_t st, bool first, int half) {
        const uint64_t b = mnmajor_base(smem_u32(smem + C::kOffQk + st * kPanel), 128);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int kk = (v & 1) + (v >> 1) * 4 + half * 2;
          mma_bf16_pair_ts(tdK, tdP + pk_col(kk), b + mnmajor_step(kk), idK,
                           (first && half == 0 && v == 0) ? 0u : 1u);
        }
      };
      // dQ over the 256 keys of the pair: K steps 0-7 key tile j0, 8-15 j1
      auto mma_dQ = [&]() {
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const uint64_t off = (uint64_t)((kk >> 3) * (kPanel >> 4)) + mnmajor_step(kk & 7);
          mma_bf16_pair(tdQ, bdSq + off, bKdq + off, idQ, kk > 0 ? 1u : 0u);
        }
        commit(bars->dq_full);
        commit(bars->ds_free);
      };
      for (uint32_t k = 0; ok; ++k) {
        const uint32_t slot = k & 1;
        if (!(ok = mbar_wait_cluster(smem_u32(&bars->item_full[slot]), (k >> 1) & 1, ab))) break;
        const int item = *static_cast<volatile int*>(&bars->item_slot[slot]);
        mbar_arrive_cluster(L(bars->item_empty[slot]));
        if (item >= sh.n_items) break;
        const Item it = decode_pair(sh, tb, item);
        int i0, i1;
        pair_band(sh, it, i0, i1);
        if (!(ok = W(bars->kv_full, k & 1))) break;
        if (!(ok = W(bars->acc_free, (k & 1) ^ 1))) break;
        if (i0 < i1) {
          if (!(ok = W(bars->qs_full, q_it & 1))) break;
          mma_S();
          if (gi > 0 && !(ok = W(bars->dq_free, (gi - 1) & 1))) break;
          if (!(ok = W(bars->dop_full, q_it & 1))) break;
          mma_dP();
          for (int i = i0; i < i1; ++i, ++q_it, ++gi) {
            const uint32_t st = q_it & 1, par2 = (q_it >> 1) & 1;
            const bool first = i == i0, more = i + 1 < i1;
            if (!(ok = W(bars->p_full, gi & 1))) break;
            PAIR_TRACE(10, gi);
            if (!(ok = W(bars->dov_full[st], par2))) break;
            PAIR_TRACE(11, gi);
            mma_dV(st, first);
            if (more) {
              if (!(ok = W(bars->qs_full, (q_it + 1) & 1))) break;
              PAIR_TRACE(12, gi);
              mma_S();
            }
            if (!(ok = W(bars->ds_half[0], gi & 1))) break;
            PAIR_TRACE(13, gi);
            if (!(ok = W(bars->qk_full[st], par2))) break;
            PAIR_TRACE(14, gi);
            mma_dK(st, first, 0);
            if (!(ok = W(bars->ds_half[1], gi & 1))) break;
            PAIR_TRACE(15, gi);
            mma_dK(st, first, 1);
            commit(bars->qk_empty[st]);
            mma_dQ();  // after dK: dQ's columns hold half of dS^T until dK has read it
            PAIR_TRACE(16, gi);
            if (more) {
              if (!(ok = W(bars->dq_free, gi & 1))) break;
              PAIR_TRACE(17, gi);
              if (!(ok = W(bars->dop_full, (q_it + 1) & 1))) break;
              PAIR_TRACE(18, gi);
              mma_dP();
            }
          }
          if (!ok) break;
        }
        commit(bars->kv_done);
      }
      if (!ok) {
        mma_commit_pair(smem_u32(&bars->drain), 1);
        mbar_wait_drain(smem_u32(&bars->drain), 0);
      }
    }
  } else if (warp < 8) {
    regs_dec<kRegsCompute>();
    // ============================================= P / dS warpgroups (both CTAs)
    const int grp = warp >> 2;             // queries [64 grp, 64 grp + 64) of the tile
    const int r = (warp & 3) * 32 + lane;  // TMEM lane = key row
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float* stat_f = reinterpret_cast<const float*>(smem + C::kOffStat);
    // this group's dS panel goes to CTA grp (which supplies those queries to
    // dQ), into the slot of this CTA's key tile
    const uint32_t dsq_local = smem_u32(smem + C::kOffdSq + rank * kPanel);
    const uint32_t dsq_dst = mapa_shared(dsq_local, (uint32_t)grp);
    const bool dsq_remote = (uint32_t)grp != rank;
    uint32_t q_it = 0, gi = 0;
    bool ok = !misaligned;
    for (uint32_t k = 0; ok; ++k) {
      const uint32_t slot = k & 1;
      if (!(ok = mbar_wait_cluster_warp(smem_u32(&bars->item_full[slot]), (k >> 1) & 1, ab))) break;
      const int item = *static_cast<volatile int*>(&bars->item_slot[slot]);
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(L(bars->item_empty[slot]));
      if (item >= sh.n_items) break;
      const Item it = decode_pair(sh, tb, item);
      int i0, i1;
      pair_band(sh, it, i0, i1);
      const int kidx0 = (2 * it.tile + (int)rank) * kTile + r;  // this thread's key
      const bool key_ok = kidx0 < it.Lk;
      for (int i = i0; i < i1; ++i, ++q_it, ++gi) {
        const uint32_t st = q_it & 1;
        if (!(ok = mbar_wait_warp(smem_u32(&bars->stat_full[st]), (q_it >> 1) & 1, ab))) break;
        const float* nlse2 = stat_f + st * (C::kStatBytes / 4) + grp * 64;
        const float* ndsum = nlse2 + kTile;
        if (!(ok = mbar_wait_warp(smem_u32(&bars->s_full), gi & 1, ab))) break;
        tc_fence_after();
        if (lane == 0 && (warp & 3) == 0) PAIR_TRACE(20, gi);
        uint32_t pk[32];
        const int qrel = kidx0 - kTile * i - grp * 64;
        const int qmin = !key_ok ? 64 : (sh.wr >= 0 ? min(64, max(0, qrel - band_off(sh, it) - sh.wr)) : 0);
        const int qmax = sh.wl >= 0 ? min(64, max(0, qrel - band_off(sh, it) + sh.wl + 1)) : 64;
        const uint64_t sc2 = f2(a.scale_log2, a.scale_log2);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t sr[32];
          tmem_ld32(tmem + lane_base + C::kTmemS + grp * 64 + c * 32, sr);
          tmem_ld_wait();
          if (qmin > 0 || qmax < 64) {
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const int q = c * 32 + e;
              const float4 l4 = *reinterpret_cast<const float4*>(nlse2 + q);
              const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
              float pe[4];
#pragma unroll
              for (int v = 0; v < 4; ++v)
                pe[v] = (q + v >= qmin && q + v < qmax)
                            ? ex2(fmaf(__uint_as_float(sr[e + v]), a.scale_log2, lv[v]))
                            : 0.f;
              pk[(q >> 1) + 0] = pack_bf16(pe[0], pe[1]);
              pk[(q >> 1) + 1] = pack_bf16(pe[2], pe[3]);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const int q = c * 32 + e;
              const float4 l4 = *reinterpret_cast<const float4*>(nlse2 + q);
              const uint64_t x01 = fma2(f2(__uint_as_float(sr[e + 0]), __uint_as_float(sr[e + 1])),
                                        sc2, f2(l4.x, l4.y));
              const uint64_t x23 = fma2(f2(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])),
                                        sc2, f2(l4.z, l4.w));
              pk[(q >> 1) + 0] = pack_bf16(ex2(f2_lo(x01)), ex2(f2_hi(x01)));
              pk[(q >> 1) + 1] = pack_bf16(ex2(f2_lo(x23)), ex2(f2_hi(x23)));
            }
          }
        }
        tmem_st32(tmem + lane_base + C::kTmemS + grp * 64, pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(L(bars->p_full));
        if (lane == 0 && (warp & 3) == 0) PAIR_TRACE(21, gi);
        // ---- dS^T = P^T ⊙ (dP^T − D): bf16 into TMEM (dK) and into the dQ operand
        if (!(ok = mbar_wait_warp(smem_u32(&bars->dp_full), gi & 1, ab))) break;
        tc_fence_after();
        if (lane == 0 && (warp & 3) == 0) PAIR_TRACE(22, gi);
        // the previous step's dK and dQ products are done with both copies
        if (gi > 0 && !(ok = mbar_wait_warp(smem_u32(&bars->ds_free), (gi - 1) & 1, ab))) break;
        if (lane == 0 && (warp & 3) == 0) PAIR_TRACE(23, gi);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t dr[32];
          tmem_ld32(tmem + lane_base + C::kTmemdP + grp * 64 + c * 32, dr);
          tmem_ld_wait();
#pragma unroll
          for (int ch = 4 * c; ch < 4 * c + 4; ++ch) {
            const int e0 = (ch & 3) * 8;
            const float4 da = *reinterpret_cast<const float4*>(ndsum + ch * 8);
            const float4 db = *reinterpret_cast<const float4*>(ndsum + ch * 8 + 4);
            const uint64_t nd2[4] = {f2(da.x, da.y), f2(da.z, da.w), f2(db.x, db.y), f2(db.z, db.w)};
            uint32_t w[4];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint64_t d2 = add2(f2(__uint_as_float(dr[e0 + 2 * v]),
                                          __uint_as_float(dr[e0 + 2 * v + 1])), nd2[v]);
              w[v] = mul_bf16x2(pk[ch * 4 + v], pack_bf16(f2_lo(d2), f2_hi(d2)));
            }
            if (dsq_remote)
              st_cluster_v4(dsq_dst + sw128_offset(r, ch), w[0], w[1], w[2], w[3]);
            else
              st_shared_v4(dsq_local + sw128_offset(r, ch), w[0], w[1], w[2], w[3]);
            // dS^T over the dP^T columns this group has read (the packed layout of P^T)
            tmem_st4(tmem + lane_base + C::kTmemdP + grp * 64 + ch * 4, w[0], w[1], w[2], w[3]);
          }
          tmem_st_wait();
          if (dsq_remote) fence_proxy_async_cluster(); else fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(L(bars->ds_half[c]));
          if (lane == 0 && (warp & 3) == 0) PAIR_TRACE(24 + c, gi);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->stat_empty[st]));
      }
    }
  } else {
    regs_inc<kRegsDq>();
    // ============================================= dQ + dK / dV epilogue (both CTAs)
    const int t = (warp & 3) * 32 + lane;  // TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int qr = (int)rank * 64 + (t & 63);  // query row of the tile this lane adds
    const int dh = t >> 6;                     // its half of the dQ columns
    const int wt = threadIdx.x - 8 * 32;
    uint32_t gi = 0;
    bool ok = !misaligned;
    // the reductions are paced as in the one-CTA kernel (fast mode only)
    long long t_prev = 0;
    int pace = a.deterministic ? 0 : kRedPaceCap;
    for (uint32_t k = 0; ok; ++k) {
      const uint32_t slot = k & 1;
      if (!(ok = mbar_wait_cluster_warp(smem_u32(&bars->item_full[slot]), (k >> 1) & 1, ab))) break;
      const int item = *static_cast<volatile int*>(&bars->item_slot[slot]);
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(L(bars->item_empty[slot]));
      if (item >= sh.n_items) break;
      const Item it = decode_pair(sh, tb, item);
      int i0, i1;
      pair_band(sh, it, i0, i1);
      const int nk = cdiv(it.Lk, kTile);
      for (int i = i0; i < i1; ++i, ++gi) {
        if (!(ok = mbar_wait_warp(smem_u32(&bars->dq_full), gi & 1, ab))) break;
        tc_fence_after();
        if (lane == 0 && warp == 8) PAIR_TRACE(30, gi);
        {
          const long long t_now = clock64();
          if (t_prev != 0 && !a.deterministic)
            pace = (int)min((long long)kRedPaceCap, (t_now - t_prev) * kRedSpread / (256 * 16));
          t_prev = t_now;
        }
        uint32_t qv[64];
        tmem_ld32(tmem + lane_base + C::kTmemdQ, *reinterpret_cast<uint32_t(*)[32]>(&qv[0]));
        tmem_ld32(tmem + lane_base + C::kTmemdQ + 32, *reinterpret_cast<uint32_t(*)[32]>(&qv[32]));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(L(bars->dq_free));
        if (lane == 0 && warp == 8) PAIR_TRACE(31, gi);
        const int64_t g = (int64_t)(it.tile_base + i) * sh.H + it.head;
        float* acc = a.ws.dq_acc + g * (kTile * 128);
        if (a.deterministic) {
          // pairs add to each tile half in descending pair order: wait for the
          // next pair above in q-tile i's band
          int* sem = a.ws.sem + 2 * g + rank;
          if (wt == 0) {
            const int last = last_kvtile(sh, it, i, nk);
            const int target = (2 * (it.tile + 1) <= last ? it.tile + 2 : 0) + a.sem_bias;
            const uint64_t t0 = globaltimer();
            while (ld_acquire_gpu(sem) != target) {
              if (ab.raised() || ld_acquire_gpu(a.ws.header) != 0 ||
                  globaltimer() - t0 > kWaitLimitNs) {
                ab.raise(kStatusTimeout);
                break;
              }
            }
          }
          named_bar_sync(1, 128);
          if (ab.raised()) { ok = false; break; }
        }
        if (pace > 0) {
          const long long t0 = clock64();
#pragma unroll
          for (int c4 = 0; c4 < 16; ++c4) {
            red_add_v4(acc + ((dh * 16 + c4) * kTile + qr) * 4, __uint_as_float(qv[c4 * 4 + 0]),
                       __uint_as_float(qv[c4 * 4 + 1]), __uint_as_float(qv[c4 * 4 + 2]),
                       __uint_as_float(qv[c4 * 4 + 3]));
            const long long due = t0 + (long long)(c4 + 1) * pace;
            while (clock64() < due) {
            }
          }
        } else {
#pragma unroll
          for (int c4 = 0; c4 < 16; ++c4)
            red_add_v4(acc + ((dh * 16 + c4) * kTile + qr) * 4, __uint_as_float(qv[c4 * 4 + 0]),
                       __uint_as_float(qv[c4 * 4 + 1]), __uint_as_float(qv[c4 * 4 + 2]),
                       __uint_as_float(qv[c4 * 4 + 3]));
        }
        if (lane == 0 && warp == 8) PAIR_TRACE(32, gi);
        if (a.deterministic) {
          named_bar_sync(1, 128);
          if (wt == 0) {
            __threadfence();
            st_release_gpu(a.ws.sem + 2 * g + rank, it.tile + 1);
          }
        }
      }
      if (!ok) break;
      // ---- epilogue: dK = s * acc, dV = acc (thread = key row t of the own tile)
      if (!(ok = mbar_wait_warp(smem_u32(&bars->kv_done), k & 1, ab))) break;
      tc_fence_after();
      const int kidx = (2 * it.tile + (int)rank) * kTile + t;
      const bool key_ok = kidx < it.Lk;
      const int krow = key_row0(sh, it) + kidx;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + C::kTmemdK + c * 32, v);
        tmem_ld_wait();
        if (i0 >= i1) {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        if (key_ok) {
          __nv_bfloat16* dst = a.dk + (int64_t)krow * a.dk_row_stride + (int64_t)it.head * 128 + c * 32;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(v[q4 * 8 + 0]) * a.scale, __uint_as_float(v[q4 * 8 + 1]) * a.scale);
            w.y = pack_bf16(__uint_as_float(v[q4 * 8 + 2]) * a.scale, __uint_as_float(v[q4 * 8 + 3]) * a.scale);
            w.z = pack_bf16(__uint_as_float(v[q4 * 8 + 4]) * a.scale, __uint_as_float(v[q4 * 8 + 5]) * a.scale);
            w.w = pack_bf16(__uint_as_float(v[q4 * 8 + 6]) * a.scale, __uint_as_float(v[q4 * 8 + 7]) * a.scale);
            *reinterpret_cast<uint4*>(dst + q4 * 8) = w;
          }
        }
      }
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + C::kTmemdV + c * 32, v);
        tmem_ld_wait();
        if (i0 >= i1) {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        if (key_ok) {
          __nv_bfloat16* dst = a.dv + (int64_t)krow * a.dv_row_stride + (int64_t)it.head * 128 + c * 32;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(v[q4 * 8 + 0]), __uint_as_float(v[q4 * 8 + 1]));
            w.y = pack_bf16(__uint_as_float(v[q4 * 8 + 2]), __uint_as_float(v[q4 * 8 + 3]));
            w.z = pack_bf16(__uint_as_float(v[q4 * 8 + 4]), __uint_as_float(v[q4 * 8 + 5]));
            w.w = pack_bf16(__uint_as_float(v[q4 * 8 + 6]), __uint_as_float(v[q4 * 8 + 7]));
            *reinterpret_cast<uint4*>(dst + q4 * 8) = w;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(L(bars->acc_free));
    }
  }

  // Both CTAs leave together: no CTA exits while its peer may still write its
  // shared memory or arrive on its barriers, and the pair frees its tensor
  // memory collectively.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
}

}  // namespace

int bwd_pair_smem_bytes() { return Cfg::kSmemBytes; }

#ifdef ATTN_TRACE
unsigned long long* g_pair_trace = nullptr;
#endif

cudaError_t launch_bwd_pair_main(const BwdLaunch& L) {
  PairArgs a;
#ifdef ATTN_TRACE
  a.trace = g_pair_trace;
#endif
  a.sem_bias = L.sem_bias;
  a.dk = reinterpret_cast<__nv_bfloat16*>(L.dk);
  a.dv = reinterpret_cast<__nv_bfloat16*>(L.dv);
  a.dk_row_stride = L.dk_row_stride;
  a.dv_row_stride = L.dv_row_stride;
  a.scale = L.scale;
  a.scale_log2 = L.scale_log2;
  a.deterministic = L.deterministic;
  a.ws = L.ws;
  a.sh = L.sh;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = L.stream;
  cudaError_t e;
  if (L.tables) {
    auto* k = attn_bwd_pair_kernel<VarlenTables>;
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  Cfg::kSmemBytes)) != cudaSuccess)
      return e;
    return cudaLaunchKernelEx(&cfg, k, L.tm_q, L.tm_q64, L.tm_k, L.tm_v, L.tm_do, L.tm_do64, a,
                              *L.tables);
  }
  auto* k = attn_bwd_pair_kernel<NoTables>;
  if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg::kSmemBytes)) != cudaSuccess)
    return e;
  return cudaLaunchKernelEx(&cfg, k, L.tm_q, L.tm_q64, L.tm_k, L.tm_v, L.tm_do, L.tm_do64, a,
                            NoTables{});
}

}  // namespace attn

#ifdef ATTN_TRACE
// Trace builds only: buffer of 2 x 512 x 64 records for the first cluster (null = off).
extern "C" void attn_pair_trace_set(void* buf) {
  attn::g_pair_trace = static_cast<unsigned long long*>(buf);
}
#endif
