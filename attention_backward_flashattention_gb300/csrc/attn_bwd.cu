// attn_bwd.cu — fused attention backward for sm_103a.
//
// The chain rule of "ops(8)：self-attention 的 CUDA 实现及优化 (下) - 深度分析"
// §2.1 (dV = P^T dO, dP = dO V^T, dS = P ⊙ (dP - rowsum(dP ⊙ P)),
// dQ = dS K / sqrt(d_k), dK = dS^T Q / sqrt(d_k)), with the row sum taken as
// D = rowsum(dO ⊙ O) (the simplification §2.3 V7 and §5.3 allude to: the two
// are equal because O = P V), P recomputed from Q, K and the forward's LSE
// instead of being stored, and dQ reduced across key tiles as in
// "深度学习反向传播优化：2-CTA MMA模式与内存访问优化" §3 (global fp32 atomics, or
// a semaphore-ordered deterministic variant, §3.2).
//
// Three launches per call, all on the caller's stream:
//   1. attn_bwd_pre_kernel   (memory-bound) D = rowsum(dO ⊙ O) and LSE·log2(e)
//      into padded per-tile workspace rows; zero the fp32 dQ accumulator, the
//      semaphores, the work counter and the status word.
//   2. attn_bwd_main_kernel  one CTA per SM, persistent; each work item is one
//      128-key tile of one (sequence, head).  K_j and V_j stay in shared
//      memory, dK_j and dV_j accumulate in tensor memory, and the loop walks
//      the query tiles i:
//         S^T  = K_j Q_i^T                    (MMA, TMEM)
//         P^T  = exp2(S^T·s·log2e − LSE2_i)   (compute warps)
//         dP^T = V_j dO_i^T                   (MMA, TMEM)
//         dV_j += P^T dO_i                    (MMA)
//         dS^T = P^T ⊙ (dP^T − D_i)           (compute warps, bf16 to smem;
//                                               dP^T − D rounded to bf16 first)
//         dK_j += dS^T Q_i                    (MMA)
//         dQ_i  = dS K_j                      (MMA, TMEM) -> fp32 reduction
//      Working transposed (keys on TMEM lanes) makes P^T and dS^T the natural
//      A operands of the dV and dK products; dQ reads the same dS^T tile
//      through an MN-major descriptor.
//   3. attn_bwd_convert_kernel  dQ = bf16(s · dQacc) into the caller's layout.
//
// Roles in the main kernel (512 threads):
//   warps 0-3, 4-7  P / dS warpgroups; thread = key row (TMEM lane); group g
//                   handles query columns [64g, 64g+64) of S^T and dP^T
//   warps 8-11      dQ warpgroup: drains dQ_i from TMEM (thread = query row) and
//                   adds it to the fp32 accumulator (spread over the q-tile
//                   step in fast mode, ordered in deterministic mode); at the
//                   end of an item stores dK and dV
//   warp 12         TMA producer and work-item claimer
//   warp 13         MMA issuer, tensor-memory owner (warps 14-15 idle)
// MMA order per q-tile: ... dV_i, S_{i+1}, dK_i (first half), dQ_i, dK_i
// (second half), dP_{i+1}, dV_{i+1} ... so that P_{i+1} is computed while dK_i
// and dQ_i run (S and dP have their own TMEM columns for d <= 128), and the
// dQ drain overlaps the second half of dK_i.
// The q-tiles of an item are those of its band (causal, window); the kernels
// built for a block mask (kMask) walk only the ones the mask keeps.  In
// deterministic mode each dQ tile's contributions arrive in descending kv-tile
// order: a per-(q-tile, head) word holds 1 + the kv tile that added last.
// For d = 128 without block masks or left window edges the main kernel can
// instead run on CTA pairs (attn_bwd_pair.cu); the preprocess and the dQ
// conversion are the same.
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kPanelBytes = kTile * 128;
constexpr int kMaxSmem = 232448;
// 16 warps: P/dS warpgroups 0 and 1, dQ warpgroup 2, and warpgroup 3 whose
// warp 12 is the TMA producer and warp 13 the MMA issuer (14, 15 idle).
constexpr int kMainThreads = 512;
constexpr int kTmaWarp = 12;
constexpr int kMmaWarp = 13;
// Registers per thread after the split.  Launched with 512 x 128 = 65536;
// the P/dS and control warpgroups give registers back, the dQ warpgroup (which
// holds a whole dQ row of the tile) takes them.  Per warpgroup:
//   P/dS x2, control, dQ    sum <= 4 x 128
template <int DQK>
struct RegSplit {
  static constexpr uint32_t kLaunch = 128;
  static constexpr uint32_t kCompute = DQK > 128 ? 88 : (DQK > 64 ? 104 : 112);
  // the MMA issuer (control warpgroup) holds every staged descriptor base:
  // 136 at d <= 128 keeps it from spilling (raised with setmaxnreg.inc)
  static constexpr uint32_t kCtl = DQK > 128 ? 128 : 136;
  static constexpr uint32_t kDq = 4 * kLaunch - 2 * kCompute - kCtl;  // 152, 168, 208
  static_assert(2 * kCompute + kCtl + kDq <= 4 * kLaunch, "register split");
  static_assert(kCompute % 8 == 0 && kCtl % 8 == 0 && kDq % 8 == 0 && kDq <= 256, "setmaxnreg");
  // the kernel lowers the P/dS and control warpgroups (setmaxnreg.dec) and
  // raises the dQ warpgroup (setmaxnreg.inc) from the launch count
  static_assert(kCompute <= kLaunch && kDq >= kLaunch, "setmaxnreg direction");
};
constexpr float kLog2e = 1.4426950408889634f;

// Optional phase tracing of CTA 0 (compiled in only with -DATTN_TRACE): the
// recording threads keep the low 32 bits of clock64 per (event, step) for the
// q-tile steps [kTraceFrom, kTraceFrom + kTraceSteps) in 512 bytes of shared
// memory past the kernel's own, and the CTA copies the 128 words to the
// caller's buffer (as 64-bit values) at exit.  Keeping the records on chip
// matters: a global store per event would queue behind the dQ reductions and
// delay the recording thread itself.
#ifdef ATTN_TRACE
#ifndef ATTN_TRACE_FROM
#define ATTN_TRACE_FROM 40
#endif
constexpr uint32_t kTraceFrom = ATTN_TRACE_FROM;
constexpr uint32_t kTraceSteps = 4;
constexpr int kTraceSmem = 512;
// record slot of an event: MMA issuer 0-6, P/dS warpgroup 0 7-12, group 1
// 13-18, dQ warpgroup 19-21, producer 22-25, load observers 26-27
__device__ __forceinline__ int trace_index(int ev, int warp) {
  switch (ev) {
    case 10: return 0;
    case 11: return 1;
    case 12: return 2;
    case 15: return 3;
    case 16: return 4;
    case 13: return 5;
    case 14: return 6;
    case 20: case 21: case 22: case 25: case 23: case 24: {
      const int b = ev == 20 ? 0 : ev == 21 ? 1 : ev == 22 ? 2 : ev == 25 ? 3 : ev == 23 ? 4 : 5;
      return 7 + (warp >= 4 ? 6 : 0) + b;
    }
    case 30: return 19;
    case 31: return 20;
    case 32: return 21;
    case 41: return 22;
    case 42: return 23;
    case 40: return 24;
    case 43: return 25;
    case 44: return 26;
    case 45: return 27;
    default: return -1;
  }
}
#define ATTN_TRACE_DECL uint32_t* const tr_smem = reinterpret_cast<uint32_t*>(smem + C::kSmemBytes)
#define ATTN_TRACE_EV(ev, step)                                                             \
  do {                                                                                      \
    const uint32_t s_ = (uint32_t)(step) - kTraceFrom;                                      \
    if (a.trace != nullptr && blockIdx.x == 0 && s_ < kTraceSteps) {                        \
      const int ix_ = trace_index(ev, warp);                                                \
      if (ix_ >= 0) tr_smem[ix_ * kTraceSteps + s_] = (uint32_t)clock64();                  \
    }                                                                                       \
  } while (0)
#define ATTN_TRACE_FLUSH                                                                    \
  do {                                                                                      \
    __syncthreads();                                                                        \
    if (a.trace != nullptr && blockIdx.x == 0 && threadIdx.x < kTraceSmem / 4)              \
      a.trace[threadIdx.x] = tr_smem[threadIdx.x];                                          \
  } while (0)
#else
constexpr int kTraceSmem = 0;
#define ATTN_TRACE_DECL \
  do {                  \
  } while (0)
#define ATTN_TRACE_EV(ev, step) \
  do {                          \
  } while (0)
#define ATTN_TRACE_FLUSH \
  do {                   \
  } while (0)
#endif

// ---------------------------------------------------------------------------
// Sequence helpers (shared by the memory-bound kernels)
// ---------------------------------------------------------------------------
template <typename Tables>
struct SeqOf;

template <>
struct SeqOf<NoTables> {
  // token row -> (sequence, position); sequences have length Tq
  __device__ static void locate(const SeqShape& sh, const NoTables&, int row, int& s, int& t) {
    s = row / sh.Tq;
    t = row - s * sh.Tq;
  }
  __device__ static int length(const SeqShape& sh, const NoTables&, int) { return sh.Tq; }
  __device__ static int row0(const SeqShape& sh, const NoTables&, int s) { return s * sh.Tq; }
  __device__ static int tile_start(const SeqShape& sh, const NoTables&, int s) {
    return s * sh.nq_tiles;
  }
  // workspace q-tile g -> (sequence, tile within it)
  __device__ static void tile_of(const SeqShape& sh, const NoTables&, int g, int& s, int& i) {
    s = g / sh.nq_tiles;
    i = g - s * sh.nq_tiles;
  }
};

template <>
struct SeqOf<VarlenTables> {
  __device__ static void locate(const SeqShape& sh, const VarlenTables& tb, int row, int& s,
                                int& t) {
    int lo = 0, hi = sh.nseq - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tb.cu[mid] <= row) lo = mid; else hi = mid - 1;
    }
    s = lo;
    t = row - tb.cu[lo];
  }
  __device__ static int length(const SeqShape&, const VarlenTables& tb, int s) {
    return tb.cu[s + 1] - tb.cu[s];
  }
  __device__ static int row0(const SeqShape&, const VarlenTables& tb, int s) { return tb.cu[s]; }
  __device__ static int tile_start(const SeqShape&, const VarlenTables& tb, int s) {
    return tb.tile_start[s];
  }
  __device__ static void tile_of(const SeqShape& sh, const VarlenTables& tb, int g, int& s,
                                 int& i) {
    int lo = 0, hi = sh.nseq - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tb.tile_start[mid] <= g) lo = mid; else hi = mid - 1;
    }
    s = lo;
    i = g - tb.tile_start[lo];
  }
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ---------------------------------------------------------------------------
// 1. preprocess
// ---------------------------------------------------------------------------
template <int DQK, int DV, typename Tables>
__global__ void __launch_bounds__(256)
    attn_bwd_pre_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                        const float* __restrict__ lse, const int64_t o_row_stride,
                        const int64_t do_row_stride, const int64_t lse_head_stride,
                        const int64_t lse_seq_stride, const int total_rows, const int n_qtiles,
                        BwdWorkspace ws, const SeqShape sh, const __grid_constant__ Tables tb) {
  using S = SeqOf<Tables>;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  const int H = sh.H;
  if (tid == 0) {
    ws.header[0] = 0;  // status
    ws.header[1] = 0;  // work-item counter
  }
  for (int64_t i = tid; i < (int64_t)n_qtiles * H * 2; i += nthreads) ws.sem[i] = 0;

  // D and LSE*log2(e) for every real (token, head) row: DV/8 threads per row,
  // 16 bytes each, consecutive threads along the row (coalesced).
  constexpr int kTPR = DV / 8;  // threads per row: 8 or 16 (a power of two)
  const int64_t n_work = (int64_t)total_rows * H * kTPR;
  // round the loop bound up so that every lane of a row group iterates together
  const int64_t n_loop = (n_work + nthreads - 1) / nthreads * nthreads;
  for (int64_t w = tid; w < n_loop; w += nthreads) {
    float part = 0.f;
    int row = 0, h = 0, ch = 0;
    const bool live = w < n_work;
    if (live) {
      const int64_t rh = w / kTPR;
      ch = (int)(w - rh * kTPR);
      row = (int)(rh / H);
      h = (int)(rh - (int64_t)row * H);
      const uint4 a = *reinterpret_cast<const uint4*>(o + (int64_t)row * o_row_stride + (int64_t)h * DV + ch * 8);
      const uint4 b = *reinterpret_cast<const uint4*>(dout + (int64_t)row * do_row_stride + (int64_t)h * DV + ch * 8);
      part = bf16_lo(a.x) * bf16_lo(b.x) + bf16_hi(a.x) * bf16_hi(b.x) +
             bf16_lo(a.y) * bf16_lo(b.y) + bf16_hi(a.y) * bf16_hi(b.y) +
             bf16_lo(a.z) * bf16_lo(b.z) + bf16_hi(a.z) * bf16_hi(b.z) +
             bf16_lo(a.w) * bf16_lo(b.w) + bf16_hi(a.w) * bf16_hi(b.w);
    }
#pragma unroll
    for (int off = kTPR / 2; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if (live && ch == 0) {
      int s, t;
      S::locate(sh, tb, row, s, t);
      const int64_t lbase = sh.varlen ? (int64_t)S::row0(sh, tb, s) : (int64_t)s * lse_seq_stride;
      const float l = lse[(int64_t)h * lse_head_stride + lbase + t];
      const int64_t g = ((int64_t)(S::tile_start(sh, tb, s) + t / kTile) * H + h) * kTile + (t % kTile);
      // stored negated: the main kernel adds them (packed FP32 pairs have no
      // negated-operand form)
      ws.ndsum[g] = -part;
      // a row that saw no key (LSE = -inf, a block mask) keeps P = 0
      ws.nlse2[g] = l == -INFINITY ? -INFINITY : -l * kLog2e;
    }
  }
  // padding rows of each sequence's last q-tile: P must come out as zero there
  for (int64_t w = tid; w < (int64_t)sh.nseq * H * kTile; w += nthreads) {
    const int s = (int)(w / (H * kTile));
    const int rem = (int)(w - (int64_t)s * H * kTile);
    const int h = rem / kTile, r = rem % kTile;
    const int L = S::length(sh, tb, s);
    const int nt = cdiv(L, kTile);
    if (nt == 0 || (nt - 1) * kTile + r < L) continue;
    const int64_t g = ((int64_t)(S::tile_start(sh, tb, s) + nt - 1) * H + h) * kTile + r;
    ws.ndsum[g] = 0.f;
    ws.nlse2[g] = -INFINITY;
  }
  // zero the dQ accumulator
  float4* acc = reinterpret_cast<float4*>(ws.dq_acc);
  const int64_t n4 = (int64_t)n_qtiles * H * kTile * DQK / 4;
  for (int64_t i = tid; i < n4; i += nthreads) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ---------------------------------------------------------------------------
// 2. main kernel
// ---------------------------------------------------------------------------
template <int DQK, int DV>
struct BwdCfg {
  static constexpr int kQPanels = DQK / 64;
  static constexpr int kVPanels = DV / 64;
  static constexpr int kKBytes = kQPanels * kPanelBytes;
  static constexpr int kVBytes = kVPanels * kPanelBytes;
  static constexpr int kQBytes = kQPanels * kPanelBytes;
  static constexpr int kdOBytes = kVPanels * kPanelBytes;
  static constexpr int kStatBytes = 2 * kTile * 4;  // -LSE2 and -D of one q-tile
  static constexpr int kStageBytes = kQBytes + kdOBytes + kStatBytes;
  static constexpr int kdSBytes = 2 * kPanelBytes;
  static constexpr int kBarBytes = 512;
  // the dynamic shared memory window starts 1024-byte aligned (checked at run time)
  static constexpr int kFixed = kKBytes + kVBytes + kdSBytes + kBarBytes;
  static constexpr int kStagesFit = (kMaxSmem - kFixed) / kStageBytes;
  static constexpr int kStages = kStagesFit > 4 ? 4 : kStagesFit;  // barrier arrays hold 4
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kKBytes;
  static constexpr int kOffdS = kOffV + kVBytes;
  static constexpr int kOffStage = kOffdS + kdSBytes;  // panels of every stage first
  static constexpr int kOffStat = kOffStage + kStages * (kQBytes + kdOBytes);
  static constexpr int kOffBar = kOffStat + kStages * kStatBytes;
  static constexpr int kSmemBytes = kOffBar + kBarBytes;
  static_assert(kStages >= 1, "shared memory too small");
  static_assert(kSmemBytes <= kMaxSmem, "shared memory budget");
  static_assert(kBarBytes >= 256, "barrier block");
  // Tensor memory plan (columns).  P^T (bf16, two per column) overwrites the
  // S^T columns each warpgroup has already read: queries 0-63 at [0, 32),
  // queries 64-127 at [64, 96).
  static constexpr bool kSharedSdP = (DQK == 192);  // S and dP take turns in one region
  static constexpr bool kDqOnDp = (DQK == 128);     // dQ reuses the dP region
  static constexpr uint32_t kTmemS = 0;
  static constexpr uint32_t kTmemdP = kSharedSdP ? 0 : 128;
  static constexpr uint32_t kTmemdV = kSharedSdP ? 192 : 256;
  static constexpr uint32_t kTmemdK = kTmemdV + DV;
  static constexpr uint32_t kTmemdQ = kSharedSdP ? 0 : (kDqOnDp ? 128 : kTmemdK + DQK);
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kTmemdK + DQK <= kTmemCols, "tensor memory budget (dK)");
  static_assert(kTmemdQ + DQK <= kTmemCols, "tensor memory budget (dQ)");
};

// Epilogue helpers: N accumulator columns of this thread's TMEM lane, scaled,
// as bf16 pairs (zeros when nothing was accumulated), and their store as one
// row of the caller's layout (32-byte stores when st32).
template <int N>
__device__ __forceinline__ void epi_read(uint32_t taddr, float sc, bool zero,
                                         uint32_t (&pk)[N / 2]) {
  if (zero) {
#pragma unroll
    for (int e = 0; e < N / 2; ++e) pk[e] = 0u;
    return;
  }
#pragma unroll
  for (int c = 0; c < N / 32; ++c) {
    uint32_t v[32];
    tmem_ld32(taddr + c * 32, v);
    tmem_ld_wait();
#pragma unroll
    for (int e = 0; e < 16; ++e)
      pk[c * 16 + e] = pack_bf16(__uint_as_float(v[2 * e]) * sc, __uint_as_float(v[2 * e + 1]) * sc);
  }
}
template <int N>
__device__ __forceinline__ void epi_store(__nv_bfloat16* dst, int st32, const uint32_t (&pk)[N / 2]) {
  if (st32) {
#pragma unroll
    for (int j = 0; j < N / 16; ++j)
      st_global_v8(dst + j * 16, pk[8 * j + 0], pk[8 * j + 1], pk[8 * j + 2], pk[8 * j + 3],
                   pk[8 * j + 4], pk[8 * j + 5], pk[8 * j + 6], pk[8 * j + 7]);
  } else {
#pragma unroll
    for (int j = 0; j < N / 8; ++j)
      *reinterpret_cast<uint4*>(dst + j * 8) =
          make_uint4(pk[4 * j + 0], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
  }
}

// TMEM column of the packed P^T operand for MMA K-step kk (16 queries).
__device__ __forceinline__ uint32_t p_col(int kk) { return (kk >> 2) * 64 + (kk & 3) * 8; }

// The block mask's column of the item's kv tile (entry of q-tile i at
// col[i * blk_nk]); null in the kernels built without block-mask support
// (kMask = false), where every walk below reduces to i, i + 1, ...
template <bool kMask>
__device__ __forceinline__ const uint8_t* mask_col(const SeqShape& sh, const Item& it) {
  if constexpr (!kMask) return nullptr;
  return sh.blk + it.seq * sh.blk_bstride + it.head * sh.blk_hstride + it.tile;
}

// The first q-tile >= i, below i1, whose pair with the item's kv tile the
// block mask keeps (i1 when there is none).  Every role of the main kernel
// walks the same q-tiles with it.
__device__ __forceinline__ int next_qtile(const SeqShape& sh, const uint8_t* col, int i, int i1) {
  if (col != nullptr)
    while (i < i1 && __ldg(col + (int64_t)i * sh.blk_nk) == 0) ++i;
  return i;
}

constexpr int kMaxStages = 4;

struct BwdBars {
  uint64_t item_full[2], item_empty[2];
  uint64_t kv_full, kv_done;
  uint64_t accv_free, acck_free;  // the epilogue has read the dV / dK accumulator
  uint64_t q_full[kMaxStages], q_empty[kMaxStages];    // Q panels + LSE2 + D of a q-tile
  uint64_t do_full[kMaxStages], do_empty[kMaxStages];  // dO panels
  uint64_t s_full, p_full, dp_full, dq_full, dq_free;
  uint64_t ds_half[2];  // dS^T columns 0-31 / 64-95 (half 0) and 32-63 / 96-127 (half 1)
  uint64_t drain;
  int item_slot[2];
  int q_last[kMaxStages];  // 1: the stage's q-tile is its item's last (written with q_full)
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(BwdBars) <= 512, "barrier block size");

struct MainArgs {
  int sem_bias;  // 0; a test sets it so that the ordered dQ wait can never succeed
  int st32;      // dK and dV rows are 32-byte aligned: 32-byte stores
#ifdef ATTN_TRACE
  unsigned long long* trace;  // kMainThreads x kTraceCap records
#endif
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int64_t dk_row_stride, dv_row_stride;
  float scale, scale_log2;
  int deterministic;
  BwdWorkspace ws;
  SeqShape sh;
};

// kMask: built with block-mask support (sh.blk non-null); the kernels without
// it carry none of the mask's walks.
template <int DQK, int DV, typename Tables, bool kMask>
__global__ void __launch_bounds__(kMainThreads, 1)
    attn_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_do, const MainArgs a,
                         const __grid_constant__ Tables tb) {
  using C = BwdCfg<DQK, DV>;
  static_assert(C::kSmemBytes + kTraceSmem <= kMaxSmem, "shared memory budget (trace)");
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // the swizzled panels need a 1024-byte aligned window
    if (threadIdx.x == 0) atomicCAS(a.ws.header, 0, kStatusInternal);
    return;
  }
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::kOffBar);
  const uint32_t sK = smem_u32(smem + C::kOffK);
  const uint32_t sV = smem_u32(smem + C::kOffV);
  const uint32_t sdS = smem_u32(smem + C::kOffdS);
  const uint32_t sStage = smem_u32(smem + C::kOffStage);
  const float* stat_f = reinterpret_cast<const float*>(smem + C::kOffStat);
  const uint32_t sStat = smem_u32(smem + C::kOffStat);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const SeqShape& sh = a.sh;
  Abort ab{&bars->abort_flag, a.ws.header};
  ATTN_TRACE_DECL;
  auto sQ_of = [&](uint32_t st) { return sStage + st * (C::kQBytes + C::kdOBytes); };
  auto sdO_of = [&](uint32_t st) { return sStage + st * (C::kQBytes + C::kdOBytes) + C::kQBytes; };

  if (threadIdx.x == 0) {
#ifdef ATTN_TRACE
    for (int t = 0; t < kTraceSmem / 4; ++t) tr_smem[t] = 0;
#endif
    bars->abort_flag = 0;
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_u32(&bars->item_full[k]), 1);
      mbar_init(smem_u32(&bars->item_empty[k]), 1 + 8 + 4);  // MMA + compute + dQ warps
    }
    mbar_init(smem_u32(&bars->kv_full), 1);
    mbar_init(smem_u32(&bars->kv_done), 1);
    mbar_init(smem_u32(&bars->accv_free), 4);
    mbar_init(smem_u32(&bars->acck_free), 4);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&bars->q_full[s]), 1);
      mbar_init(smem_u32(&bars->q_empty[s]), 1);
      mbar_init(smem_u32(&bars->do_full[s]), 1);
      mbar_init(smem_u32(&bars->do_empty[s]), 1);
    }
    mbar_init(smem_u32(&bars->s_full), 1);
    mbar_init(smem_u32(&bars->p_full), 8);
    mbar_init(smem_u32(&bars->dp_full), 1);
    mbar_init(smem_u32(&bars->ds_half[0]), 8);
    mbar_init(smem_u32(&bars->ds_half[1]), 8);
    mbar_init(smem_u32(&bars->dq_full), 1);
    mbar_init(smem_u32(&bars->dq_free), 4);
    mbar_init(smem_u32(&bars->drain), 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp >= 12) {
   if constexpr (RegSplit<DQK>::kCtl > RegSplit<DQK>::kLaunch) regs_inc<RegSplit<DQK>::kCtl>();
   else regs_dec<RegSplit<DQK>::kCtl>();
   if (warp == kTmaWarp && lane == 0) {
    // ================================================= producer / claimer
    {
      uint32_t q_it = 0, kq = 0, q_issued = 0, do_issued = 0;
      bool ok = true, kv_issued = false;
      for (uint32_t k = 0;; ++k) {
        const uint32_t slot = k & 1;
        if (!(ok = mbar_wait(smem_u32(&bars->item_empty[slot]), ((k >> 1) & 1) ^ 1, ab))) break;
        // stop handing out work once any CTA has failed
        const int item = ld_acquire_gpu(a.ws.header) != 0 ? sh.n_items
                                                           : atomicAdd(&a.ws.header[1], 1);
        bars->item_slot[slot] = item;
        mbar_arrive(smem_u32(&bars->item_full[slot]));
        if (item >= sh.n_items) break;
        const Item it = decode_item(sh, tb, item, false);
        const int krow = key_row0(sh, it) + it.tile * kTile;
        // K_j, V_j once per item (the previous item's MMAs must be done with them)
        if (!(ok = mbar_wait(smem_u32(&bars->kv_done), (k & 1) ^ 1, ab))) break;
        const uint32_t kvb = smem_u32(&bars->kv_full);
        mbar_arrive_expect_tx(kvb, C::kKBytes + C::kVBytes);
        kv_issued = true;
        kq = k;
        for (int p = 0; p < C::kQPanels; ++p)
          tma_load_3d(sK + p * kPanelBytes, &tm_k, kvb, p * 64, it.head, krow);
        for (int p = 0; p < C::kVPanels; ++p)
          tma_load_3d(sV + p * kPanelBytes, &tm_v, kvb, p * 64, it.head, krow);
        const int nq = cdiv(it.Lq, kTile);
        const int i0 = first_qtile(sh, it, it.tile), i1 = last_qtile(sh, it, it.tile, nq) + 1;
        const uint8_t* col = mask_col<kMask>(sh, it);
        for (int i = next_qtile(sh, col, i0, i1), inext; i < i1; i = inext, ++q_it) {
          inext = next_qtile(sh, col, i + 1, i1);
          const uint32_t st = q_it % C::kStages;
          const uint32_t par = ((q_it / C::kStages) & 1) ^ 1;
          const int qrow = it.row0 + i * kTile;
          const int64_t g = (int64_t)(it.tile_base + i) * sh.H + it.head;
          // Q (with the row statistics) and dO of the q-tile.  dO's stage is
          // released by dV, early in a step, and Q's by dK, late in it: at
          // d <= 128 dO goes first, so that it lands a step ahead of dP; at
          // d = 192 (S and dP share their columns) Q first measured faster.
          auto load_q = [&]() -> bool {
            if (!mbar_wait(smem_u32(&bars->q_empty[st]), par, ab)) return false;
            ATTN_TRACE_EV(40, q_it);
            // under a block mask the MMA issuer learns from this flag whether
            // another q-tile follows (published by the arrive below, read
            // after its wait on q_full)
            if constexpr (kMask) bars->q_last[st] = inext >= i1 ? 1 : 0;
            const uint32_t qb = smem_u32(&bars->q_full[st]);
            mbar_arrive_expect_tx(qb, C::kQBytes + C::kStatBytes);
            for (int p = 0; p < C::kQPanels; ++p)
              tma_load_3d(sQ_of(st) + p * kPanelBytes, &tm_q, qb, p * 64, it.head, qrow);
            bulk_load(sStat + st * C::kStatBytes, a.ws.nlse2 + g * kTile, kTile * 4, qb);
            bulk_load(sStat + st * C::kStatBytes + kTile * 4, a.ws.ndsum + g * kTile, kTile * 4, qb);
            q_issued = q_it + 1;
            ATTN_TRACE_EV(43, q_it);
            return true;
          };
          auto load_do = [&]() -> bool {
            if (!mbar_wait(smem_u32(&bars->do_empty[st]), par, ab)) return false;
            ATTN_TRACE_EV(41, q_it);
            const uint32_t db = smem_u32(&bars->do_full[st]);
            mbar_arrive_expect_tx(db, C::kdOBytes);
            for (int p = 0; p < C::kVPanels; ++p)
              tma_load_3d(sdO_of(st) + p * kPanelBytes, &tm_do, db, p * 64, it.head, qrow);
            do_issued = q_it + 1;
            ATTN_TRACE_EV(42, q_it);
            return true;
          };
          if constexpr (C::kSharedSdP) {
            if (!(ok = load_q() && load_do())) break;
          } else {
            if (!(ok = load_do() && load_q())) break;
          }
        }
        if (!ok) break;
      }
      if (!ok) {
        // let every copy already issued land before the CTA's memory is released
        if (kv_issued) mbar_wait_drain(smem_u32(&bars->kv_full), kq & 1);
        for (uint32_t t = q_issued > (uint32_t)C::kStages ? q_issued - C::kStages : 0; t < q_issued; ++t)
          mbar_wait_drain(smem_u32(&bars->q_full[t % C::kStages]), (t / C::kStages) & 1);
        for (uint32_t t = do_issued > (uint32_t)C::kStages ? do_issued - C::kStages : 0; t < do_issued; ++t)
          mbar_wait_drain(smem_u32(&bars->do_full[t % C::kStages]), (t / C::kStages) & 1);
      }
    }
   } else if (warp == kMmaWarp && lane == 0) {
    // ================================================= MMA issuer
    {
      constexpr uint32_t idS = idesc_bf16(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t idV = idesc_bf16(128, DV, false, true);    // dV += P^T dO
      constexpr uint32_t idK = idesc_bf16(128, DQK, false, true);   // dK += dS^T Q
      constexpr uint32_t idQ = idesc_bf16(128, DQK, true, true);    // dQ = dS K
      uint32_t q_it = 0, gi = 0;
      bool ok = true;
      auto W = [&](uint64_t& bar, uint32_t parity) -> bool {
        if (!mbar_wait(smem_u32(&bar), parity, ab)) return false;
        tc_fence_after();
        return true;
      };
      // Descriptor bases: fixed buffers once, staged buffers per call; each
      // MMA then only adds a constant (see kmajor_step / mnmajor_step).
      const uint64_t bK_k = kmajor_base(sK), bK_mn = mnmajor_base(sK, 128);
      const uint64_t bV_k = kmajor_base(sV);
      const uint64_t bdS_k = kmajor_base(sdS), bdS_mn = mnmajor_base(sdS, 128);
      const uint32_t tS = tmem + C::kTmemS, tdP = tmem + C::kTmemdP;
      const uint32_t tdV = tmem + C::kTmemdV, tdK = tmem + C::kTmemdK, tdQ = tmem + C::kTmemdQ;
      auto mma_S = [&](uint32_t st) {
        const uint64_t bQ = kmajor_base(sQ_of(st));
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk)
          mma_bf16(tS, bK_k + kmajor_step(kk, 128), bQ + kmajor_step(kk, 128), idS,
                   kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(&bars->s_full));
      };
      auto mma_dP = [&](uint32_t st) {
        const uint64_t bdO = kmajor_base(sdO_of(st));
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk)
          mma_bf16(tdP, bV_k + kmajor_step(kk, 128), bdO + kmajor_step(kk, 128), idS,
                   kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(&bars->dp_full));
      };
      auto mma_dV = [&](uint32_t st, bool first) {
        const uint64_t bdO = mnmajor_base(sdO_of(st), 128);
        mma_bf16_ts(tdV, tS + p_col(0), bdO, idV, first ? 0u : 1u);
#pragma unroll
        for (int kk = 1; kk < kTile / 16; ++kk)
          mma_bf16_ts(tdV, tS + p_col(kk), bdO + mnmajor_step(kk), idV, 1u);
      };
      // dK += dS^T Q in two halves: K steps {0,1,4,5} read the dS^T columns the
      // compute warps finish first, {2,3,6,7} the rest
      auto mma_dK = [&](uint32_t st, bool first, int half) {
        const uint64_t bQ = mnmajor_base(sQ_of(st), 128);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int kk = (u & 1) + (u >> 1) * 4 + half * 2;
          mma_bf16(tdK, bdS_k + kmajor_step(kk, 128), bQ + mnmajor_step(kk), idK,
                   (first && half == 0 && u == 0) ? 0u : 1u);
        }
      };
      auto mma_dQ = [&]() {
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_bf16(tdQ, bdS_mn + mnmajor_step(kk), bK_mn + mnmajor_step(kk), idQ,
                   kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(&bars->dq_full));
      };
      for (uint32_t k = 0; ok; ++k) {
        const uint32_t slot = k & 1;
        if (!(ok = mbar_wait(smem_u32(&bars->item_full[slot]), (k >> 1) & 1, ab))) break;
        const int item = bars->item_slot[slot];
        if (item >= sh.n_items) break;
        const Item it = decode_item(sh, tb, item, false);
        const int nq = cdiv(it.Lq, kTile);
        const int i0 = first_qtile(sh, it, it.tile), i1 = last_qtile(sh, it, it.tile, nq) + 1;
        // Without a block mask the q-tiles are i0 .. i1-1.  With one, the
        // producer's per-stage flag says whether a stage's q-tile is the
        // item's last (read right after the stage's q_full wait, one step
        // before it is needed, so that the load's latency is hidden).
        const bool none = next_qtile(sh, mask_col<kMask>(sh, it), i0, i1) >= i1;
        auto last_flag = [&](uint32_t st) {
          return *static_cast<volatile int*>(&bars->q_last[st]) != 0;
        };
        if (!(ok = W(bars->kv_full, k & 1))) break;
        if (none) {
          // dK/dV accumulators of the previous item read out by the epilogue
          if (!(ok = W(bars->accv_free, (k & 1) ^ 1) && W(bars->acck_free, (k & 1) ^ 1))) break;
        }
        if (none) {
          // no query sees this kv tile (a local window or a block mask): the
          // epilogue writes zeros; nothing to compute
        } else if (!C::kSharedSdP) {
          // S and dP of the first q-tile; afterwards S_{i+1} is issued right
          // after dV_i so that P_{i+1} is computed while dK_i and dQ_i run.
          const uint32_t st0 = q_it % C::kStages;
          if (!(ok = W(bars->q_full[st0], (q_it / C::kStages) & 1))) break;
          bool more_next = kMask ? !last_flag(st0) : true;  // kMask: another q-tile follows
          mma_S(st0);
          if (C::kDqOnDp && gi > 0 && !(ok = W(bars->dq_free, (gi - 1) & 1))) break;
          if (!(ok = W(bars->do_full[st0], (q_it / C::kStages) & 1))) break;
          mma_dP(st0);
          // the previous item's dK/dV accumulators must be read out by its
          // epilogue before this item's first dV; waiting here, after the first
          // S and dP, lets the epilogue overlap them (at d <= 128 the epilogue
          // releases both accumulators at once)
          if (!(ok = W(bars->accv_free, (k & 1) ^ 1))) break;
          bool go = true;  // kMask: the previous q-tile was not the item's last
          for (int i = i0; kMask ? go : i < i1; ++i, ++q_it, ++gi) {
            const uint32_t st = q_it % C::kStages;
            const uint32_t st1 = (q_it + 1) % C::kStages;
            const uint32_t par1 = ((q_it + 1) / C::kStages) & 1;
            const bool first = (i == i0), more = kMask ? more_next : i + 1 < i1;
            go = more;
            if (!(ok = W(bars->p_full, gi & 1))) break;
            ATTN_TRACE_EV(10, gi);
            mma_dV(st, first);
            mma_commit(smem_u32(&bars->do_empty[st]));
            if (more) {
              if (!(ok = W(bars->q_full[st1], par1))) break;
              ATTN_TRACE_EV(11, gi);
              if constexpr (kMask) more_next = !last_flag(st1);
              mma_S(st1);
            }
            if (!(ok = W(bars->ds_half[0], gi & 1))) break;
            ATTN_TRACE_EV(12, gi);
            mma_dK(st, first, 0);
            if (!(ok = W(bars->ds_half[1], gi & 1))) break;
            ATTN_TRACE_EV(15, gi);
            // dQ before the second half of dK: the dQ warpgroup starts draining
            // (and dP_{i+1} can follow) while dK finishes
            if (!C::kDqOnDp && gi > 0 && !(ok = W(bars->dq_free, (gi - 1) & 1))) break;
            mma_dQ();
            ATTN_TRACE_EV(16, gi);
            mma_dK(st, first, 1);
            mma_commit(smem_u32(&bars->q_empty[st]));
            if (more) {
              if (C::kDqOnDp && !(ok = W(bars->dq_free, gi & 1))) break;
              ATTN_TRACE_EV(13, gi);
              if (!(ok = W(bars->do_full[st1], par1))) break;
              ATTN_TRACE_EV(14, gi);
              mma_dP(st1);
            }
          }
        } else {
          // S and dP share columns, and dQ covers them: one q-tile at a time
          bool go = true;  // kMask: the previous q-tile was not the item's last
          for (int i = i0; kMask ? go : i < i1; ++i, ++q_it, ++gi) {
            const uint32_t st = q_it % C::kStages;
            const uint32_t par = (q_it / C::kStages) & 1;
            const bool first = (i == i0);
            if (!(ok = W(bars->q_full[st], par))) break;
            if constexpr (kMask) go = !last_flag(st);
            if (gi > 0 && !(ok = W(bars->dq_free, (gi - 1) & 1))) break;
            mma_S(st);
            if (!(ok = W(bars->p_full, gi & 1))) break;
            if (!(ok = W(bars->do_full[st], par))) break;
            // the previous item's dK/dV accumulators read out by its epilogue,
            // which overlaps this item's first S and P
            if (first && !(ok = W(bars->accv_free, (k & 1) ^ 1) && W(bars->acck_free, (k & 1) ^ 1)))
              break;
            mma_dV(st, first);
            mma_dP(st);  // overwrites the S/P columns after dV has read P
            mma_commit(smem_u32(&bars->do_empty[st]));
            if (!(ok = W(bars->ds_half[0], gi & 1))) break;
            mma_dK(st, first, 0);
            if (!(ok = W(bars->ds_half[1], gi & 1))) break;
            mma_dK(st, first, 1);
            mma_commit(smem_u32(&bars->q_empty[st]));
            mma_dQ();
          }
        }
        if (!ok) break;
        mma_commit(smem_u32(&bars->kv_done));
        mbar_arrive(smem_u32(&bars->item_empty[slot]));
      }
      if (!ok) {
        mma_commit(smem_u32(&bars->drain));
        mbar_wait_drain(smem_u32(&bars->drain), 0);
      }
    }
   }
#ifdef ATTN_TRACE
   else if ((warp == 14 || warp == 15) && lane == 0 && a.trace != nullptr && blockIdx.x == 0) {
    // trace builds only: record when the traced steps' dO (warp 14) and Q
    // (warp 15) stages land
    uint64_t* full = warp == 14 ? bars->do_full : bars->q_full;
    for (uint32_t t = 0; t < kTraceFrom + kTraceSteps; ++t) {
      if (!mbar_wait(smem_u32(&full[t % C::kStages]), (t / C::kStages) & 1, ab)) break;
      ATTN_TRACE_EV(warp == 14 ? 44 : 45, t);
    }
   }
#endif
  } else if (warp < 8) {
    regs_dec<RegSplit<DQK>::kCompute>();
    // ================================================= P / dS warpgroups
    const int grp = warp >> 2;                      // 0: queries 0-63, 1: queries 64-127
    const int r = (warp & 3) * 32 + lane;           // TMEM lane = key row of S^T / dP^T
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    uint32_t q_it = 0, gi = 0;
    bool ok = true;
    for (uint32_t k = 0; ok; ++k) {
      const uint32_t slot = k & 1;
      if (!(ok = mbar_wait_warp(smem_u32(&bars->item_full[slot]), (k >> 1) & 1, ab))) break;
      const int item = bars->item_slot[slot];
      if (item >= sh.n_items) break;
      const Item it = decode_item(sh, tb, item, false);
      const int nq = cdiv(it.Lq, kTile);
      const int i0 = first_qtile(sh, it, it.tile), i1 = last_qtile(sh, it, it.tile, nq) + 1;
      const int kidx0 = it.tile * kTile + r;  // this thread's key
      const bool key_ok = kidx0 < it.Lk;
      const uint8_t* col = mask_col<kMask>(sh, it);
      for (int i = next_qtile(sh, col, i0, i1); i < i1;
           i = next_qtile(sh, col, i + 1, i1), ++q_it, ++gi) {
        const uint32_t st = q_it % C::kStages;
        const float* nlse2 = stat_f + st * (C::kStatBytes / 4) + grp * 64;  // -LSE * log2(e)
        const float* ndsum = nlse2 + kTile;                                  // -D
        // ---- P^T = exp2(S^T * s*log2e - LSE2), masked; bf16 pairs -> TMEM
        if (!(ok = mbar_wait_warp(smem_u32(&bars->s_full), gi & 1, ab))) break;
        tc_fence_after();
        if (lane == 0 && (warp & 3) == 0) ATTN_TRACE_EV(20, gi);
        uint32_t pk[32];  // P^T of this thread's key row, 64 queries as bf16 pairs
        // key kidx is visible to query q iff kidx - off - wr <= q <= kidx - off + wl
        // (band bounds; -1 = open): this group's visible query columns are
        // [qmin, qmax), none for a key past the sequence end
        const int qrel = kidx0 - kTile * i - grp * 64;  // kidx - (first query of the group)
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
              const int q = c * 32 + e;  // query column within this group
              const float4 l4 = *reinterpret_cast<const float4*>(nlse2 + q);
              const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
              float pe[4];
#pragma unroll
              for (int u = 0; u < 4; ++u)
                pe[u] = (q + u >= qmin && q + u < qmax)
                            ? ex2(fmaf(__uint_as_float(sr[e + u]), a.scale_log2, lv[u]))
                            : 0.f;
              pk[(q >> 1) + 0] = pack_bf16(pe[0], pe[1]);
              pk[(q >> 1) + 1] = pack_bf16(pe[2], pe[3]);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const int q = c * 32 + e;
              const float4 l4 = *reinterpret_cast<const float4*>(nlse2 + q);
              // two scores per packed FMA: S * s*log2e - LSE2
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
        if (lane == 0) mbar_arrive(smem_u32(&bars->p_full));
        if (lane == 0 && (warp & 3) == 0) ATTN_TRACE_EV(21, gi);
        // ---- dS^T = P^T ⊙ (dP^T − D) -> bf16 panel `grp` of sdS
        if (!(ok = mbar_wait_warp(smem_u32(&bars->dp_full), gi & 1, ab))) break;
        tc_fence_after();
        if (lane == 0 && (warp & 3) == 0) ATTN_TRACE_EV(22, gi);
        // The previous dS tile has been consumed: its dK and dQ products were
        // issued before this dP, and the commit behind dp_full tracks every
        // product issued before it, so no separate wait is needed here.
        if (lane == 0 && (warp & 3) == 0) ATTN_TRACE_EV(25, gi);
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
            // dS = P * (dP - D): the difference in fp32 (packed pairs), rounded
            // to bf16, then multiplied by the bf16 P pair (the product is
            // rounded to bf16 for the MMAs anyway)
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint64_t d2 = add2(f2(__uint_as_float(dr[e0 + 2 * u]),
                                          __uint_as_float(dr[e0 + 2 * u + 1])), nd2[u]);
              w[u] = mul_bf16x2(pk[ch * 4 + u], pack_bf16(f2_lo(d2), f2_hi(d2)));
            }
            st_shared_v4(sdS + grp * kPanelBytes + sw128_offset(r, ch), w[0], w[1], w[2], w[3]);
          }
          // this half of the dS^T columns is ready for dK
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->ds_half[c]));
          if (lane == 0 && (warp & 3) == 0) ATTN_TRACE_EV(23 + c, gi);
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->item_empty[slot]));
    }
  } else {
    regs_inc<RegSplit<DQK>::kDq>();
    // ================================================= dQ reduction + dK/dV epilogue
    // warps 8-11: thread = TMEM lane = query row of dQ, key row of dK / dV
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int wt = threadIdx.x - 8 * 32;  // 0..127 within this warpgroup
    uint32_t gi = 0;
    bool ok = true;
    // Pacing of the dQ reductions.  Issued back to back, the 128 threads'
    // DQK/4 vector reductions fill the SM's queue to the L2 faster than it
    // drains (32 bytes per clock), and every shared-memory access and
    // barrier wait of the other roles queues behind them — the MMA issuer's
    // waits and the dS stores stall for about a thousand cycles per q-tile.
    // Spreading the reductions over about 80 % of the q-tile step (measured
    // between consecutive dQ tiles, capped) keeps the queue short.
    // In deterministic mode the next kv tile's contribution waits for this
    // one's reductions, so they go out unpaced.
    long long t_prev = 0;
    int pace = a.deterministic ? 0 : kRedPaceCap;
    // Deterministic mode at d <= 128: the "added" mark of a q-tile is released
    // after the NEXT q-tile's drain, so that the fence it needs (the
    // reductions must reach the L2 first) does not hold up that drain — the
    // kv tile below, which reaches this q-tile about one step later, finds it
    // by then.  At d = 192 (no registers to spare) it goes out at once.
    constexpr bool kDeferRelease = !C::kSharedSdP;
    int64_t rel_word = -1;
    int rel_val = 0;
    for (uint32_t k = 0; ok; ++k) {
      const uint32_t slot = k & 1;
      if (!(ok = mbar_wait_warp(smem_u32(&bars->item_full[slot]), (k >> 1) & 1, ab))) break;
      const int item = bars->item_slot[slot];
      if (item >= sh.n_items) break;
      const Item it = decode_item(sh, tb, item, false);
      const int nq = cdiv(it.Lq, kTile);
      const int nk = cdiv(it.Lk, kTile);
      const int i1 = last_qtile(sh, it, it.tile, nq) + 1;
      const uint8_t* col = mask_col<kMask>(sh, it);
      const int ifirst = next_qtile(sh, col, first_qtile(sh, it, it.tile), i1);
      for (int i = ifirst; i < i1; i = next_qtile(sh, col, i + 1, i1), ++gi) {
        // deterministic order: contributions to q-tile i are added in
        // descending kv-tile order.  The tile's word holds 1 + the kv tile
        // that added to it last (0: none yet); this one waits for the
        // contributor just above it: the next kv tile up within q-tile i's
        // band (that the block mask keeps).
        auto wait_target = [&]() {
          const int last = last_kvtile(sh, it, i, nk);
          int above = it.tile + 1;
          if constexpr (kMask)
            while (above <= last && !tile_on(sh, it, i, above)) ++above;
          return (above <= last ? above + 1 : 0) + a.sem_bias;
        };
        // under a block mask the search reads the mask: done before the dQ
        // row is loaded, while few registers are live
        int target_m = 0;
        if constexpr (kMask)
          if (a.deterministic && wt == 0) target_m = wait_target();
        if (!(ok = mbar_wait_warp(smem_u32(&bars->dq_full), gi & 1, ab))) break;
        tc_fence_after();
        {
          const long long t_now = clock64();
          if (t_prev != 0) {
            const long long step = t_now - t_prev;
            pace = a.deterministic ? 0
                   : kRedSpread > 0
                       ? (int)min((long long)kRedPaceCap, step * kRedSpread / (256 * (DQK / 4)))
                       : kRedPaceCap;
          }
          t_prev = t_now;
        }
        if (lane == 0 && warp == 8) ATTN_TRACE_EV(30, gi);
        uint32_t qv[DQK];
#pragma unroll
        for (int c = 0; c < DQK / 32; ++c)
          tmem_ld32(tmem + lane_base + C::kTmemdQ + c * 32,
                    *reinterpret_cast<uint32_t(*)[32]>(&qv[c * 32]));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->dq_free));
        if (lane == 0 && warp == 8) ATTN_TRACE_EV(31, gi);
        if (kDeferRelease && wt == 0 && rel_word >= 0) {  // the previous q-tile's mark
          __threadfence();
          st_release_gpu(a.ws.sem + rel_word, rel_val);
          rel_word = -1;
        }
        const int64_t g = (int64_t)(it.tile_base + i) * sh.H + it.head;
        float* acc = a.ws.dq_acc + g * (kTile * DQK);
        if (a.deterministic) {
          int* sem = a.ws.sem + 2 * g;
          if (wt == 0) {
            const int target = kMask ? target_m : wait_target();
            const uint64_t t0 = globaltimer();
            while (ld_acquire_gpu(sem) != target) {
              // give up on our own limit, or as soon as any CTA has failed
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
          for (int c4 = 0; c4 < DQK / 4; ++c4) {
            red_add_v4(acc + (c4 * kTile + r) * 4, __uint_as_float(qv[c4 * 4 + 0]),
                       __uint_as_float(qv[c4 * 4 + 1]), __uint_as_float(qv[c4 * 4 + 2]),
                       __uint_as_float(qv[c4 * 4 + 3]));
            const long long due = t0 + (long long)(c4 + 1) * pace;
            while (clock64() < due) {
            }
          }
        } else {
#pragma unroll
          for (int c4 = 0; c4 < DQK / 4; ++c4)
            red_add_v4(acc + (c4 * kTile + r) * 4, __uint_as_float(qv[c4 * 4 + 0]),
                       __uint_as_float(qv[c4 * 4 + 1]), __uint_as_float(qv[c4 * 4 + 2]),
                       __uint_as_float(qv[c4 * 4 + 3]));
        }
        if (lane == 0 && warp == 8) ATTN_TRACE_EV(32, gi);
        if (a.deterministic) {
          named_bar_sync(1, 128);  // every thread's reductions issued
          if (wt == 0) {
            if constexpr (kDeferRelease) {
              rel_word = 2 * g;
              rel_val = it.tile + 1;
            } else {
              __threadfence();
              st_release_gpu(a.ws.sem + 2 * g, it.tile + 1);
            }
          }
        }
      }
      // the item's last mark goes out before the epilogue
      if (kDeferRelease && wt == 0 && rel_word >= 0) {
        __threadfence();
        st_release_gpu(a.ws.sem + rel_word, rel_val);
        rel_word = -1;
      }
      if (!ok) break;
      // ---- epilogue: dK = s * acc, dV = acc (thread = key row r)
      if (!(ok = mbar_wait_warp(smem_u32(&bars->kv_done), k & 1, ab))) break;
      tc_fence_after();
      const int kidx = it.tile * kTile + r;
      const bool key_ok = kidx < it.Lk;
      const int krow = key_row0(sh, it) + kidx;
      const bool nothing = ifirst >= i1;  // no query sees this kv tile: zeros
      auto dk_row = [&]() { return a.dk + (int64_t)krow * a.dk_row_stride + (int64_t)it.head * DQK; };
      auto dv_row = [&]() { return a.dv + (int64_t)krow * a.dv_row_stride + (int64_t)it.head * DV; };
      if constexpr (C::kSharedSdP) {
        // d = 192: each accumulator is read whole into bf16 pairs and released
        // before its row is stored (32-byte stores when aligned), so that the
        // next item's first dV and dK need not wait for the stores
        {
          uint32_t pk[DV / 2];
          epi_read<DV>(tmem + lane_base + C::kTmemdV, 1.0f, nothing, pk);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->accv_free));
          if (key_ok) epi_store<DV>(dv_row(), a.st32, pk);
        }
        {
          uint32_t pk[DQK / 2];
          epi_read<DQK>(tmem + lane_base + C::kTmemdK, a.scale, nothing, pk);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->acck_free));
          if (key_ok) epi_store<DQK>(dk_row(), a.st32, pk);
        }
      } else {
        // d <= 128: 32 columns at a time, each read followed by its stores
        // (spacing the stores out; 32-byte stores when aligned), both
        // accumulators released at the end — this measured faster here than
        // releasing them early
#pragma unroll 1
        for (int c = 0; c < DQK / 32; ++c) {
          uint32_t pk[16];
          epi_read<32>(tmem + lane_base + C::kTmemdK + c * 32, a.scale, nothing, pk);
          if (key_ok) epi_store<32>(dk_row() + c * 32, a.st32, pk);
        }
#pragma unroll 1
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t pk[16];
          epi_read<32>(tmem + lane_base + C::kTmemdV + c * 32, 1.0f, nothing, pk);
          if (key_ok) epi_store<32>(dv_row() + c * 32, a.st32, pk);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&bars->accv_free));
          mbar_arrive(smem_u32(&bars->acck_free));
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&bars->item_empty[slot]));
      }
    }
  }

  ATTN_TRACE_FLUSH;
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// 3. dQ conversion: one CTA per half (64 rows) of a (q-tile, head)
// ---------------------------------------------------------------------------
template <int DQK, typename Tables>
__global__ void __launch_bounds__(256)
    attn_bwd_convert_kernel(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dq,
                            const int64_t dq_row_stride, const float scale, const SeqShape sh,
                            const __grid_constant__ Tables tb) {
  using S = SeqOf<Tables>;
  extern __shared__ float tile_s[];  // [64][DQK + 4]
  constexpr int kLd = DQK + 4;
  constexpr int kR = 64;
  const int th = blockIdx.x >> 1, hf = blockIdx.x & 1;
  const int g = th / sh.H;
  const int h = th - g * sh.H;
  int s, i;
  S::tile_of(sh, tb, g, s, i);
  const int L = S::length(sh, tb, s);
  const int rows = max(0, min(kR, L - i * kTile - hf * kR));
  const float4* src = reinterpret_cast<const float4*>(dq_acc + (int64_t)th * kTile * DQK);
  for (int idx = threadIdx.x; idx < kR * DQK / 4; idx += blockDim.x) {
    const int c4 = idx / kR, r = idx - c4 * kR;
    const float4 v = src[c4 * kTile + hf * kR + r];
    float* d = tile_s + r * kLd + c4 * 4;
    d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
  }
  __syncthreads();
  const int64_t row0 = S::row0(sh, tb, s) + (int64_t)i * kTile + hf * kR;
  for (int idx = threadIdx.x; idx < rows * (DQK / 8); idx += blockDim.x) {
    const int r = idx / (DQK / 8), c8 = idx - r * (DQK / 8);
    const float* f = tile_s + r * kLd + c8 * 8;
    uint4 w;
    w.x = pack_bf16(f[0] * scale, f[1] * scale);
    w.y = pack_bf16(f[2] * scale, f[3] * scale);
    w.z = pack_bf16(f[4] * scale, f[5] * scale);
    w.w = pack_bf16(f[6] * scale, f[7] * scale);
    *reinterpret_cast<uint4*>(dq + (row0 + r) * dq_row_stride + (int64_t)h * DQK + c8 * 8) = w;
  }
}

#ifdef ATTN_TRACE
unsigned long long* g_trace_buf = nullptr;
#endif

template <int DQK, int DV, typename Tables>
cudaError_t launch_all(const BwdLaunch& L, const Tables& tb) {
  using C = BwdCfg<DQK, DV>;
  const int total_rows = L.sh.varlen ? L.tables->cu[L.sh.nseq] : L.sh.nseq * L.sh.Tq;
  // 1. preprocess
  {
    cudaLaunchConfig_t cfg = {};
    // many small blocks: each thread has one O / dO pair in flight per loop
    // step, so occupancy carries the bandwidth (32 blocks per SM measured best)
    cfg.gridDim = dim3(L.num_sms * 32);
    cfg.blockDim = dim3(256);
    cfg.stream = L.stream;
    cudaError_t e;
    if (L.prof_aux[0] && (e = cudaEventRecord(L.prof_aux[0], L.stream)) != cudaSuccess) return e;
    e = cudaLaunchKernelEx(
        &cfg, attn_bwd_pre_kernel<DQK, DV, Tables>, reinterpret_cast<const __nv_bfloat16*>(L.o),
        reinterpret_cast<const __nv_bfloat16*>(L.dout), L.lse, L.o_row_stride, L.do_row_stride,
        L.lse_head_stride, L.lse_seq_stride, total_rows, L.n_qtiles, L.ws, L.sh, tb);
    if (e != cudaSuccess) return e;
    if (L.prof_aux[1] && (e = cudaEventRecord(L.prof_aux[1], L.stream)) != cudaSuccess) return e;
  }
  // 2. main
  {
    MainArgs a;
    a.dk = reinterpret_cast<__nv_bfloat16*>(L.dk);
    a.dv = reinterpret_cast<__nv_bfloat16*>(L.dv);
    a.dk_row_stride = L.dk_row_stride;
    a.dv_row_stride = L.dv_row_stride;
    a.scale = L.scale;
    a.scale_log2 = L.scale_log2;
    a.deterministic = L.deterministic;
    a.sem_bias = L.sem_bias;
    a.st32 = ((reinterpret_cast<uintptr_t>(L.dk) | reinterpret_cast<uintptr_t>(L.dv)) & 31u) == 0 &&
             (L.dk_row_stride * 2) % 32 == 0 && (L.dv_row_stride * 2) % 32 == 0;
#ifdef ATTN_TRACE
    a.trace = g_trace_buf;
#endif
    a.ws = L.ws;
    a.sh = L.sh;
    cudaError_t e;
    if (L.prof_start && (e = cudaEventRecord(L.prof_start, L.stream)) != cudaSuccess) return e;
    if (L.pair) {
      e = launch_bwd_pair_main(L);
    } else {
      auto* k = L.sh.blk != nullptr ? attn_bwd_main_kernel<DQK, DV, Tables, true>
                                    : attn_bwd_main_kernel<DQK, DV, Tables, false>;
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::kSmemBytes + kTraceSmem);
      if (e != cudaSuccess) return e;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(L.grid);
      cfg.blockDim = dim3(kMainThreads);
      cfg.dynamicSmemBytes = C::kSmemBytes + kTraceSmem;
      cfg.stream = L.stream;
      e = cudaLaunchKernelEx(&cfg, k, L.tm_q, L.tm_k, L.tm_v, L.tm_do, a, tb);
    }
    if (e != cudaSuccess) return e;
    if (L.prof_stop && (e = cudaEventRecord(L.prof_stop, L.stream)) != cudaSuccess) return e;
  }
  // 3. dQ conversion
  {
    const int smem = 64 * (DQK + 4) * 4;
    auto* k = attn_bwd_convert_kernel<DQK, Tables>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.n_qtiles * L.sh.H * 2);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    if (L.prof_aux[2] && (e = cudaEventRecord(L.prof_aux[2], L.stream)) != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, k, static_cast<const float*>(L.ws.dq_acc),
                           reinterpret_cast<__nv_bfloat16*>(L.dq), L.dq_row_stride, L.scale, L.sh, tb);
    if (e != cudaSuccess) return e;
    if (L.prof_aux[3] && (e = cudaEventRecord(L.prof_aux[3], L.stream)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int DQK, int DV>
cudaError_t launch_typed(const BwdLaunch& L) {
  if (L.tables) return launch_all<DQK, DV, VarlenTables>(L, *L.tables);
  return launch_all<DQK, DV, NoTables>(L, NoTables{});
}

}  // namespace

#ifdef ATTN_TRACE
// Trace builds only: buffer of kMainThreads x 64 records for CTA 0 (null = off).
extern "C" void attn_trace_set(void* buf) { g_trace_buf = static_cast<unsigned long long*>(buf); }
#endif

int bwd_smem_bytes(int dqk, int dv) {
  if (dqk == 64 && dv == 64) return BwdCfg<64, 64>::kSmemBytes;
  if (dqk == 128 && dv == 128) return BwdCfg<128, 128>::kSmemBytes;
  if (dqk == 192 && dv == 128) return BwdCfg<192, 128>::kSmemBytes;
  return -1;
}

cudaError_t launch_bwd(const BwdLaunch& L, int dqk, int dv) {
  if (dqk == 64 && dv == 64) return launch_typed<64, 64>(L);
  if (dqk == 128 && dv == 128) return launch_typed<128, 128>(L);
  if (dqk == 192 && dv == 128) return launch_typed<192, 128>(L);
  return cudaErrorInvalidValue;
}

}  // namespace attn
