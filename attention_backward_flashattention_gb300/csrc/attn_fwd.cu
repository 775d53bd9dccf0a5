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
// One CTA (192 threads) per SM, persistent over work items (see
// attn_common.cuh for the item order):
//   warps 0-3  softmax: thread r owns query row r of the tile (TMEM lane r)
//   warp 4     TMA producer: Q tile once per item, K/V tiles into a ring
//   warp 5     MMA issuer: S = Q K^T into one of two TMEM buffers, then
//              O += P V into a TMEM accumulator
// Tensor memory: S buffers at columns [0,128) and [128,256), O at [256, 256+dv).
// P goes through shared memory as bf16 in the 128-byte-swizzled panel layout
// the MMA reads.  The running maximum is only moved (and O rescaled) when it
// grows by more than 2^8, so most tiles skip the rescale.
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kFwdThreads = 192;
constexpr int kPanelBytes = kTile * 128;  // [128 rows][64] bf16
constexpr int kMaxSmem = 232448;

template <int DQK, int DV>
struct FwdCfg {
  static constexpr int kQPanels = DQK / 64;
  static constexpr int kVPanels = DV / 64;
  static constexpr int kQBytes = kQPanels * kPanelBytes;
  static constexpr int kKBytes = kQPanels * kPanelBytes;
  static constexpr int kVBytes = kVPanels * kPanelBytes;
  static constexpr int kPBytes = 2 * kPanelBytes;
  static constexpr int kFixed = kQBytes + kPBytes + 1024 /*barriers*/ + 1024 /*alignment*/;
  // K and V have rings of their own: S(t) needs only a K slot, so it can be
  // issued while V of the previous tile is still being read by O += P V.
  // Two K slots at least; V slots from what is left (one suffices).
  static constexpr int kPairsFit = (kMaxSmem - kFixed) / (kKBytes + kVBytes);
  static constexpr int kKStages = kPairsFit >= 4 ? 4 : (kPairsFit >= 2 ? kPairsFit : 2);
  static constexpr int kVStagesFit = (kMaxSmem - kFixed - kKStages * kKBytes) / kVBytes;
  static constexpr int kVStages = kVStagesFit > kKStages ? kKStages : kVStagesFit;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kQBytes;
  static constexpr int kOffV = kOffK + kKStages * kKBytes;
  static constexpr int kOffP = kOffV + kVStages * kVBytes;
  static constexpr int kOffBar = kOffP + kPBytes;
  static constexpr int kSmemBytes = kOffBar + 1024 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTmemS = 0;
  static constexpr uint32_t kTmemO = 256;
  static_assert(kVStages >= 1, "shared memory too small");
  static_assert(kKStages <= 4 && kVStages <= 4, "barrier arrays hold 4 stages");
  static_assert(kSmemBytes <= kMaxSmem, "shared memory budget");
};

// Barrier slots inside the barrier block.
struct FwdBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, o_done;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

template <int DQK, int DV, typename Tables>
__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ out,
                    float* __restrict__ lse, const int64_t o_row_stride,
                    const int64_t lse_head_stride, const int64_t lse_seq_stride,
                    const float scale_log2, int* status, const SeqShape sh,
                    const __grid_constant__ Tables tb) {
  using C = FwdCfg<DQK, DV>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FwdBars* bars = reinterpret_cast<FwdBars*>(smem + C::kOffBar);
  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  const uint32_t sK = smem_u32(smem + C::kOffK);
  const uint32_t sV = smem_u32(smem + C::kOffV);
  const uint32_t sP = smem_u32(smem + C::kOffP);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  Abort ab{&bars->abort_flag, status};

  if (threadIdx.x == 0) {
    bars->abort_flag = 0;
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
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars->s_full[b]), 1);
      mbar_init(smem_u32(&bars->s_free[b]), 4);
    }
    mbar_init(smem_u32(&bars->p_full), 4);
    mbar_init(smem_u32(&bars->o_done), 1);
    mbar_init(smem_u32(&bars->drain), 1);
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(&bars->tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t kv_it = 0, item_iter = 0, q_issued = 0, k_issued = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < sh.n_items; item += gridDim.x, ++item_iter) {
        const Item it = decode_item(sh, tb, item, true);
        const int nk = cdiv(it.Lk, kTile);
        const int nkv = sh.causal ? min(it.tile + 1, nk) : nk;
        if (!(ok = mbar_wait(smem_u32(&bars->q_empty), (item_iter & 1) ^ 1, ab))) break;
        mbar_arrive_expect_tx(smem_u32(&bars->q_full), C::kQBytes);
        q_issued = item_iter + 1;
        for (int pnl = 0; pnl < C::kQPanels; ++pnl)
          tma_load_3d(sQ + pnl * kPanelBytes, &tm_q, smem_u32(&bars->q_full), pnl * 64, it.head,
                      it.row0 + it.tile * kTile);
        const int krow0 = key_row0(sh, it);
        for (int j = 0; j < nkv; ++j, ++kv_it) {
          const uint32_t sk = kv_it % C::kKStages, sv = kv_it % C::kVStages;
          if (!(ok = mbar_wait(smem_u32(&bars->k_empty[sk]), ((kv_it / C::kKStages) & 1) ^ 1, ab)))
            break;
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
        }
      }
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
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idO = idesc_bf16(128, DV, false, true);
      uint32_t kv_it = 0, sc = 0, item_iter = 0;
      bool ok = true;
      // descriptor bases (each MMA then only adds a constant)
      const uint64_t bQ_k = kmajor_base(sQ), bP_k = kmajor_base(sP);
      const uint32_t tO = tmem + C::kTmemO;
      auto issue_pv = [&](uint32_t t_kv, uint32_t t_s, bool first) -> bool {
        if (!mbar_wait(smem_u32(&bars->p_full), t_s & 1, ab)) return false;
        tc_fence_after();
        const uint32_t sv = t_kv % C::kVStages;
        if (!mbar_wait(smem_u32(&bars->v_full[sv]), (t_kv / C::kVStages) & 1, ab)) return false;
        const uint64_t bV = mnmajor_base(sV + sv * C::kVBytes, 128);
        mma_bf16(tO, bP_k, bV, idO, first ? 0u : 1u);
#pragma unroll
        for (int kk = 1; kk < kTile / 16; ++kk)
          mma_bf16(tO, bP_k + kmajor_step(kk, 128), bV + mnmajor_step(kk), idO, 1u);
        mma_commit(smem_u32(&bars->o_done));
        mma_commit(smem_u32(&bars->v_empty[sv]));
        return true;
      };
      for (int item = blockIdx.x; ok && item < sh.n_items; item += gridDim.x, ++item_iter) {
        const Item it = decode_item(sh, tb, item, true);
        const int nk = cdiv(it.Lk, kTile);
        const int nkv = sh.causal ? min(it.tile + 1, nk) : nk;
        if (!(ok = mbar_wait(smem_u32(&bars->q_full), item_iter & 1, ab))) break;
        tc_fence_after();
        for (int j = 0; j < nkv; ++j) {
          const uint32_t t = kv_it + j;
          const uint32_t ts = sc + j;
          const uint32_t sk = t % C::kKStages;
          const uint32_t b = ts & 1;
          if (!(ok = mbar_wait(smem_u32(&bars->k_full[sk]), (t / C::kKStages) & 1, ab))) break;
          if (!(ok = mbar_wait(smem_u32(&bars->s_free[b]), ((ts >> 1) & 1) ^ 1, ab))) break;
          tc_fence_after();
          const uint64_t bK = kmajor_base(sK + sk * C::kKBytes);
          const uint32_t tS = tmem + C::kTmemS + b * 128;
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk)
            mma_bf16(tS, bQ_k + kmajor_step(kk, 128), bK + kmajor_step(kk, 128), idS,
                     kk > 0 ? 1u : 0u);
          mma_commit(smem_u32(&bars->s_full[b]));
          mma_commit(smem_u32(&bars->k_empty[sk]));
          if (j == nkv - 1) mma_commit(smem_u32(&bars->q_empty));
          if (j > 0 && !(ok = issue_pv(t - 1, ts - 1, j == 1))) break;
        }
        if (!ok) break;
        if (!(ok = issue_pv(kv_it + nkv - 1, sc + nkv - 1, nkv == 1))) break;
        kv_it += nkv;
        sc += nkv;
      }
      if (!ok) {
        mma_commit(smem_u32(&bars->drain));
        mbar_wait_drain(smem_u32(&bars->drain), 0);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x;  // query row within the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    uint32_t sc = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < sh.n_items; item += gridDim.x) {
      const Item it = decode_item(sh, tb, item, true);
      const int nk = cdiv(it.Lk, kTile);
      const int nkv = sh.causal ? min(it.tile + 1, nk) : nk;
      const int qidx = it.tile * kTile + r;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nkv; ++j, ++sc) {
        const uint32_t b = sc & 1;
        if (!(ok = mbar_wait_warp(smem_u32(&bars->s_full[b]), (sc >> 1) & 1, ab))) break;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_base + C::kTmemS + b * 128 + c * 32, sr[c]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->s_free[b]));
        const int kbase = j * kTile;
        const bool need_mask = (sh.causal && j == nkv - 1) || (kbase + kTile > it.Lk);
        float rowmax = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            float x = __uint_as_float(sr[c][e]) * scale_log2;
            if (need_mask) {
              const int kidx = kbase + c * 32 + e;
              if (kidx >= it.Lk || (sh.causal && kidx > qidx)) x = -INFINITY;
            }
            sr[c][e] = __float_as_uint(x);
            rowmax = fmaxf(rowmax, x);
          }
        }
        const float m_new = fmaxf(m, rowmax);
        const bool resc = (m_new - m) > 8.0f;  // also true on the first tile (m = -inf)
        const float m_use = resc ? m_new : m;
        const float alpha = resc ? ex2(m - m_use) : 1.0f;
        float rs = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float pe = ex2(__uint_as_float(sr[c][e]) - m_use);
            sr[c][e] = __float_as_uint(pe);
            rs += pe;
          }
        }
        if (j > 0) {
          // previous P consumed and O up to date
          if (!(ok = mbar_wait_warp(smem_u32(&bars->o_done), (sc - 1) & 1, ab))) break;
          tc_fence_after();
          if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
            for (int c = 0; c < DV / 32; ++c) {
              uint32_t ov[32];
              const uint32_t ta = tmem + lane_base + C::kTmemO + c * 32;
              tmem_ld32(ta, ov);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
              tmem_st32(ta, ov);
            }
            tmem_st_wait();
          }
        }
        l = l * alpha + rs;
        m = m_use;
        // P row -> shared memory (panel 0: keys 0-63, panel 1: keys 64-127)
#pragma unroll
        for (int ch = 0; ch < 16; ++ch) {
          const int c = ch >> 2, e0 = (ch & 3) * 8;
          const uint32_t addr = sP + (ch >> 3) * kPanelBytes + sw128_offset(r, ch & 7);
          st_shared_v4(addr,
                       pack_bf16(__uint_as_float(sr[c][e0 + 0]), __uint_as_float(sr[c][e0 + 1])),
                       pack_bf16(__uint_as_float(sr[c][e0 + 2]), __uint_as_float(sr[c][e0 + 3])),
                       pack_bf16(__uint_as_float(sr[c][e0 + 4]), __uint_as_float(sr[c][e0 + 5])),
                       pack_bf16(__uint_as_float(sr[c][e0 + 6]), __uint_as_float(sr[c][e0 + 7])));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->p_full));
      }
      if (!ok) break;
      // epilogue: O / l and the log-sum-exp
      if (!(ok = mbar_wait_warp(smem_u32(&bars->o_done), (sc - 1) & 1, ab))) break;
      tc_fence_after();
      const bool valid = qidx < it.Lq;
      const float inv_l = 1.0f / l;
      __nv_bfloat16* orow =
          out + (int64_t)(it.row0 + qidx) * o_row_stride + (int64_t)it.head * DV;
#pragma unroll 1
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tmem + lane_base + C::kTmemO + c * 32, ov);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(ov[q4 * 8 + 0]) * inv_l, __uint_as_float(ov[q4 * 8 + 1]) * inv_l);
            v.y = pack_bf16(__uint_as_float(ov[q4 * 8 + 2]) * inv_l, __uint_as_float(ov[q4 * 8 + 3]) * inv_l);
            v.z = pack_bf16(__uint_as_float(ov[q4 * 8 + 4]) * inv_l, __uint_as_float(ov[q4 * 8 + 5]) * inv_l);
            v.w = pack_bf16(__uint_as_float(ov[q4 * 8 + 6]) * inv_l, __uint_as_float(ov[q4 * 8 + 7]) * inv_l);
            *reinterpret_cast<uint4*>(orow + c * 32 + q4 * 8) = v;
          }
        }
      }
      tc_fence_before();
      if (lse != nullptr && valid) {
        const int64_t base = sh.varlen ? (int64_t)it.row0 : (int64_t)it.seq * lse_seq_stride;
        lse[(int64_t)it.head * lse_head_stride + base + qidx] =
            (m + log2f(l)) * 0.69314718055994530942f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int DQK, int DV>
cudaError_t launch_typed(const FwdLaunch& L) {
  using C = FwdCfg<DQK, DV>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.grid);
  cfg.blockDim = dim3(kFwdThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = L.stream;
  if (L.tables) {
    auto* k = attn_fwd_kernel<DQK, DV, VarlenTables>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, k, L.tm_q, L.tm_k, L.tm_v,
                              reinterpret_cast<__nv_bfloat16*>(L.o), L.lse, L.o_row_stride,
                              L.lse_head_stride, L.lse_seq_stride, L.scale_log2, L.status, L.sh,
                              *L.tables);
  }
  auto* k = attn_fwd_kernel<DQK, DV, NoTables>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, k, L.tm_q, L.tm_k, L.tm_v, reinterpret_cast<__nv_bfloat16*>(L.o),
                            L.lse, L.o_row_stride, L.lse_head_stride, L.lse_seq_stride,
                            L.scale_log2, L.status, L.sh, NoTables{});
}

}  // namespace

// Sticky status word of the forward kernels on each device (a bounded wait
// that gave up writes its code here; attn_fwd_status reads and clears it).
__device__ int g_fwd_status = 0;

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
