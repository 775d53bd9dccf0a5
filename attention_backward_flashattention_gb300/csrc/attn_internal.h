// attn_internal.h — what the C-ABI layer (attn_api.cu) hands to the kernel
// launchers (attn_fwd.cu, attn_bwd.cu).  Host-side C++ only; not part of the
// public interface (include/attn.h is).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attn_common.cuh"

namespace attn {

// Forward launch description.
struct FwdLaunch {
  CUtensorMap tm_q, tm_k, tm_v;  // panel maps over (d, H, rows)
  void* o;                       // bf16 output
  float* lse;                    // fp32 statistics or null (inference)
  int64_t o_row_stride;          // elements between token rows of O
  int64_t lse_head_stride;       // elements between heads of LSE
  int64_t lse_seq_stride;        // fixed length: elements between sequences; varlen: 0
  float scale_log2;              // scale * log2(e)
  int* status;                   // device status word
  int* claim;                    // device counters (items claimed, CTAs done), zero at launch
  SeqShape sh;
  const VarlenTables* tables;    // null for fixed-length batches
  int grid;
  cudaStream_t stream;
};

// Backward workspace (caller-owned device memory), carved in this order.
struct BwdWorkspace {
  int* header;      // [0] status, [1] work-item counter
  int* sem;         // per (q-tile, head, tile half): the key tile (or pair) that added last
                    // (deterministic mode; the one-CTA kernel uses half 0)
  float* nlse2;     // per (q-tile, head, row): -LSE * log2(e); -inf past the sequence end
  float* ndsum;     // per (q-tile, head, row): -D = -rowsum(dO * O); 0 past the end
  float* dq_acc;    // per (q-tile, head): [dqk/4][128][4] fp32 partial dQ
};

struct BwdLaunch {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // panel maps over (d, H, rows)
  CUtensorMap tm_q64, tm_do64;          // 64-row boxes of q and dO (CTA-pair kernel)
  int pair;                             // 1: the main kernel runs on CTA pairs
  const void* o;         // bf16 O, for D
  const void* dout;      // bf16 dO, for D
  const float* lse;      // fp32 LSE from the forward
  void* dq;              // bf16 outputs
  void* dk;
  void* dv;
  int64_t q_row_stride, k_row_stride, v_row_stride;     // inputs
  int64_t o_row_stride, do_row_stride;                   // O and dO
  int64_t dq_row_stride, dk_row_stride, dv_row_stride;   // outputs
  int64_t lse_head_stride, lse_seq_stride;
  float scale;        // softmax scale
  float scale_log2;   // scale * log2(e)
  int n_qtiles;       // q-tiles over all sequences (workspace tile space)
  int deterministic;
  int sem_bias;       // fault injection for tests (0 in normal use)
  cudaEvent_t prof_start, prof_stop;  // recorded around the main kernel when set
  cudaEvent_t prof_aux[4];            // around the preprocess (0, 1) and dQ conversion (2, 3)
  BwdWorkspace ws;
  SeqShape sh;        // n_items = kv-tile items
  const VarlenTables* tables;
  int grid;
  int num_sms;
  cudaStream_t stream;
};

// Each returns cudaSuccess or the launch error.
cudaError_t launch_fwd(const FwdLaunch& L, int dqk, int dv);
cudaError_t launch_bwd(const BwdLaunch& L, int dqk, int dv);
// The backward main kernel on CTA pairs (dqk = dv = 128; L.grid even, items = key-tile pairs).
cudaError_t launch_bwd_pair_main(const BwdLaunch& L);
int bwd_pair_smem_bytes();

// Device address of the forward kernels' status word on the current device.
int* fwd_status_ptr();
// Device address of forward work-item counter `slot` on the current device.
constexpr int kFwdClaimSlots = 256;
int* fwd_claim_ptr(int slot);

// Dynamic shared memory the kernels need (for validation / tests).
int fwd_smem_bytes(int dqk, int dv);
int bwd_smem_bytes(int dqk, int dv);

}  // namespace attn
