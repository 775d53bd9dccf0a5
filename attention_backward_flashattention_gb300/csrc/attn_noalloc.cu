// attn_noalloc.cu — attn_bwd_noalloc: the backward pass for callers that must
// not allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is not an option — a plugin
// whose host framework owns every byte of device memory through its own
// caching allocator, or a latency-critical loop that may not call cudaMalloc
// because it can synchronise the whole device and can fail at any moment.
// Such callers cannot provide the backward workspace that attn_bwd needs.
//
// How: the workspace lives in a file-scope device array of fixed size,
// kScratchBytes (32 MiB).  It is part of this file's device code, so every
// GPU on which this code is loaded holds those 32 MiB until the process exits.
// Host code cannot use the array's name as a device address (in host code it
// is only a stand-in), so the first call on each device looks the address up
// with cudaGetSymbolAddress while that device is current and caches it; make
// that first call on a device before any stream capture.
//
// Every call uses the same array and leaves its contents behind.  Each call
// starts by clearing what must start at zero (its first kernel zeroes the dQ
// accumulator, the semaphores, the work counter and the status word and
// rewrites every per-row statistic), so one call never sees another's data —
// but calls whose kernels overlap on the GPU (different streams, or different
// host threads, without ordering between them) race on the array and give
// wrong results.  Order such calls on one stream.
#include <mutex>

#include "../../include/attn.h"
#include "attn_internal.h"

namespace {

constexpr size_t kScratchBytes = 32ull << 20;  // 32 MiB

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device (set up once per device).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                const void* dO, const float* lse, void* dq, void* dk,
                                void* dv_out, int B, int H, int Tq, int Tk, int dqk, int dv,
                                int causal, float scale, const int* cu_seqlens, int layout,
                                int deterministic, void* stream) {
  const size_t need = attn_bwd_workspace_size(B, H, Tq, Tk, dqk, dv, cu_seqlens != nullptr,
                                               deterministic);
  if (need == 0) return ATTN_ERR_INVALID_ARG;
  if (need > kScratchBytes) return ATTN_ERR_SCRATCH_TOO_SMALL;
  void* ws = nullptr;
  const int rc = scratch_address(&ws);
  if (rc != ATTN_OK) return rc;
  return attn_bwd(q, k, v, o, dO, lse, dq, dk, dv_out, B, H, Tq, Tk, dqk, dv, causal, scale,
                  cu_seqlens, layout, deterministic, ws, kScratchBytes, stream);
}
