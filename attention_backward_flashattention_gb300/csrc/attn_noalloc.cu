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
// is only a stand-in), so the first call in each CUDA context looks the
// address up with cudaGetSymbolAddress while that context's device is current
// and caches it per device, together with the context it belongs to; a call
// that finds another context current on the device (the primary context was
// reset and re-created, which reloads the module) looks the address up again.
// Make that first call on a device before any stream capture.
//
// Every call uses the same array and leaves its contents behind.  Each call
// starts by clearing what must start at zero (its first kernel zeroes the dQ
// accumulator, the semaphores, the work counter and the status word and
// rewrites every per-row statistic), so one call never sees another's data —
// but calls whose kernels overlap on the GPU (different streams, or different
// host threads, without ordering between them) race on the array and give
// wrong results.  Order such calls on one stream.  The array's first word is
// the status word of the last call; attn_bwd_noalloc_status reads it.
#include <cuda.h>

#include <mutex>

#include "../../include/attn.h"
#include "attn_internal.h"

namespace {

constexpr size_t kScratchBytes = 32ull << 20;  // 32 MiB

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The driver's cuCtxGetCurrent, found through the runtime (no link to libcuda).
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of g_scratch in the current context (looked up once per
// context and device).  cudaGetSymbolAddress also makes the device's primary
// context current when this thread has none yet.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  CtxGetCurrentFn get = ctx_get_current();
  if (get == nullptr) return ATTN_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (ctx == nullptr || g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return ATTN_ERR_CUDA;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
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

extern "C" int attn_bwd_noalloc_status(void* stream) {
  void* ws = nullptr;
  const int rc = scratch_address(&ws);
  if (rc != ATTN_OK) return rc;
  return attn_bwd_status(ws, stream);
}
