// attn_host.cu — attn_step_host: forward + backward for inputs and gradients
// that live in (pinned) host memory, with the host<->device copies overlapped
// with the kernels.
//
// The heads are independent problems, so the call cuts them into groups of at
// most G heads (half-size groups at both ends) and runs a three-stage pipeline
// over the groups:
//
//   h2d stream:      copy q, k, v, dO of group g into device set g % 2
//   compute stream:  attn_fwd (once q, k, v are in) + attn_bwd (once dO is) on set g % 2
//   d2h stream:      copy dq, dk, dv (and o) of set g % 2 into the host tensors
//
// so that group g+1's inputs travel and group g-1's gradients come back while
// group g is computed.  A head group is a strided slice of a (B,T,H,d) host
// tensor — B*T rows of G*d contiguous elements, H*d elements apart — which
// cudaMemcpy2DAsync moves as one copy into a contiguous (B,T,G,d) device
// buffer; the kernels then see a fixed-length problem with G heads.
//
// Two device sets alternate.  Set s is reused by group g+2 only after
//   - the kernels of group g are done with its inputs (h2d waits comp[s]),
//   - the gradients of group g have left the device (compute waits d2h[s]).
// The caller's stream waits for the last copies, so synchronising that stream
// (or recording an event on it) covers the whole call.  After each group's
// backward the status word of its workspace is copied into a per-group array
// at the end of the scratch, where attn_step_host_status() reads it.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "../../include/attn.h"
#include "attn_internal.h"

namespace {

size_t r256(size_t x) { return (x + 255) & ~size_t(255); }

// Byte offsets of the buffers of one device set (G heads).
struct SetLayout {
  size_t q, k, v, dO, o, lse, dq, dk, dv, ws, bytes;
  size_t ws_bytes;
};

SetLayout set_layout(int B, int G, int T, int dqk, int dv, int deterministic) {
  const size_t rows = (size_t)B * T;
  const size_t eq = rows * G * dqk * 2, ev = rows * G * dv * 2;
  SetLayout s;
  size_t off = 0;
  s.q = off;   off += r256(eq);
  s.k = off;   off += r256(eq);
  s.v = off;   off += r256(ev);
  s.dO = off;  off += r256(ev);
  s.o = off;   off += r256(ev);
  s.lse = off; off += r256(rows * G * sizeof(float));
  s.dq = off;  off += r256(eq);
  s.dk = off;  off += r256(eq);
  s.dv = off;  off += r256(ev);
  s.ws_bytes = attn_bwd_workspace_size(B, G, T, T, dqk, dv, 0, deterministic);
  s.ws = off;  off += r256(s.ws_bytes);
  s.bytes = off;
  return s;
}

// Default group size: half the heads, so that the groups are H/4, H/2, H/4.
// Each group costs a few launches and a load-balancing tail, and the copies of
// a group of H/2 heads take well under its kernels' time (measured: smaller
// groups were slower end to end).
int pick_group(int H, int heads_per_group) {
  if (heads_per_group > 0) return std::min(heads_per_group, H);
  return (H + 1) / 2;
}

// Head-group sizes, none above G.  The first and the last group are about
// half as large: nothing overlaps the first group's inputs or the last
// group's results, so smaller end groups shorten the pipeline's fill and drain.
std::vector<int> group_sizes(int H, int G) {
  std::vector<int> s;
  if (H <= G) return {H};
  const int half = (G + 1) / 2;
  s.push_back(half);
  int rem = H - half;
  while (rem > G + half) {
    s.push_back(G);
    rem -= G;
  }
  if (rem > G) {
    s.push_back(rem - half);
    s.push_back(half);
  } else {
    s.push_back(rem);
  }
  return s;
}

struct Events {
  cudaEvent_t entry = nullptr, qkv[2] = {}, h2d[2] = {}, comp[2] = {}, d2h[2] = {};
  bool ok = true;
  Events() {
    ok = cudaEventCreateWithFlags(&entry, cudaEventDisableTiming) == cudaSuccess;
    for (int s = 0; s < 2 && ok; ++s)
      ok = cudaEventCreateWithFlags(&qkv[s], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&h2d[s], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&comp[s], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&d2h[s], cudaEventDisableTiming) == cudaSuccess;
  }
  // Destroying an event whose work is still queued is allowed: its resources
  // are released once the device has passed it.
  ~Events() {
    if (entry) cudaEventDestroy(entry);
    for (int s = 0; s < 2; ++s) {
      if (qkv[s]) cudaEventDestroy(qkv[s]);
      if (h2d[s]) cudaEventDestroy(h2d[s]);
      if (comp[s]) cudaEventDestroy(comp[s]);
      if (d2h[s]) cudaEventDestroy(d2h[s]);
    }
  }
};

// One head slice of a (B,T,H,d) host tensor <-> a contiguous (B,T,Gg,d) device buffer.
cudaError_t copy_slice(void* dst, const void* src, int d, int h0, int Gg, int H, size_t rows,
                       bool to_device, cudaStream_t s) {
  const size_t width = (size_t)Gg * d * 2, host_pitch = (size_t)H * d * 2;
  if (to_device) {
    const char* hsrc = static_cast<const char*>(src) + (size_t)h0 * d * 2;
    return cudaMemcpy2DAsync(dst, width, hsrc, host_pitch, width, rows, cudaMemcpyHostToDevice, s);
  }
  char* hdst = static_cast<char*>(dst) + (size_t)h0 * d * 2;
  return cudaMemcpy2DAsync(hdst, host_pitch, src, width, width, rows, cudaMemcpyDeviceToHost, s);
}

}  // namespace

extern "C" {

size_t attn_step_host_scratch_size(int B, int H, int T, int dqk, int dv, int heads_per_group,
                                   int deterministic) {
  if (B <= 0 || H <= 0 || T <= 0 || heads_per_group < 0) return 0;
  if (attn_bwd_workspace_size(B, 1, T, T, dqk, dv, 0, deterministic) == 0) return 0;
  const int G = pick_group(H, heads_per_group);
  return 2 * set_layout(B, G, T, dqk, dv, deterministic).bytes + r256((size_t)H * sizeof(int));
}

int attn_step_host(const void* q, const void* k, const void* v, const void* dO, void* o,
                   void* dq, void* dk, void* dv_out, int B, int H, int T, int dqk, int dv,
                   int causal, float scale, int deterministic, int heads_per_group,
                   void* scratch, size_t scratch_bytes, void* stream, void* stream2,
                   void* h2d_stream, void* d2h_stream) {
  if (!q || !k || !v || !dO || !dq || !dk || !dv_out || !scratch) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(scratch) & 255u) || heads_per_group < 0)
    return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || T <= 0) return ATTN_ERR_INVALID_ARG;
  const size_t need = attn_step_host_scratch_size(B, H, T, dqk, dv, heads_per_group, deterministic);
  if (need == 0) return ATTN_ERR_UNSUPPORTED;
  if (scratch_bytes < need) return ATTN_ERR_WORKSPACE_TOO_SMALL;

  const int G = pick_group(H, heads_per_group);
  const std::vector<int> sizes = group_sizes(H, G);
  const int ngroups = (int)sizes.size();
  const SetLayout L = set_layout(B, G, T, dqk, dv, deterministic);
  const size_t rows = (size_t)B * T;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // set s computes on css[s]: with two streams one group's kernels can fill
  // the SMs that the previous group's last work items leave idle
  const cudaStream_t css[2] = {cs, stream2 ? static_cast<cudaStream_t>(stream2) : cs};
  cudaStream_t hs = h2d_stream ? static_cast<cudaStream_t>(h2d_stream) : cs;
  cudaStream_t ds = d2h_stream ? static_cast<cudaStream_t>(d2h_stream) : cs;

  int* status = reinterpret_cast<int*>(static_cast<char*>(scratch) + 2 * L.bytes);
  Events ev;
  if (!ev.ok) return ATTN_ERR_CUDA;
  // the copy streams start after whatever the caller queued before this call
  if (cudaEventRecord(ev.entry, cs) != cudaSuccess ||
      cudaStreamWaitEvent(hs, ev.entry, 0) != cudaSuccess ||
      cudaStreamWaitEvent(ds, ev.entry, 0) != cudaSuccess ||
      cudaStreamWaitEvent(css[1], ev.entry, 0) != cudaSuccess)
    return ATTN_ERR_CUDA;

  for (int g = 0, h0 = 0; g < ngroups; h0 += sizes[g], ++g) {
    const int s = g & 1;
    const int Gg = sizes[g];
    char* base = static_cast<char*>(scratch) + s * L.bytes;
    void *q_d = base + L.q, *k_d = base + L.k, *v_d = base + L.v, *do_d = base + L.dO;
    void* o_d = base + L.o;
    float* lse = reinterpret_cast<float*>(base + L.lse);
    void *gq = base + L.dq, *gk = base + L.dk, *gv = base + L.dv;
    void* ws = base + L.ws;
    // stage 1: inputs (after the kernels of group g-2 are done with this set);
    // q, k, v first: the forward needs only those, dO travels while it runs
    if (g >= 2 && cudaStreamWaitEvent(hs, ev.comp[s], 0) != cudaSuccess) return ATTN_ERR_CUDA;
    if (copy_slice(q_d, q, dqk, h0, Gg, H, rows, true, hs) ||
        copy_slice(k_d, k, dqk, h0, Gg, H, rows, true, hs) ||
        copy_slice(v_d, v, dv, h0, Gg, H, rows, true, hs) ||
        cudaEventRecord(ev.qkv[s], hs) != cudaSuccess ||
        copy_slice(do_d, dO, dv, h0, Gg, H, rows, true, hs) ||
        cudaEventRecord(ev.h2d[s], hs) != cudaSuccess)
      return ATTN_ERR_CUDA;
    // stage 2: kernels (after the inputs, and after group g-2's results left)
    cudaStream_t c = css[s];
    if (cudaStreamWaitEvent(c, ev.qkv[s], 0) != cudaSuccess ||
        (g >= 2 && cudaStreamWaitEvent(c, ev.d2h[s], 0) != cudaSuccess))
      return ATTN_ERR_CUDA;
    int rc = attn_fwd(q_d, k_d, v_d, o_d, lse, B, Gg, T, T, dqk, dv, causal, scale, nullptr,
                      ATTN_LAYOUT_BTHD, c);
    if (rc) return rc;
    if (cudaStreamWaitEvent(c, ev.h2d[s], 0) != cudaSuccess) return ATTN_ERR_CUDA;
    rc = attn_bwd(q_d, k_d, v_d, o_d, do_d, lse, gq, gk, gv, B, Gg, T, T, dqk, dv, causal, scale,
                  nullptr, ATTN_LAYOUT_BTHD, deterministic, ws, L.ws_bytes, c);
    if (rc) return rc;
    // keep this group's device status: the next backward on the set resets it
    if (cudaMemcpyAsync(status + g, ws, sizeof(int), cudaMemcpyDeviceToDevice, c) != cudaSuccess ||
        cudaEventRecord(ev.comp[s], c) != cudaSuccess)
      return ATTN_ERR_CUDA;
    // stage 3: results back to the host
    if (cudaStreamWaitEvent(ds, ev.comp[s], 0) != cudaSuccess) return ATTN_ERR_CUDA;
    if (copy_slice(dq, gq, dqk, h0, Gg, H, rows, false, ds) ||
        copy_slice(dk, gk, dqk, h0, Gg, H, rows, false, ds) ||
        copy_slice(dv_out, gv, dv, h0, Gg, H, rows, false, ds) ||
        (o && copy_slice(o, o_d, dv, h0, Gg, H, rows, false, ds)) ||
        cudaEventRecord(ev.d2h[s], ds) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  for (int s = 0; s < std::min(ngroups, 2); ++s)
    if (cudaStreamWaitEvent(cs, ev.d2h[s], 0) != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

int attn_step_host_status(const void* scratch, int B, int H, int T, int dqk, int dv,
                          int heads_per_group, int deterministic, void* stream) {
  if (!scratch) return ATTN_ERR_INVALID_ARG;
  if (attn_step_host_scratch_size(B, H, T, dqk, dv, heads_per_group, deterministic) == 0)
    return ATTN_ERR_INVALID_ARG;
  const int G = pick_group(H, heads_per_group);
  const int ngroups = (int)group_sizes(H, G).size();
  const SetLayout L = set_layout(B, G, T, dqk, dv, deterministic);
  int rc = attn_fwd_status(stream);  // synchronises the stream
  if (rc != ATTN_OK) return rc;
  std::vector<int> st(ngroups, 0);
  const char* words = static_cast<const char*>(scratch) + 2 * L.bytes;
  if (cudaMemcpy(st.data(), words, ngroups * sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  for (int g = 0; g < ngroups; ++g)
    if (st[g] != ATTN_OK) return st[g];
  return ATTN_OK;
}

}  // extern "C"
