// attn_api.cu — the C ABI of include/attn.h: argument validation, layouts,
// workspace carving, variable-length schedule tables, TMA tensor maps and the
// launches.  Everything here is host code; all arithmetic runs in the kernels
// of attn_fwd.cu and attn_bwd.cu.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/attn.h"
#include "attn_internal.h"
#include "tmap.h"

using namespace attn;

namespace {

constexpr float kLog2e = 1.4426950408889634f;
// Whether the library's choice for eligible backward calls is the CTA-pair
// main kernel.
constexpr bool kPairByDefault = false;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_dims(int dqk, int dv) {
  return (dqk == 64 && dv == 64) || (dqk == 128 && dv == 128) || (dqk == 192 && dv == 128);
}

int num_sms_current() {
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  std::lock_guard<std::mutex> g(mu);
  if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    cache[dev] = n;
  }
  return cache[dev];
}

// Common shape checks of the forward and backward entry points.  cu / cuk:
// query / key offsets of a variable-length batch (cuk == cu when the keys
// share the queries' offsets).  Returns ATTN_OK or an error.
int check_shape(int B, int H, int Tq, int Tk, int dqk, int dv, int causal, const int* cu,
                const int* cuk, int layout, int wl = -1, int wr = -1) {
  if (wl < -1 || wr < -1) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || Tq <= 0 || Tk <= 0) return ATTN_ERR_INVALID_ARG;
  if (layout != ATTN_LAYOUT_BTHD && layout != ATTN_LAYOUT_PACKED_QKV) return ATTN_ERR_INVALID_ARG;
  if (!supported_dims(dqk, dv)) return ATTN_ERR_UNSUPPORTED;
  if (layout == ATTN_LAYOUT_PACKED_QKV && (dqk != dv || Tq != Tk || cu != cuk))
    return ATTN_ERR_UNSUPPORTED;
  if (cu == nullptr && cuk != nullptr) return ATTN_ERR_INVALID_ARG;
  if (cu != nullptr) {
    if (B > ATTN_MAX_VARLEN_SEQS) return ATTN_ERR_UNSUPPORTED;
    if (cu[0] != 0 || cu[B] != Tq || cuk[0] != 0 || cuk[B] != Tk) return ATTN_ERR_INVALID_ARG;
    for (int b = 0; b < B; ++b) {
      const int lq = cu[b + 1] - cu[b], lk = cuk[b + 1] - cuk[b];
      if (lq < 0 || lk < 0) return ATTN_ERR_INVALID_ARG;
      // queries need keys; a causal or windowed sequence needs Lq <= Lk
      // (its queries are the last Lq key positions)
      if (lq > 0 && lk == 0) return ATTN_ERR_INVALID_ARG;
      if ((causal || wl >= 0 || wr >= 0) && lq > lk) return ATTN_ERR_UNSUPPORTED;
    }
  } else {
    // causal (or a local window) with fewer queries than keys aligns the
    // queries with the last Tq keys; more queries than keys would leave rows
    // with no visible key
    if ((causal || wl >= 0 || wr >= 0) && Tq > Tk) return ATTN_ERR_UNSUPPORTED;
    if ((int64_t)B * Tq > INT32_MAX || (int64_t)B * Tk > INT32_MAX) return ATTN_ERR_UNSUPPORTED;
  }
  // every row of every tensor must fit the 32-bit coordinates of the TMA maps
  if ((int64_t)H * 3 * dqk > (1 << 20)) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

// Sequences by work, Lq * Lk, most first (ties: lower index first); with
// shared offsets (cuk == cu) that is longest first.
int order_impl(const int* cu, const int* cuk, int nseq, int* order) {
  if (cu == nullptr || cuk == nullptr || order == nullptr || nseq <= 0 ||
      nseq > ATTN_MAX_VARLEN_SEQS)
    return ATTN_ERR_INVALID_ARG;
  for (int b = 0; b < nseq; ++b) {
    if (cu[b + 1] < cu[b] || cuk[b + 1] < cuk[b]) return ATTN_ERR_INVALID_ARG;
    order[b] = b;
  }
  auto work = [cu, cuk](int b) {
    return (int64_t)(cu[b + 1] - cu[b]) * (int64_t)(cuk[b + 1] - cuk[b]);
  };
  std::stable_sort(order, order + nseq, [&](int a, int b) { return work(a) > work(b); });
  return ATTN_OK;
}

// Kinds of schedule table: forward items, backward items (key tiles), backward
// items on CTA pairs (pairs of key tiles).
enum TableKind { kFwdTable = 0, kBwdTable = 1, kBwdPairTable = 2 };

// Variable-length tables: sequences by work; items per sequence are (its
// 256-row query units (forward), kv-tiles or kv-tile pairs (backward)) x H;
// q-tiles numbered sequence by sequence.
void build_tables(const int* cu, const int* cuk, int nseq, int H, int kind, VarlenTables* t,
                  int* n_items, int* n_qtiles) {
  std::memset(t, 0, sizeof(*t));
  for (int b = 0; b <= nseq; ++b) {
    t->cu[b] = cu[b];
    t->cuk[b] = cuk[b];
  }
  order_impl(cu, cuk, nseq, t->order);
  int acc = 0;
  for (int k = 0; k < nseq; ++k) {
    t->item_start[k] = acc;
    const int s = t->order[k];
    const int lq = cu[s + 1] - cu[s], lk = cuk[s + 1] - cuk[s];
    acc += (kind == kFwdTable ? cdiv(lq, kFwdRows)
                              : (kind == kBwdTable ? cdiv(lk, kTile) : cdiv(lk, 2 * kTile))) * H;
  }
  t->item_start[nseq] = acc;
  *n_items = acc;
  int tiles = 0;
  for (int s = 0; s < nseq; ++s) {
    t->tile_start[s] = tiles;
    tiles += cdiv(cu[s + 1] - cu[s], kTile);
  }
  t->tile_start[nseq] = tiles;
  *n_qtiles = tiles;
}

// Host-side cache of what every call would otherwise rebuild: the TMA tensor
// maps (keyed by the base pointer and every encoding parameter) and the
// variable-length schedule tables (keyed by the offsets' contents, the head
// count and the kernel).  The cuDNN graph of "ops(8)..." §1.3 is built once
// and executed many times; this is the same idea for the library's host work.
// Least recently used entries are replaced; one mutex guards both caches.
class HostCache {
 public:
  bool map(CUtensorMap* out, const void* base, int64_t d, int64_t heads, int64_t rows,
           int64_t head_stride, int64_t row_stride, uint32_t box_rows) {
    const MapKey key{base, d, heads, rows, head_stride, row_stride, box_rows};
    std::lock_guard<std::mutex> g(mu_);
    MapEntry* victim = &maps_[0];
    for (MapEntry& e : maps_) {
      if (e.used != 0 && std::memcmp(&e.key, &key, sizeof(key)) == 0) {
        e.used = ++clock_;
        *out = e.map;
        ++stats_[1];
        return true;
      }
      if (e.used < victim->used) victim = &e;
    }
    if (!make_panel_map(&victim->map, base, d, heads, rows, head_stride, row_stride, box_rows)) {
      victim->used = 0;
      return false;
    }
    victim->key = key;
    victim->used = ++clock_;
    *out = victim->map;
    ++stats_[0];
    return true;
  }

  void tables(const int* cu, const int* cuk, int nseq, int H, int kind, VarlenTables* out,
              int* n_items, int* n_qtiles) {
    std::lock_guard<std::mutex> g(mu_);
    TabEntry* victim = &tabs_[0];
    for (TabEntry& e : tabs_) {
      if (e.used != 0 && e.nseq == nseq && e.H == H && e.kind == kind &&
          std::memcmp(e.t.cu, cu, (nseq + 1) * sizeof(int)) == 0 &&
          std::memcmp(e.t.cuk, cuk, (nseq + 1) * sizeof(int)) == 0) {
        e.used = ++clock_;
        std::memcpy(out, &e.t, sizeof(VarlenTables));
        *n_items = e.n_items;
        *n_qtiles = e.n_qtiles;
        ++stats_[3];
        return;
      }
      if (e.used < victim->used) victim = &e;
    }
    build_tables(cu, cuk, nseq, H, kind, &victim->t, &victim->n_items, &victim->n_qtiles);
    victim->nseq = nseq;
    victim->H = H;
    victim->kind = kind;
    victim->used = ++clock_;
    std::memcpy(out, &victim->t, sizeof(VarlenTables));
    *n_items = victim->n_items;
    *n_qtiles = victim->n_qtiles;
    ++stats_[2];
  }

  // tensor-map encodes, tensor-map hits, table builds, table hits
  void stats(long long* out) {
    std::lock_guard<std::mutex> g(mu_);
    for (int i = 0; i < 4; ++i) out[i] = stats_[i];
  }

 private:
  struct MapKey {
    const void* base;
    int64_t d, heads, rows, head_stride, row_stride;
    uint64_t box_rows;  // 64-bit so that the key has no padding bytes for memcmp
  };
  struct MapEntry {
    MapKey key;
    CUtensorMap map;
    uint64_t used = 0;  // 0: empty
  };
  struct TabEntry {
    int nseq = 0, H = 0;
    int kind = -1;
    int n_items = 0, n_qtiles = 0;
    VarlenTables t;
    uint64_t used = 0;
  };
  std::mutex mu_;
  MapEntry maps_[64];
  TabEntry tabs_[8];
  uint64_t clock_ = 0;
  long long stats_[4] = {0, 0, 0, 0};
};

HostCache& host_cache() {
  static HostCache* c = new HostCache();  // never destroyed: calls may come during exit
  return *c;
}

struct Layout {
  int64_t q_row, k_row, v_row;   // element distance between token rows of q / k / v
  int64_t o_row;                 // ... of o and dO
  int64_t g_q_row, g_k_row, g_v_row;  // ... of dq / dk / dv
};

Layout make_layout(int layout, int H, int dqk, int dv) {
  Layout L;
  if (layout == ATTN_LAYOUT_PACKED_QKV) {
    const int64_t r = 3ll * H * dqk;
    L.q_row = L.k_row = L.v_row = r;
    L.g_q_row = L.g_k_row = L.g_v_row = r;
  } else {
    L.q_row = L.k_row = L.g_q_row = L.g_k_row = (int64_t)H * dqk;
    L.v_row = L.g_v_row = (int64_t)H * dv;
  }
  L.o_row = (int64_t)H * dv;
  return L;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsSizes {
  size_t header, sem, stat, acc, total;
};

WsSizes ws_sizes(int n_qtiles, int H, int dqk) {
  WsSizes w;
  w.header = 256;
  w.sem = round256((size_t)n_qtiles * H * 2 * sizeof(int));
  w.stat = round256((size_t)n_qtiles * H * kTile * sizeof(float));
  w.acc = round256((size_t)n_qtiles * H * kTile * dqk * sizeof(float));
  w.total = w.header + w.sem + 2 * w.stat + w.acc;
  return w;
}

int qtiles_bound(int B, int Tq, bool varlen) {
  return varlen ? cdiv(Tq, kTile) + B : B * cdiv(Tq, kTile);
}

int cuda_err(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

// Block-mask fields of the kernels' shape (mask may be null).  Returns
// ATTN_OK or ATTN_ERR_INVALID_ARG.
int set_block_mask(SeqShape* sh, const unsigned char* mask, int mask_batches, int mask_heads,
                   int B, int H, int Tq, int Tk, const int* cu, const int* cuk) {
  sh->blk = nullptr;
  sh->blk_bstride = sh->blk_hstride = 0;
  sh->blk_nk = 0;
  if (mask == nullptr) return ATTN_OK;
  if ((mask_batches != 1 && mask_batches != B) || (mask_heads != 1 && mask_heads != H))
    return ATTN_ERR_INVALID_ARG;
  int nq = cdiv(Tq, kTile), nk = cdiv(Tk, kTile);
  if (cu != nullptr) {  // blocks of the longest sequence (queries, keys)
    int lq = 0, lk = 0;
    for (int b = 0; b < B; ++b) {
      lq = std::max(lq, cu[b + 1] - cu[b]);
      lk = std::max(lk, cuk[b + 1] - cuk[b]);
    }
    nq = cdiv(lq, kTile);
    nk = cdiv(lk, kTile);
  }
  sh->blk = mask;
  sh->blk_nk = nk;
  sh->blk_hstride = mask_heads == 1 ? 0 : (int64_t)nq * nk;
  sh->blk_bstride = mask_batches == 1 ? 0 : (int64_t)mask_heads * nq * nk;
  return ATTN_OK;
}

// Which backward main kernel runs when the CTA-pair kernel can (0: the
// library's choice, 1: one CTA per key tile, 2: CTA pairs).
std::atomic<int> g_bwd_variant{0};

// Host-side fault injection (tests only): added to every ordered-dQ wait
// target of deterministic backward calls, so that the wait can never succeed.
std::atomic<int> g_sem_bias{0};

// Optional CUDA events recorded around the backward main kernel (benchmark
// instrumentation; null = off).
std::atomic<void*> g_prof_start{nullptr};
std::atomic<void*> g_prof_stop{nullptr};
// ... and around the preprocess and the dQ conversion kernels
std::atomic<void*> g_prof_aux[4] = {{nullptr}, {nullptr}, {nullptr}, {nullptr}};

}  // namespace

extern "C" {

const char* attn_strerror(int code) {
  switch (code) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device wait timed out";
    case ATTN_ERR_INTERNAL: return "internal kernel set-up error";
    case ATTN_ERR_SCRATCH_TOO_SMALL: return "problem needs more than the built-in 32 MiB scratch";
    default: return "unknown error";
  }
}

int attn_varlen_order(const int* cu_seqlens, int nseq, int* order_out) {
  return order_impl(cu_seqlens, cu_seqlens, nseq, order_out);
}

size_t attn_bwd_workspace_size(int B, int H, int Tq, int Tk, int dqk, int dv, int varlen,
                               int deterministic) {
  (void)deterministic;
  (void)Tk;
  if (B <= 0 || H <= 0 || Tq <= 0 || !supported_dims(dqk, dv)) return 0;
  return ws_sizes(qtiles_bound(B, Tq, varlen != 0), H, dqk).total;
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int Tq, int Tk, int dqk, int dv, int causal, float scale, const int* cu_seqlens,
             int layout, void* stream) {
  return attn_fwd_window(q, k, v, o, lse, B, H, Tq, Tk, dqk, dv, causal, -1, -1, scale,
                         cu_seqlens, layout, stream);
}

int attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                    int H, int Tq, int Tk, int dqk, int dv, int causal, int window_left,
                    int window_right, float scale, const int* cu_seqlens, int layout,
                    void* stream) {
  return attn_fwd_ex(q, k, v, o, lse, B, H, Tq, Tk, dqk, dv, causal, window_left, window_right,
                     nullptr, 1, 1, scale, cu_seqlens, nullptr, layout, stream);
}

int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int Tq, int Tk, int dqk, int dv, int causal, int window_left, int window_right,
                const unsigned char* block_mask, int mask_batches, int mask_heads, float scale,
                const int* cu_seqlens_q, const int* cu_seqlens_k, int layout, void* stream) {
  const int* cu_seqlens = cu_seqlens_q;
  const int* cuk = cu_seqlens_k != nullptr ? cu_seqlens_k : cu_seqlens_q;
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;  // running max assumes s > 0
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return ATTN_ERR_INVALID_ARG;
  int rc = check_shape(B, H, Tq, Tk, dqk, dv, causal, cu_seqlens, cuk, layout, window_left,
                       window_right);
  if (rc) return rc;
  if (block_mask != nullptr && ((mask_batches != 1 && mask_batches != B) ||
                                (mask_heads != 1 && mask_heads != H)))
    return ATTN_ERR_INVALID_ARG;

  FwdLaunch L;
  std::memset(&L, 0, sizeof(L));
  static thread_local VarlenTables tables;
  const bool varlen = cu_seqlens != nullptr;
  const Layout lay = make_layout(layout, H, dqk, dv);
  const int64_t rows_q = varlen ? Tq : (int64_t)B * Tq;
  const int64_t rows_k = varlen ? Tk : (int64_t)B * Tk;
  HostCache& hc = host_cache();
  if (!hc.map(&L.tm_q, q, dqk, H, rows_q, dqk, lay.q_row, kTile) ||
      !hc.map(&L.tm_k, k, dqk, H, rows_k, dqk, lay.k_row, kTile) ||
      !hc.map(&L.tm_v, v, dv, H, rows_k, dv, lay.v_row, kTile))
    return ATTN_ERR_CUDA;
  L.sh.nseq = B;
  L.sh.H = H;
  L.sh.varlen = varlen ? 1 : 0;
  L.sh.Tq = Tq;
  L.sh.Tk = Tk;
  L.sh.nq_tiles = cdiv(Tq, kTile);
  L.sh.nk_tiles = cdiv(Tk, kTile);
  L.sh.nq_units = cdiv(Tq, kFwdRows);
  L.sh.causal = causal ? 1 : 0;
  L.sh.band_off = varlen ? 0 : Tk - Tq;
  L.sh.wl = window_left;
  L.sh.wr = causal ? 0 : window_right;
  L.sh.descending = 0;
  // Rank-major forward order when every head's K and V fit in L2 together
  // (measured: the GPT-2-shaped layer, 25 MB of K and V, 8 % faster than
  // head-major); head-major keeps a few heads' K and V in L2 otherwise.
  constexpr int64_t kL2FitBytes = 48ll << 20;
  L.sh.rank_major = !varlen && (int64_t)B * Tk * H * (dqk + dv) * 2 <= kL2FitBytes ? 1 : 0;
  rc = set_block_mask(&L.sh, block_mask, mask_batches, mask_heads, B, H, Tq, Tk, cu_seqlens,
                      cuk);
  if (rc) return rc;
  if (varlen) {
    int n_items = 0, n_qt = 0;
    hc.tables(cu_seqlens, cuk, B, H, kFwdTable, &tables, &n_items, &n_qt);
    L.sh.n_items = n_items;
    L.tables = &tables;
    L.lse_head_stride = Tq;
    L.lse_seq_stride = 0;
  } else {
    L.sh.n_items = B * H * L.sh.nq_units;
    L.tables = nullptr;
    L.lse_head_stride = Tq;
    L.lse_seq_stride = (int64_t)H * Tq;
  }
  if (L.sh.n_items == 0) return ATTN_OK;
  L.o = o;
  L.lse = lse;
  L.o_row_stride = lay.o_row;
  L.scale_log2 = scale * kLog2e;
  L.status = fwd_status_ptr();
  if (!L.status) return ATTN_ERR_CUDA;
  // work-item counters of its own (the previous kernel on them left them at zero)
  static std::atomic<unsigned> next_claim{0};
  L.claim = fwd_claim_ptr((int)(next_claim.fetch_add(1) % kFwdClaimSlots));
  if (!L.claim) return ATTN_ERR_CUDA;
  const int sms = num_sms_current();
  if (sms <= 0) return ATTN_ERR_CUDA;
  L.grid = std::min(L.sh.n_items, sms);
  L.stream = static_cast<cudaStream_t>(stream);
  return cuda_err(launch_fwd(L, dqk, dv));
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
             const float* lse, void* dq, void* dk, void* dv_out, int B, int H, int Tq, int Tk,
             int dqk, int dv, int causal, float scale, const int* cu_seqlens, int layout,
             int deterministic, void* workspace, size_t workspace_bytes, void* stream) {
  return attn_bwd_window(q, k, v, o, dO, lse, dq, dk, dv_out, B, H, Tq, Tk, dqk, dv, causal, -1,
                         -1, scale, cu_seqlens, layout, deterministic, workspace,
                         workspace_bytes, stream);
}

int attn_bwd_window(const void* q, const void* k, const void* v, const void* o, const void* dO,
                    const float* lse, void* dq, void* dk, void* dv_out, int B, int H, int Tq,
                    int Tk, int dqk, int dv, int causal, int window_left, int window_right,
                    float scale, const int* cu_seqlens, int layout, int deterministic,
                    void* workspace, size_t workspace_bytes, void* stream) {
  return attn_bwd_ex(q, k, v, o, dO, lse, dq, dk, dv_out, B, H, Tq, Tk, dqk, dv, causal,
                     window_left, window_right, nullptr, 1, 1, scale, cu_seqlens, nullptr, layout,
                     deterministic, workspace, workspace_bytes, stream);
}

int attn_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dO,
                const float* lse, void* dq, void* dk, void* dv_out, int B, int H, int Tq, int Tk,
                int dqk, int dv, int causal, int window_left, int window_right,
                const unsigned char* block_mask, int mask_batches, int mask_heads, float scale,
                const int* cu_seqlens_q, const int* cu_seqlens_k, int layout, int deterministic,
                void* workspace, size_t workspace_bytes, void* stream) {
  const int* cu_seqlens = cu_seqlens_q;
  const int* cuk = cu_seqlens_k != nullptr ? cu_seqlens_k : cu_seqlens_q;
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv_out || !workspace)
    return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv_out) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_ERR_INVALID_ARG;
  int rc = check_shape(B, H, Tq, Tk, dqk, dv, causal, cu_seqlens, cuk, layout, window_left,
                       window_right);
  if (rc) return rc;
  if (block_mask != nullptr && ((mask_batches != 1 && mask_batches != B) ||
                                (mask_heads != 1 && mask_heads != H)))
    return ATTN_ERR_INVALID_ARG;
  const bool varlen = cu_seqlens != nullptr;
  if (workspace_bytes < attn_bwd_workspace_size(B, H, Tq, Tk, dqk, dv, varlen, deterministic))
    return ATTN_ERR_WORKSPACE_TOO_SMALL;

  BwdLaunch L;
  std::memset(&L, 0, sizeof(L));
  static thread_local VarlenTables tables;
  const Layout lay = make_layout(layout, H, dqk, dv);
  const int64_t rows_q = varlen ? Tq : (int64_t)B * Tq;
  const int64_t rows_k = varlen ? Tk : (int64_t)B * Tk;
  HostCache& hc = host_cache();
  if (!hc.map(&L.tm_q, q, dqk, H, rows_q, dqk, lay.q_row, kTile) ||
      !hc.map(&L.tm_k, k, dqk, H, rows_k, dqk, lay.k_row, kTile) ||
      !hc.map(&L.tm_v, v, dv, H, rows_k, dv, lay.v_row, kTile) ||
      !hc.map(&L.tm_do, dO, dv, H, rows_q, dv, lay.o_row, kTile))
    return ATTN_ERR_CUDA;
  L.sh.nseq = B;
  L.sh.H = H;
  L.sh.varlen = varlen ? 1 : 0;
  L.sh.Tq = Tq;
  L.sh.Tk = Tk;
  L.sh.nq_tiles = cdiv(Tq, kTile);
  L.sh.nk_tiles = cdiv(Tk, kTile);
  L.sh.causal = causal ? 1 : 0;
  L.sh.band_off = varlen ? 0 : Tk - Tq;
  L.sh.wl = window_left;
  L.sh.wr = causal ? 0 : window_right;
  L.sh.descending = deterministic ? 1 : 0;
  rc = set_block_mask(&L.sh, block_mask, mask_batches, mask_heads, B, H, Tq, Tk, cu_seqlens,
                      cuk);
  if (rc) return rc;
  const int sms = num_sms_current();
  if (sms <= 0) return ATTN_ERR_CUDA;
  // The CTA-pair main kernel covers d = 128 without a block mask or a left
  // window edge (causal, non-causal, right-bounded bands; fixed or variable
  // length), on at least two SMs.
  const int variant = g_bwd_variant.load();
  const bool pair_ok = dqk == 128 && dv == 128 && block_mask == nullptr && window_left < 0 &&
                       sms >= 2;
  L.pair = pair_ok && variant != 1 && (variant == 2 || kPairByDefault) ? 1 : 0;
  if (L.pair && (!hc.map(&L.tm_q64, q, dqk, H, rows_q, dqk, lay.q_row, 64) ||
                 !hc.map(&L.tm_do64, dO, dv, H, rows_q, dv, lay.o_row, 64)))
    return ATTN_ERR_CUDA;
  int n_qtiles;
  if (varlen) {
    int n_items = 0;
    hc.tables(cu_seqlens, cuk, B, H, L.pair ? kBwdPairTable : kBwdTable, &tables, &n_items,
              &n_qtiles);
    L.sh.n_items = n_items;
    L.tables = &tables;
    L.lse_head_stride = Tq;
    L.lse_seq_stride = 0;
  } else {
    L.sh.n_items = B * H * (L.pair ? cdiv(L.sh.nk_tiles, 2) : L.sh.nk_tiles);
    n_qtiles = B * L.sh.nq_tiles;
    L.tables = nullptr;
    L.lse_head_stride = Tq;
    L.lse_seq_stride = (int64_t)H * Tq;
  }
  if (L.sh.n_items == 0) return ATTN_OK;
  // carve the workspace (sizes from the bound, offsets fixed by the query)
  const WsSizes w = ws_sizes(qtiles_bound(B, Tq, varlen), H, dqk);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  L.ws.header = reinterpret_cast<int*>(base);
  L.ws.sem = reinterpret_cast<int*>(base + w.header);
  L.ws.nlse2 = reinterpret_cast<float*>(base + w.header + w.sem);
  L.ws.ndsum = reinterpret_cast<float*>(base + w.header + w.sem + w.stat);
  L.ws.dq_acc = reinterpret_cast<float*>(base + w.header + w.sem + 2 * w.stat);
  L.o = o;
  L.dout = dO;
  L.lse = lse;
  L.dq = dq;
  L.dk = dk;
  L.dv = dv_out;
  L.q_row_stride = lay.q_row;
  L.k_row_stride = lay.k_row;
  L.v_row_stride = lay.v_row;
  L.o_row_stride = lay.o_row;
  L.do_row_stride = lay.o_row;
  L.dq_row_stride = lay.g_q_row;
  L.dk_row_stride = lay.g_k_row;
  L.dv_row_stride = lay.g_v_row;
  L.scale = scale;
  L.scale_log2 = scale * kLog2e;
  L.n_qtiles = n_qtiles;
  L.deterministic = deterministic ? 1 : 0;
  L.sem_bias = g_sem_bias.load();
  L.prof_start = static_cast<cudaEvent_t>(g_prof_start.load());
  L.prof_stop = static_cast<cudaEvent_t>(g_prof_stop.load());
  for (int e = 0; e < 4; ++e) L.prof_aux[e] = static_cast<cudaEvent_t>(g_prof_aux[e].load());
  L.num_sms = sms;
  L.grid = L.pair ? 2 * std::min(L.sh.n_items, sms / 2) : std::min(L.sh.n_items, sms);
  L.stream = static_cast<cudaStream_t>(stream);
  return cuda_err(launch_bwd(L, dqk, dv));
}

int attn_profile_main_kernel(void* event_start, void* event_stop) {
  if ((event_start == nullptr) != (event_stop == nullptr)) return ATTN_ERR_INVALID_ARG;
  g_prof_start.store(event_start);
  g_prof_stop.store(event_stop);
  return ATTN_OK;
}

int attn_profile_aux_kernels(void* pre_start, void* pre_stop, void* convert_start,
                             void* convert_stop) {
  void* ev[4] = {pre_start, pre_stop, convert_start, convert_stop};
  const bool any = ev[0] || ev[1] || ev[2] || ev[3];
  const bool all = ev[0] && ev[1] && ev[2] && ev[3];
  if (any && !all) return ATTN_ERR_INVALID_ARG;
  for (int e = 0; e < 4; ++e) g_prof_aux[e].store(ev[e]);
  return ATTN_OK;
}

int attn_debug_set_bwd_variant(int variant) {
  if (variant < 0 || variant > 2) return ATTN_ERR_INVALID_ARG;
  g_bwd_variant.store(variant);
  return ATTN_OK;
}

int attn_debug_cache_stats(long long* out4) {
  if (out4 == nullptr) return ATTN_ERR_INVALID_ARG;
  host_cache().stats(out4);
  return ATTN_OK;
}

int attn_debug_set_wait_bias(int bias) {
  g_sem_bias.store(bias);
  return ATTN_OK;
}

int attn_bwd_status(const void* workspace, void* stream) {
  if (!workspace) return ATTN_ERR_INVALID_ARG;
  int st = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&st, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
  return st;
}

int attn_fwd_status(void* stream) {
  int* p = fwd_status_ptr();
  if (!p) return ATTN_ERR_CUDA;
  int st = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&st, p, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (cudaMemsetAsync(p, 0, sizeof(int), s) != cudaSuccess) return ATTN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
  return st;
}

}  // extern "C"
