// attn_common.cuh — parameters and work decomposition shared by the forward
// and backward kernels.
//
// Token rows.  Every input is viewed as rows of tokens: a fixed-length batch
// (B, T, H, d) is the same memory as (B*T, H, d), and a variable-length batch
// is (sum T, H, d) with sequence s occupying rows cu[s] .. cu[s+1]-1.  The
// packed (B, T, 3, H, d) layout only changes the distance between rows.
//
// Tiles.  Queries and keys are cut into tiles of 128 consecutive rows of one
// sequence and one head.  A q-tile is the unit of the forward and of the dQ
// reduction; a kv-tile is the unit of the backward.  The last tile of a
// sequence may be ragged; rows past the sequence end are masked.
//
// Work items and their order (the scheduling the first page describes in
// §3.2 "确定性执行实现": CTA order swizzled over heads/batches for L2 reuse,
// longest-processing-time-first over batches, and shortest-first over causal
// kv-tiles for the deterministic dQ reduction):
//   forward   item = (sequence, head, 256-row unit m: two q-tiles), claimed
//             dynamically (a per-call counter): all units of one (sequence,
//             head) are consecutive, the longest causal row range first (m
//             descending), so one head's K and V stay in L2 while ~one SM count
//             of its units run, and the last items claimed are the shortest.
//             When every head's K and V fit in L2 together (fixed length), the
//             units go rank-major instead (longest of every head first), which
//             balances better when each CTA gets only a few items.
//   backward  item = (sequence, head, kv-tile n); all tiles of one (sequence,
//             head) are consecutive, so one head's Q, dO and fp32 dQ
//             accumulator stay in L2 while ~one SM count of its kv-tiles run.
//             Fast mode runs n ascending (the longest causal column range
//             first); deterministic mode runs n descending, which is also the
//             order in which each dQ tile receives its contributions, so a CTA
//             only ever waits on work that was claimed before its own.
//   Variable-length batches run sequence by sequence, most work (Lq * Lk) first.
#pragma once

#include <stdint.h>

namespace attn {

constexpr int kTile = 128;
constexpr int kFwdRows = 2 * kTile;  // query rows of one forward work item (two Q tiles)
constexpr int kMaxSeqs = 1024;  // sequences in one variable-length call
// Pacing of the backward's fp32 dQ reductions (fast mode): one thread's
// reductions of a dQ tile are spread over kRedSpread/256 of the previous
// q-tile step (the time between the two previous dQ tiles), with at most
// kRedPaceCap clocks between two of them.
constexpr int kRedPaceCap = 128;
constexpr long long kRedSpread = 205;

// Host-computed tables for variable-length batches (passed by value).
struct VarlenTables {
  int cu[kMaxSeqs + 1];          // token offset of each sequence's queries
  int cuk[kMaxSeqs + 1];         // ... and of its keys (equal to cu unless given apart)
  int order[kMaxSeqs];           // sequences, most work (Lq * Lk) first (ties: lower id first)
  int item_start[kMaxSeqs + 1];  // first work item of the k-th sequence in `order`
  int tile_start[kMaxSeqs + 1];  // first q-tile of sequence s in the workspace tile space
                                 // (item_start counts 256-row units in the forward)
};
struct NoTables {};

struct SeqShape {
  int nseq;        // B (number of sequences)
  int H;           // heads
  int varlen;      // 1: lengths come from VarlenTables
  int Tq, Tk;      // fixed-length sequence lengths (varlen: total token counts)
  int nq_tiles;    // fixed-length: ceil(Tq/128)
  int nk_tiles;    // fixed-length: ceil(Tk/128)
  int nq_units;    // fixed-length: ceil(Tq/256), forward work items per (b, h)
  int n_items;     // number of work items of the kernel
  int causal;
  // The band of visible keys: key j is visible to query i iff
  //   i + off - wl <= j <= i + off + wr   (wl, wr = -1: that side open)
  // causal is wr = 0; off = Lk - Lq of the sequence (the queries are the last
  // Lq positions of the key sequence), kept per item (Item::band_off);
  // band_off here is the fixed-length Tk - Tq.
  int band_off;
  int wl, wr;
  int descending;  // backward only: 1 = kv-tiles n descending (deterministic mode)
  int rank_major;  // forward, fixed length: 1 = units rank-major ((b, h) fastest)
  // Block mask (null: every tile pair in the band takes part).  Byte
  // [b][h][qt][kt] of a (mask batches, mask heads, q-tiles, kv-tiles) array;
  // a zero byte drops the pair (query tile qt, key tile kt) of sequence b,
  // head h.  A stride of 0 shares one mask over sequences or heads.
  const uint8_t* blk;
  int64_t blk_bstride, blk_hstride;  // bytes between sequences / heads
  int blk_nk;                        // kv-tiles per mask row
};

struct Item {
  int seq, head, tile;  // tile = q-tile (forward) or kv-tile (backward)
  int row0;             // first token row of the sequence's queries
  int krow0;            // first token row of its keys
  int Lq, Lk;           // sequence lengths (queries, keys)
  int band_off;         // Lk - Lq: query i sits at key position i + band_off
  int tile_base;        // first q-tile of this sequence in the workspace tile space
};

__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }

template <typename Tables>
__device__ __forceinline__ Item decode_item(const SeqShape& sh, const Tables& tb, int item,
                                            bool forward);

// Fixed length (items claimed dynamically): item / (units or kv-tiles per head)
// is the (b, h), the remainder the unit's or tile's rank.
template <>
__device__ __forceinline__ Item decode_item<NoTables>(const SeqShape& sh, const NoTables&,
                                                      int item, bool forward) {
  Item it;
  int bh, rank;
  if (forward) {  // 256-row units longest first; it.tile = unit
    if (sh.rank_major) {  // unit rank major, (b, h) fastest
      const int nbh = sh.nseq * sh.H;
      rank = item / nbh;
      bh = item - rank * nbh;
    } else {              // (b, h) major
      bh = item / sh.nq_units;
      rank = item - bh * sh.nq_units;
    }
    it.tile = sh.nq_units - 1 - rank;
  } else {        // (b, h) major, tile rank fastest
    bh = item / sh.nk_tiles;
    rank = item - bh * sh.nk_tiles;
    it.tile = sh.descending ? sh.nk_tiles - 1 - rank : rank;
  }
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

// Variable length: sequence-major in `order`; within a sequence as above.
template <>
__device__ __forceinline__ Item decode_item<VarlenTables>(const SeqShape& sh,
                                                          const VarlenTables& tb, int item,
                                                          bool forward) {
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
  // forward items: 256-row query units; backward items: kv-tiles
  const int nt = forward ? cdiv(it.Lq, kFwdRows) : cdiv(it.Lk, kTile);
  // head, then tile rank
  it.head = local / nt;
  const int rank = local - it.head * nt;
  if (forward) it.tile = nt - 1 - rank;
  else it.tile = sh.descending ? nt - 1 - rank : rank;
  it.tile_base = tb.tile_start[it.seq];
  return it;
}

// The band offset of the item's sequence, Lk - Lq.  Fixed-length items carry
// the kernel-wide Tk - Tq, so this folds to the kernel parameter there.
__host__ __device__ __forceinline__ int band_off(const SeqShape& sh, const Item& it) {
  return sh.varlen ? it.band_off : sh.band_off;
}

// Tile ranges of the band: q-tile qt sees kv-tiles first_kvtile .. last_kvtile,
// kv-tile kt is seen by q-tiles first_qtile .. last_qtile (a tile pair is in
// the band when any of its (query, key) pairs is).  Numerators of the clamped
// bounds may be negative; C++ division truncates toward zero, which the clamp
// to 0 (first_*) absorbs and last_qtile corrects.
__host__ __device__ __forceinline__ int first_kvtile(const SeqShape& sh, const Item& it, int qt) {
  return sh.wl >= 0 ? max(0, (qt * kTile + band_off(sh, it) - sh.wl) / kTile) : 0;
}
__host__ __device__ __forceinline__ int last_kvtile(const SeqShape& sh, const Item& it, int qt, int nk) {
  return sh.wr >= 0 ? min(nk - 1, (qt * kTile + kTile - 1 + band_off(sh, it) + sh.wr) / kTile)
                    : nk - 1;
}
__host__ __device__ __forceinline__ int first_qtile(const SeqShape& sh, const Item& it, int kt) {
  return sh.wr >= 0 ? max(0, (kt * kTile - band_off(sh, it) - sh.wr) / kTile) : 0;
}
__host__ __device__ __forceinline__ int last_qtile(const SeqShape& sh, const Item& it, int kt, int nq) {
  if (sh.wl < 0) return nq - 1;
  const int num = kt * kTile + kTile - 1 - band_off(sh, it) + sh.wl;
  return num < 0 ? -1 : min(nq - 1, num / kTile);
}

// Whether the block mask keeps the tile pair (q-tile qt, kv-tile kt) of the
// item's sequence and head (both tiles inside the sequence).
__device__ __forceinline__ bool tile_on(const SeqShape& sh, const Item& it, int qt, int kt) {
  return sh.blk == nullptr ||
         __ldg(sh.blk + it.seq * sh.blk_bstride + it.head * sh.blk_hstride +
               (int64_t)qt * sh.blk_nk + kt) != 0;
}

// First token row of the keys of a sequence.
__device__ __forceinline__ int key_row0(const SeqShape&, const Item& it) { return it.krow0; }

}  // namespace attn
