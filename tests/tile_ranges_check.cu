// Host-side exhaustive check of the band's tile ranges (attn_common.cuh),
// compiled and run by tests/test_tile_ranges.py (no GPU needed).
//
// For every shape tried, with the rows of a tile taken as the positions
// qt*128 .. qt*128+127 (padding rows follow the band like real ones):
//   (1) first_kvtile / last_kvtile of each q-tile are the smallest / largest
//       kv-tile holding a (query, key) pair of the band, and every kv-tile in
//       between holds one;
//   (2) the same for first_qtile / last_qtile of each kv-tile;
//   (3) kv-tile kt is in q-tile qt's range iff qt is in kt's range — the
//       deterministic dQ order relies on it (a kv-tile waits for the next
//       kv-tile above it in the q-tile's range, which must visit that q-tile).
#include <cstdio>
#include <cstdlib>
#include "../attention_backward_flashattention_gb300/csrc/attn_common.cuh"

using namespace attn;

static bool visible(int i, int j, int off, int wl, int wr) {
  return (wl < 0 || j >= i + off - wl) && (wr < 0 || j <= i + off + wr);
}

// any pair of the band in (q-tile qt, kv-tile kt); keys past Tk are not keys
static bool pair_in_band(int qt, int kt, int Tk, int off, int wl, int wr) {
  for (int i = qt * kTile; i < qt * kTile + kTile; ++i)
    for (int j = kt * kTile; j < kt * kTile + kTile && j < Tk; ++j)
      if (visible(i, j, off, wl, wr)) return true;
  return false;
}

int main() {
  unsigned seed = 12345;
  auto rnd = [&](int n) { seed = seed * 1103515245u + 12345u; return (int)((seed >> 8) % n); };
  const int wins[] = {-1, 0, 1, 5, 40, 127, 128, 129, 200, 255, 256, 300, 1000};
  long checked = 0, bad = 0;
  for (int c = 0; c < 3000; ++c) {
    const int Tk = 1 + rnd(1100);
    const bool causal = rnd(3) == 0;
    int wl = wins[rnd(13)], wr = wins[rnd(13)];
    if (causal) wr = 0;
    const bool banded = causal || wl >= 0 || wr >= 0;
    const int Tq = banded ? 1 + rnd(Tk) : 1 + rnd(1100);
    SeqShape sh{};
    sh.wl = wl;
    sh.wr = wr;
    sh.band_off = Tk - Tq;
    sh.varlen = (c & 1);  // both ways of reading the offset
    Item it{};
    it.band_off = Tk - Tq;
    const int nq = cdiv(Tq, kTile), nk = cdiv(Tk, kTile), off = Tk - Tq;
    for (int qt = 0; qt < nq; ++qt) {
      int lo = -1, hi = -1;
      for (int kt = 0; kt < nk; ++kt)
        if (pair_in_band(qt, kt, Tk, off, wl, wr)) { if (lo < 0) lo = kt; hi = kt; }
      const int f = first_kvtile(sh, it, qt), l = last_kvtile(sh, it, qt, nk);
      bool ok = lo < 0 ? (f > l) : (f == lo && l == hi);
      for (int kt = lo; ok && lo >= 0 && kt <= hi; ++kt) ok = pair_in_band(qt, kt, Tk, off, wl, wr);
      ++checked;
      if (!ok && bad++ < 10)
        printf("kv range: Tq=%d Tk=%d wl=%d wr=%d qt=%d: got [%d,%d] want [%d,%d]\n", Tq, Tk, wl,
               wr, qt, f, l, lo, hi);
    }
    for (int kt = 0; kt < nk; ++kt) {
      int lo = -1, hi = -1;
      for (int qt = 0; qt < nq; ++qt)
        if (pair_in_band(qt, kt, Tk, off, wl, wr)) { if (lo < 0) lo = qt; hi = qt; }
      const int f = first_qtile(sh, it, kt), l = last_qtile(sh, it, kt, nq);
      bool ok = lo < 0 ? (f > l) : (f == lo && l == hi);
      for (int qt = lo; ok && lo >= 0 && qt <= hi; ++qt) ok = pair_in_band(qt, kt, Tk, off, wl, wr);
      ++checked;
      if (!ok && bad++ < 10)
        printf("q range: Tq=%d Tk=%d wl=%d wr=%d kt=%d: got [%d,%d] want [%d,%d]\n", Tq, Tk, wl,
               wr, kt, f, l, lo, hi);
      for (int qt = 0; qt < nq; ++qt) {
        const bool a = kt >= first_kvtile(sh, it, qt) && kt <= last_kvtile(sh, it, qt, nk);
        const bool b = qt >= first_qtile(sh, it, kt) && qt <= last_qtile(sh, it, kt, nq);
        ++checked;
        if (a != b && bad++ < 10)
          printf("symmetry: Tq=%d Tk=%d wl=%d wr=%d qt=%d kt=%d: %d vs %d\n", Tq, Tk, wl, wr, qt,
                 kt, a, b);
      }
    }
  }
  printf("checked %ld, bad %ld\n", checked, bad);
  return bad == 0 ? 0 : 1;
}
