// Exhaustive check of the stream-K work schedule (dense_gemm_14_gb300/csrc/
// streamk.cuh) on the host: every (tile, k-block) is covered exactly once;
// PARTIAL segments come first and HEAD segments last in a worker's stream-K
// range; a HEAD's contributors cover the rest of its tile in order; the
// loaders' flat-iteration map agrees with the segment list.
#define __host__
#define __device__
#include "streamk.cuh"
#include <cstdio>
#include <vector>
using namespace gemm14;
int main() {
  int bad = 0;
  for (int tiles : {1, 2, 7, 128, 151, 152, 153, 288, 300, 1024, 2048, 396})
   for (int L : {1, 2, 17, 64, 96, 128})
    for (int G : {1, 2, 76, 152}) {
      for (bool ws : {false, true}) {
        StreamK sk = make_stream_k(tiles, L, G, ws);
        std::vector<int> cover((size_t)tiles * L, 0);
        int workers = ws && sk.dp_tiles < tiles ? sk.G : (tiles < G ? tiles : G);
        if (sk.G > G) { bad++; printf("more workers than allowed\n"); }
        for (int w = 0; w < sk.G; ++w) {
          if (sk.dp_tiles == 0 && sk.sk_start(w + 1) <= sk.sk_start(w)) { bad++; printf("empty stream-K range\n"); }
          long long it = 0;
          int n = sk.segments(w);
          if (w >= workers && n) { bad++; printf("idle worker has work\n"); }
          for (int i = 0; i < n; ++i) {
            int t, a, b, kind; sk.segment(w, i, t, a, b, kind);
            if (t < 0 || t >= tiles || a < 0 || b > L || a >= b) { bad++; printf("bad seg t=%d a=%d b=%d\n", t, a, b); continue; }
            if (kind == kSegPartial && i != sk.dp_count(w)) { bad++; printf("partial not first\n"); }
            if (kind == kSegHead && i != n - 1) { bad++; printf("head not last\n"); }
            for (int k = a; k < b; ++k) { cover[(size_t)t * L + k]++;
              int t2, k2; sk.iteration(w, it++, t2, k2); if (t2 != t || k2 != k) { bad++; printf("iter map mismatch\n"); } }
            if (kind == kSegHead) {  // contributors must cover [b, L) exactly, in order
              int pos = b; int c = w;
              while ((c = sk.next_contributor(c, t)) >= 0) {
                int t0, a0, b0, k0; sk.segment(c, sk.dp_count(c), t0, a0, b0, k0);
                if (t0 != t || a0 != pos || b0 <= a0 || k0 != kSegPartial) { bad++; printf("contrib mismatch\n"); break; }
                pos = b0;
              }
              if (pos != L) { bad++; printf("head coverage %d != %d (tiles %d L %d G %d)\n", pos, L, tiles, L, G); }
            }
          }
          if (it != sk.iterations(w)) { bad++; printf("iterations mismatch\n"); }
          // the decoded table gives the same segments and the same contributors
          SkTable tab; tab.fill(sk, w);
          if (tab.n_sk > kMaxSk) { bad++; printf("too many stream-K segments: %d\n", tab.n_sk); }
          if (tab.segments() != n) { bad++; printf("table segment count\n"); }
          for (int i = 0; i < n && tab.n_sk <= kMaxSk; ++i) {
            int t1, a1, b1, k1, t2, a2, b2, k2;
            sk.segment(w, i, t1, a1, b1, k1); tab.get(i, t2, a2, b2, k2);
            if (t1 != t2 || a1 != a2 || b1 != b2 || k1 != k2) { bad++; printf("table mismatch\n"); }
            if (k1 == kSegHead) {
              int last = w; for (int c = sk.next_contributor(w, t1); c >= 0; c = sk.next_contributor(c, t1)) last = c;
              if (last != tab.head_last) { bad++; printf("head_last mismatch\n"); }
              for (int c = w + 1; c <= last; ++c) if (sk.sk_start(c + 1) <= sk.sk_start(c)) { bad++; printf("empty contributor in range\n"); }
            }
          }
          // the loaders' cursor (the kernels use the table walk only when
          // tiles are split, the plain walk otherwise) visits the same k-blocks
          const bool split = sk.dp_tiles < sk.tiles;
          SegmentCursor cur;
          if (split) cur.start<true>(tab, w, sk.dp_count(w), L);
          else cur.start<false>(tab, w, sk.dp_count(w), L);
          for (long long j = 0; j < sk.iterations(w); ++j) {
            int t2, k2; sk.iteration(w, j, t2, k2);
            if (cur.tile != t2 || cur.kb != k2) { bad++; printf("cursor mismatch\n"); break; }
            if (split) cur.next<true>(tab, sk.G); else cur.next<false>(tab, sk.G);
          }
        }
        for (size_t x = 0; x < cover.size(); ++x) if (cover[x] != 1) { bad++; printf("cover %zu = %d (tiles %d L %d G %d ws %d)\n", x, cover[x], tiles, L, G, ws); break; }
      }
    }
  printf("bad = %d\n", bad);
  return bad != 0;
}
