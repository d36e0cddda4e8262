// streamk.cuh -- the work schedule shared by the persistent kernels: whole
// output tiles round-robin ("data-parallel"), then an even split of the
// remaining tiles' k-blocks over all workers ("stream-K").
//
// Flat iteration space: tile t, k-block kb -> t * L + kb (L k-blocks a tile).
// Tiles [0, dp_tiles) go whole to worker t % G. The k-block iterations of the
// stream-K tiles [dp_tiles, tiles) are cut into G contiguous ranges, worker w
// taking range w. A range may start inside a tile and end inside another, so
// a tile can be shared by several consecutive workers. Each worker's range is
// a list of segments (tile, kb0, kb1):
//   FULL     kb0 == 0 and kb1 == L: the worker stores the tile to C;
//   PARTIAL  kb0 > 0 (only a range's FIRST segment): the worker stores its
//            partial sums to workspace slot w and publishes flag w = epoch;
//   HEAD     kb0 == 0, kb1 < L (only a range's LAST segment): the worker owns
//            the tile: it adds, in worker order, the partial sums of the
//            workers w+1, w+2, ... that hold the rest of the tile, and stores C.
// A worker publishes its PARTIAL before it waits for anything, and waits only
// for higher-numbered workers' PARTIALs, so no wait depends on a worker that
// is itself waiting: every wait ends even if the workers are not all resident.
// Sums are added in a fixed order, so results are deterministic run to run.
#pragma once

#include <cstdint>

namespace gemm14 {

enum : int { kSegFull = 0, kSegPartial = 1, kSegHead = 2 };

struct StreamK {
  int tiles;     // output tiles
  int L;         // k-blocks per tile
  int G;         // workers (CTAs or CTA pairs)
  int dp_tiles;  // tiles done whole, round-robin (tile t by worker t % G)

  __host__ __device__ int64_t sk_iters() const {
    return static_cast<int64_t>(tiles - dp_tiles) * L;
  }
  // First stream-K flat iteration (relative to tile dp_tiles) of worker w.
  __host__ __device__ int64_t sk_start(int w) const { return sk_iters() * w / G; }
  __host__ __device__ int dp_count(int w) const {
    return w < dp_tiles ? (dp_tiles - 1 - w) / G + 1 : 0;
  }

  // Segments of worker w: dp_count(w) whole tiles, then its stream-K range.
  __host__ __device__ int sk_segments(int w) const {
    const int64_t s = sk_start(w), e = sk_start(w + 1);
    if (e <= s) return 0;
    return static_cast<int>((e - 1) / L - s / L + 1);
  }
  __host__ __device__ int segments(int w) const { return dp_count(w) + sk_segments(w); }
  __host__ __device__ int64_t iterations(int w) const {
    return static_cast<int64_t>(dp_count(w)) * L + (sk_start(w + 1) - sk_start(w));
  }

  // Segment i of worker w -> tile, k-block range and kind.
  __host__ __device__ void segment(int w, int i, int& tile, int& kb0, int& kb1, int& kind) const {
    const int ndp = dp_count(w);
    if (i < ndp) {
      tile = w + i * G;
      kb0 = 0;
      kb1 = L;
      kind = kSegFull;
      return;
    }
    const int64_t s = sk_start(w), e = sk_start(w + 1);
    const int64_t t = s / L + (i - ndp);
    const int64_t lo = s > t * L ? s : t * L;
    const int64_t hi = e < (t + 1) * L ? e : (t + 1) * L;
    tile = dp_tiles + static_cast<int>(t);
    kb0 = static_cast<int>(lo - t * L);
    kb1 = static_cast<int>(hi - t * L);
    kind = kb0 > 0 ? kSegPartial : (kb1 == L ? kSegFull : kSegHead);
  }

  // Flat iteration j of worker w -> (tile, kb), for the loaders.
  __host__ __device__ void iteration(int w, int64_t j, int& tile, int& kb) const {
    const int64_t dp_it = static_cast<int64_t>(dp_count(w)) * L;
    if (j < dp_it) {
      tile = w + static_cast<int>(j / L) * G;
      kb = static_cast<int>(j % L);
      return;
    }
    const int64_t p = sk_start(w) + (j - dp_it);
    tile = dp_tiles + static_cast<int>(p / L);
    kb = static_cast<int>(p % L);
  }

  // For a HEAD segment of tile (relative) t owned by w: the next contributor
  // after worker c, or -1. Contributors are w+1, w+2, ... while their ranges
  // start inside the tile.
  __host__ __device__ int next_contributor(int c, int tile) const {
    const int64_t end = static_cast<int64_t>(tile - dp_tiles + 1) * L;
    for (int n = c + 1; n < G && sk_start(n) < end; ++n)
      if (sk_start(n + 1) > sk_start(n)) return n;  // skip workers with empty ranges
    return -1;
  }
};

// A worker's schedule, decoded once at kernel start (by one thread, into
// shared memory) so that the loops never divide: dp whole tiles w, w+G, ...,
// then at most kMaxSk stream-K segments (fewer than 2G tiles are split, so a
// range spans at most 3 tiles), and for a HEAD the last contributing worker.
constexpr int kMaxSk = 4;
struct SkTable {
  int n_dp, n_sk, G, L, w;
  int tile[kMaxSk], kb0[kMaxSk], kb1[kMaxSk], kind[kMaxSk];
  int head_last;  // last worker whose partial the HEAD adds (w: none)

  __host__ __device__ void fill(const StreamK& sk, int worker) {
    w = worker;
    G = sk.G;
    L = sk.L;
    n_dp = sk.dp_count(worker);
    n_sk = sk.sk_segments(worker);
    head_last = worker;
    for (int i = 0; i < n_sk && i < kMaxSk; ++i) {
      sk.segment(worker, n_dp + i, tile[i], kb0[i], kb1[i], kind[i]);
      if (kind[i] == kSegHead)
        for (int c = sk.next_contributor(worker, tile[i]); c >= 0;
             c = sk.next_contributor(c, tile[i]))
          head_last = c;
    }
  }
  __host__ __device__ int segments() const { return n_dp + n_sk; }
  __host__ __device__ void get(int i, int& t, int& k0, int& k1, int& kd) const {
    if (i < n_dp) {
      t = w + i * G;
      k0 = 0;
      k1 = L;
      kd = kSegFull;
    } else {
      const int j = i - n_dp;
      t = tile[j];
      k0 = kb0[j];
      k1 = kb1[j];
      kd = kind[j];
    }
  }
};

// Walks a worker's k-block iterations in order, one at a time, without
// dividing: data-parallel tiles w, w+G, ... (kSK false) or the decoded table.
struct SegmentCursor {
  int seg, nseg, tile, kb, kb1;
  template <bool kSK>
  __host__ __device__ void start(const SkTable& t, int w, int n_dp, int L) {
    seg = 0;
    kb = 0;
    if (kSK) {
      nseg = t.segments();
      int kd;
      if (nseg > 0) t.get(0, tile, kb, kb1, kd);
    } else {
      nseg = n_dp;
      tile = w;
      kb1 = L;
    }
  }
  template <bool kSK>
  __host__ __device__ void next(const SkTable& t, int G) {
    if (++kb < kb1) return;
    if (++seg >= nseg) return;
    if (kSK) {
      int kd;
      t.get(seg, tile, kb, kb1, kd);
    } else {
      tile += G;
      kb = 0;
    }
  }
};

// Host-side choice of the data-parallel share: with a workspace, whole waves
// stay data-parallel except the last one and a half (or all tiles, when there
// are fewer than two waves), whose k-blocks are spread evenly over the G
// workers; without one, or when the tiles fill whole waves, every tile is
// data-parallel. The caller launches sk.G workers.
// With fewer than two waves every tile is split and the worker count is
// capped at the number of k-block iterations, so that no range is empty.
//
// Splitting pays in two regimes: few tiles (fewer than G/2: their k-blocks
// spread over many idle SMs) and one or more full waves (the last one and a
// half waves balanced). In between, a range holds fewer k-blocks than a tile
// and the owner of a split tile would wait for a contributor whose part is
// longer than its own range, so those shapes stay data-parallel.
inline bool stream_k_pays(int tiles, int G) {
  return G > 1 && tiles % G != 0 && (2 * tiles < G || tiles >= G);
}

inline StreamK make_stream_k(int tiles, int L, int G, bool have_workspace) {
  StreamK sk{tiles, L, G, tiles};
  if (!have_workspace || !stream_k_pays(tiles, G)) return sk;
  const int sk_tiles = tiles < 2 * G ? tiles : G + tiles % G;
  sk.dp_tiles = tiles - sk_tiles;
  if (sk.dp_tiles == 0) {
    const int64_t iters = static_cast<int64_t>(tiles) * L;
    if (iters < G) sk.G = static_cast<int>(iters);
  }
  return sk;
}

}  // namespace gemm14
