// plan.cu -- the launch policy of plan.h: kernel and tile choice, stream-K
// splitting, and the workspace copies of operands, with the measurements that
// set each rule.
#include <cstring>

#include "kernels.h"
#include "plan.h"

namespace gemm14 {

std::atomic<int> g_pair_enabled{1};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool is_tf32_mode(int dtype) {
  return dtype == GEMM14_DTYPE_TF32 || dtype == GEMM14_DTYPE_F32_3XTF32;
}
int elem_bytes_of(int dtype) {
  return dtype == GEMM14_DTYPE_F32 || is_tf32_mode(dtype) ? 4 : 2;
}

int hgemm_bn_for(int64_t N) { return N <= 64 ? 64 : N <= 128 ? 128 : 256; }

// Every kernel's TMA loader serves every storage: a stored transpose is an
// M-major A or a K-major B in shared memory (the fp32 kernel's thread mapping
// follows A's layout and it transposes K-major B tiles in shared memory; the
// tensor-core kernels take either major-ness).
// fp32 products above this many FLOP (2MNK) whose call has a workspace stay
// on the large kernel even with few tiles: its stream-K split over every SM
// beat the small-product kernel from about 1 GFLOP on GB300 (1024^3: 55.9
// against 67.8 us; 2048 x 1024 x 1024: 86.8 against 121.1 us; 512^3: 38.8
// against 16.3 us; 256 x 4096 x 256: 31.3 against 22.5 us).
constexpr double kSmallSplitFlops = 1073741824.0;

void plan_for(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K, const void* A,
              int64_t lda, const void* B, int64_t ldb, const void* C, int64_t ldc, int sm_count,
              gemm14_plan* p, bool split_ok) {
  std::memset(p, 0, sizeof *p);
  if (M == 0 || N == 0 || K == 0) return;  // nothing launched (K == 0: a memset)
  p->vec_store = aligned(C, 16) && (ldc % 4 == 0);
  if (is_tf32_mode(dtype)) {
    // fp32 inputs on the tensor cores: TMA-addressable operands on CTA pairs;
    // anything else on the fp32 SIMT kernel (exact fp32 products, so at least
    // as accurate as either tensor-core mode).
    if (aligned(A, 16) && aligned(B, 16) && lda % 4 == 0 && ldb % 4 == 0 && sm_count >= 2) {
      if (dtype == GEMM14_DTYPE_TF32 && !transa && transb && g_pair_enabled.load()) {
        // TF32 with both operands K-major as stored: the 16-bit pair kernel's
        // mainloop with kind::tf32 MMAs (k-blocks of 32 fp32), no conversion
        using P = PairShape;
        p->kernel = 5;
        p->loader = 1;
        p->bm = P::BM;
        p->bn = P::BN;
        p->bk = 32;
        p->stages = P::STAGES;
        p->threads = P::THREADS;
        p->smem_bytes = P::SMEM_BYTES;
        p->tiles = ((M + P::BM - 1) / P::BM) * ((N + P::BN - 1) / P::BN);
        const int64_t clusters = sm_count / 2;
        p->grid = static_cast<int>(2 * (p->tiles < clusters ? p->tiles : clusters));
        return;
      }
      using T = Tf32Shape;
      p->kernel = 4;
      p->loader = 1;
      p->bm = T::BM;
      p->bn = T::BN;
      p->bk = T::BK;
      p->stages = T::op_stages(dtype == GEMM14_DTYPE_F32_3XTF32);
      p->threads = T::threads(dtype == GEMM14_DTYPE_F32_3XTF32);
      p->smem_bytes = T::SMEM_BYTES;
      p->tiles = ((M + T::BM - 1) / T::BM) * ((N + T::BN - 1) / T::BN);
      const int64_t clusters = sm_count / 2;
      p->grid = static_cast<int>(2 * (p->tiles < clusters ? p->tiles : clusters));
      return;
    }
    dtype = GEMM14_DTYPE_F32;
  }
  if (dtype == GEMM14_DTYPE_F32) {
    using S = SgemmShape;
    const int64_t big_tiles = ((M + S::BM - 1) / S::BM) * ((N + S::BN - 1) / S::BN);
    const double flops = 2.0 * static_cast<double>(M) * static_cast<double>(N) *
                         static_cast<double>(K);
    if (2 * big_tiles <= sm_count && !(split_ok && flops > kSmallSplitFlops)) {
      // Fewer 128 x 256 tiles than half the SMs: 64 x 64 tiles, the k range of
      // each split over a cluster of up to 8 CTAs while the grid stays within
      // four CTAs per SM (and each CTA keeps at least one k-block).
      using Q = SmallShape;
      p->kernel = 6;
      p->loader = (!transa && !transb && aligned(A, 16) && aligned(B, 16) && lda % 4 == 0 &&
                   ldb % 4 == 0) ? 1 : 2;
      p->bm = Q::BM;
      p->bn = Q::BN;
      p->bk = Q::BK;
      p->stages = Q::STAGES;
      p->threads = Q::THREADS;
      p->smem_bytes = Q::SMEM_BYTES;
      p->tiles = ((M + Q::BM - 1) / Q::BM) * ((N + Q::BN - 1) / Q::BN);
      const int64_t L = (K + Q::BK - 1) / Q::BK;
      int64_t split = 1;
      while (split < 8 && p->tiles * split * 2 <= 4 * static_cast<int64_t>(sm_count) &&
             split * 2 <= L)
        split *= 2;
      p->grid = static_cast<int>(split * p->tiles);
      return;
    }
    p->kernel = 1;
    p->loader = (aligned(A, 16) && aligned(B, 16) && lda % 4 == 0 && ldb % 4 == 0) ? 1 : 2;
    p->bm = S::BM;
    p->bn = S::BN;
    p->bk = S::BK;
    // the TMA loader's shared-memory layout: A stored K x M (bit 0), B stored
    // N x K (bit 1, transposed in shared memory)
    const int lay = p->loader == 1 ? (transa ? 1 : 0) | (transb ? 2 : 0) : 0;
    p->stages = S::stages(lay);
    p->threads = S::THREADS;
    p->smem_bytes = S::smem_bytes(lay);
  } else {
    const int bn = hgemm_bn_for(N);
    // TMA for each operand it can read; the software loader for the others
    // (3: A only, 4: B only, 2: both)
    const bool a_tma = aligned(A, 16) && lda % 8 == 0, b_tma = aligned(B, 16) && ldb % 8 == 0;
    p->loader = a_tma && b_tma ? 1 : !a_tma && !b_tma ? 2 : !a_tma ? 3 : 4;
    if (p->loader == 1 && M > 128 && N > 128 && g_pair_enabled.load() && sm_count >= 2) {
      // 256 x 256 tiles on CTA pairs; grid = 2 x clusters
      using P = PairShape;
      p->kernel = 3;
      p->bm = P::BM;
      p->bn = P::BN;
      p->bk = P::BK;
      p->stages = P::STAGES;
      p->threads = P::THREADS;
      p->smem_bytes = P::SMEM_BYTES;
      p->tiles = ((M + P::BM - 1) / P::BM) * ((N + P::BN - 1) / P::BN);
      const int64_t clusters = sm_count / 2;
      p->grid = static_cast<int>(2 * (p->tiles < clusters ? p->tiles : clusters));
      return;
    }
    // One SM per tile: 128-row tiles, or 64-row tiles (M = 64 MMAs) when even
    // the 64-row tiles fit in one wave (the 128-row ones fill at most half the
    // SMs). Measured on GB300 (bf16, K = 4096): a tile's k-blocks stream at
    // about the same rate per CTA whatever the tile's rows, so the plain call
    // gains nothing from the smaller tiles (1024 to 8192 x 64: 21.7-22.6 us
    // back to back either way) and loses when they spill past one wave
    // (16384 x 64: 256 tiles, 41.3 against 26.9 us); the split call gains
    // from the finer work (128 x 2048: 52.8 -> 27.6 us; 1024 x 64: 20.1 ->
    // 16.6 us).
    const int64_t tiles128 = ((M + 127) / 128) * ((N + bn - 1) / bn);
    const int bm = 2 * tiles128 <= sm_count ? 64 : 128;
    p->kernel = 2;
    p->bm = bm;
    p->bn = bn;
    p->bk = HgemmShape::BK;
    p->stages = HgemmShape::stages(bn, bm);
    p->threads = p->loader == 1 ? HgemmShape::THREADS : HgemmShape::SOFT_THREADS;
    p->smem_bytes = HgemmShape::smem_bytes(bn, bm);
  }
  p->tiles = ((M + p->bm - 1) / p->bm) * ((N + p->bn - 1) / p->bn);
  const int64_t sms = sm_count > 0 ? sm_count : 1;
  p->grid = static_cast<int>(p->tiles < sms ? p->tiles : sms);
}
void plan_for(int dtype, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
              const void* B, int64_t ldb, const void* C, int64_t ldc, int sm_count,
              gemm14_plan* p, bool split_ok) {
  plan_for(dtype, 0, 0, M, N, K, A, lda, B, ldb, C, ldc, sm_count, p, split_ok);
}

// Stream-K workspace the call would use with a workspace (0: it uses none).
// One tile slot per worker, for its PARTIAL: a HEAD adds the later workers'
// slots into its accumulators (registers on the fp32 kernel, TMEM on the
// tensor-core kernels). The pair kernel's worker is a cluster of two SMs with
// a 256 x 256 tile: one 128 x 256 slot (and flag) per CTA, i.e. per SM, like
// the one-SM kernels.
int slots_per_worker(const gemm14_plan&) { return 1; }

// The CTA-pair kernel's split, measured on GB300 against its unsplit run:
// - between one and one and a half waves of tiles with long k (>= 64
//   k-blocks a tile): every tile split, 2304x2560x8192 (1.18 waves) 86 -> 74
//   us, TF32 2304x2560x4096 81 -> 69 us; with the last wave more than half
//   full the idle SMs are few and the split lost (bf16 3072x3072x8192, 1.89
//   waves, 86.6 us unsplit against 103.5 split; TF32 3072^3 66.9 against
//   79.4; 2816^2, 1.59 waves, 1.4-1.7 %);
// - beyond two waves, splitting every tile gained nothing (8192^3,
//   16384x11008x4096: within 1 %) or lost (4096x4096x16384: +21 %: ranges
//   that start mid-tile no longer sweep k together, so clusters stop sharing
//   A and B in L2); splitting only the last one and a half waves (the rest
//   data-parallel, as on the one-SM kernels) gains what the partial last wave
//   wasted: bf16 8192^3 (13.47 waves) -1.6 %, 16384x11008x4096 -1.4 %, fp16
//   8192^3 -2.5 %;
// - few tiles split over every cluster made the owner add up to ~19 partial
//   sums one after another (512x512x16384: no gain): there the workers are
//   capped at 4 per tile and at ranges of at least 32 k-blocks.
// Returns the workers (clusters) to split over, or 0 to run unsplit.
int pair_split_workers(int64_t tiles, int64_t L, int clusters) {
  if (clusters <= 1 || tiles <= 0) return 0;
  if (2 * tiles < clusters) {
    int64_t g = clusters;
    if (g > 4 * tiles) g = 4 * tiles;
    if (g > tiles * L / 32) g = tiles * L / 32;
    return g >= 2 * tiles ? static_cast<int>(g) : 0;
  }
  if (tiles > clusters && 2 * (tiles - clusters) < clusters && L >= 64) return clusters;
  if (tiles >= 2 * static_cast<int64_t>(clusters) && tiles % clusters != 0) return clusters;
  return 0;
}

// The one-SM kernels' split: the workers to spread the k-blocks over, or 0 to
// run data-parallel. fp32 k-blocks are long (a 128 x 256 x 32 block is about
// 2 MFLOP of FFMA work), so every SM takes a range. A 16-bit k-block streams
// 24-48 KB in well under a microsecond, while each further worker adds a
// partial sum that the tile's owner reads back; measured on GB300 (bf16,
// N = 64 or 128, K = 4096-16384), the best split had about 4 workers per tile
// and ranges of 16 or more k-blocks: 128x64x4096 25.0 us unsplit, 20.7 us on
// 4 workers, 150 us on 64; 512x128x8192 45.2 us unsplit, 33.0 us on 16, 153 us
// on 152. Between one and two waves, a 16-bit product splits only when its
// last wave is less than half full, as on the pair kernel: bf16 N = 64, K =
// 4096: 1.18 waves 48.3 -> 39.8 us split, but 1.87 waves 52.8 us unsplit
// against 56.7 split (N = 128, K = 2048: 33.7 against 39.7); fp32 gains at 1.89
// waves (3072^3: 0.959 -> 0.944 ms).
int one_sm_split_workers(int kernel, int64_t tiles, int64_t L, int G) {
  if (tiles <= 0 || tiles > INT32_MAX || !stream_k_pays(static_cast<int>(tiles), G)) return 0;
  if (kernel != 1 && tiles >= G && tiles < 2 * static_cast<int64_t>(G) && 2 * (tiles - G) >= G)
    return 0;
  if (kernel == 1 || 2 * tiles >= G) return G;
  int64_t g = G;
  if (g > 4 * tiles) g = 4 * tiles;
  if (g > tiles * L / 16) g = tiles * L / 16;
  return g >= 2 * tiles ? static_cast<int>(g) : 0;
}

size_t workspace_need(const gemm14_plan& plan, int sm_count, int64_t K, int k_terms) {
  if (plan.tiles > INT32_MAX) return 0;
  if (plan.kernel == 6) return 0;  // its split is added up in shared memory
  if (plan.kernel == 3 || plan.kernel == 5) {
    const int64_t L = (K + plan.bk - 1) / plan.bk * (k_terms > 1 ? k_terms : 1);
    if (!pair_split_workers(plan.tiles, L, sm_count / 2)) return 0;
    return streamk_workspace_bytes(sm_count, PairShape::BM / 2, PairShape::BN, 1);
  }
  if (plan.kernel != 1 && plan.kernel != 2) return 0;
  const int64_t L = (K + plan.bk - 1) / plan.bk;
  if (!one_sm_split_workers(plan.kernel, plan.tiles, L, sm_count)) return 0;
  return streamk_workspace_bytes(sm_count, plan.bm, plan.bn, slots_per_worker(plan));
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Fills *r for a call on `sms` SMs; r->a / r->b false when TMA can read the
// operand as it is (then the call never copies it).
void plan_repitch(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K,
                  const void* A, int64_t lda, const void* B, int64_t ldb, const void* C,
                  int64_t ldc, int sms, Repitch* r) {
  *r = Repitch{};
  r->transa = transa;
  r->transb = transb;
  if (M <= 0 || N <= 0 || K <= 0) return;
  const int eb = elem_bytes_of(dtype);
  const int64_t q = 16 / eb;
  r->a = !(aligned(A, 16) && lda % q == 0);
  r->b = !(aligned(B, 16) && ldb % q == 0);
  // TF32: the tensor cores read fp32 operands straight from TMA only K-major
  // (A stored M x K, B stored N x K, plan kernel 5); other storages are
  // transposed into that form (the converter kernel runs at about a quarter
  // of the speed).
  // 3xTF32 the same way, with lo(A) and lo(B) written beside them: the pair
  // kernel then runs 3 x the TF32 product's MMAs from K-major operands, while
  // the converter kernel splits the raw tiles as they arrive and its ring's
  // turnaround bounds it.
  const bool split = dtype == GEMM14_DTYPE_F32_3XTF32 && g_pair_enabled.load() && sms >= 2;
  if ((dtype == GEMM14_DTYPE_TF32 || split) && g_pair_enabled.load() && sms >= 2) {
    r->a_t = transa != 0;
    r->b_t = transb == 0;
    r->a = r->a || r->a_t;
    r->b = r->b || r->b_t;
    r->transa = 0;
    r->transb = 1;
    r->split = split;
  }
  // fp32 FFMA: B stored N x K, whose tiles the kernel transposes in shared
  // memory stage by stage, measured 70 % of the FFMA peak at 3072^3, against
  // 76 % for B stored K x N (A stored K x M is the fastest storage of A,
  // 80.5 %): with a workspace B is transposed into K x N ahead.
  // The small-product kernel reads any storage and pitch as it is: nothing
  // is copied for it.
  if (dtype == GEMM14_DTYPE_F32 || (is_tf32_mode(dtype) && !r->split &&
                                    !(dtype == GEMM14_DTYPE_TF32 && g_pair_enabled.load() &&
                                      sms >= 2))) {
    gemm14_plan as_stored;
    plan_for(dtype, transa, transb, M, N, K, A, lda, B, ldb, C, ldc, sms, &as_stored, true);
    if (as_stored.kernel == 6) {
      r->a = r->b = false;
      return;
    }
  }
  if (dtype == GEMM14_DTYPE_F32 && transb) {
    r->b_t = true;
    r->b = true;
    r->transb = 0;
  }
  // ... and A stored M x K (76 % at 3072^3) is transposed into K x M (80.5 %,
  // the same bits) when N is wide enough for the gain (about 5 % of the
  // product) to outweigh the transpose (8 M K bytes through HBM, about 40 / N
  // of the product's time): from N = 2048.
  if (dtype == GEMM14_DTYPE_F32 && !transa && N >= 2048) {
    r->a_t = true;
    r->a = true;
    r->transa = 1;
  }
  if (!r->a && !r->b && !r->split) return;
  // Stored shape of each copy: as the source, or transposed.
  const int64_t rows_a = r->transa ? K : M, cols_a = r->transa ? M : K;
  const int64_t rows_b = r->transb ? N : K, cols_b = r->transb ? K : N;
  r->lda = r->a ? (cols_a + q - 1) / q * q : lda;
  r->ldb = r->b ? (cols_b + q - 1) / q * q : ldb;
  // The plan of the copies: only their alignment and storage enter it.
  const void* base = reinterpret_cast<const void*>(uintptr_t(1) << 12);
  gemm14_plan plan;
  plan_for(r->split ? GEMM14_DTYPE_TF32 : dtype, r->transa, r->transb, M, N, K,
           r->a ? base : A, r->lda, r->b ? base : B, r->ldb, C, ldc, sms, &plan, true);
  const size_t sk = workspace_need(plan, sms, K, r->split ? 3 : 1);
  r->sk_bytes = sk;
  const size_t flags = streamk_flag_bytes(sms);
  r->a_off = round256(sk > flags ? sk : flags);
  const size_t a_bytes = r->a ? static_cast<size_t>(rows_a * r->lda * eb) : 0;
  r->b_off = round256(r->a_off + a_bytes);
  r->total = r->b ? r->b_off + static_cast<size_t>(rows_b * r->ldb * eb) : r->a_off + a_bytes;
  if (r->split) {
    // lo(A) M x K and lo(B) N x K, K-major, rows of K rounded up to 4 floats
    // (the pitch of A's and B's own copies, when they are copied)
    r->ld_lo = (K + q - 1) / q * q;
    r->a_lo_off = round256(r->total);
    r->b_lo_off = round256(r->a_lo_off + static_cast<size_t>(M * r->ld_lo * eb));
    r->total = r->b_lo_off + static_cast<size_t>(N * r->ld_lo * eb);
  }
}

}  // namespace gemm14
