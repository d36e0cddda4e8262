// sgemm_simt.cu -- fp32 GEMM on the CUDA cores (FFMA), C = A * B, row-major.
//
// Design (sm_103a):
//  * Persistent grid: one CTA (8 warps) per SM walks output tiles blockIdx.x,
//    +gridDim.x, ... Its work is one flat list of (tile, k-block) iterations,
//    so the loads of the next tile start while the current tile is still
//    being computed and stored.
//  * Multistage ring: 4 shared-memory stages guarded by full/empty mbarriers.
//    Loads for iteration j + 3 are issued as soon as every warp has finished
//    iteration j - 1, overlapping transfer and compute -- the double-buffering
//    of "Kernel 优化指南" (cuda-kernel-academy module 02), "Level 3: Double
//    Buffering", and of gpu-hpc-book ch.06 "高级 cuda 特性 —— 从矩阵乘法(gemm)说起",
//    "调度优化" (batching loads along k, asynchronous copies), with a deeper ring.
//  * Loads: thread 0 issues TMA boxes (A: 32 k x 128 m with the 128-byte
//    swizzle; B: 256 n x 32 k; stored transposes in their own layouts, see
//    Lay below). When an operand breaks TMA's 16-byte rules all 256 threads
//    fill the untransposed shared-memory layout with 4-byte cp.async copies
//    instead. Either way out-of-range elements are zero-filled: the
//    guarded zero-fill of the pages' tiled kernels ("矩阵乘法中的分块与数据复用",
//    matmul_l1 and matmul_l1_reg).
//  * Register tiling: each thread owns an 8 x 16 block of C and per k does
//    its 8 x 16 multiply-adds from 8 A values and 16 B values as 64 packed
//    fp32x2 FMAs (fma.rn.f32x2: two IEEE fp32 FMAs per instruction, each
//    accumulator summed over k in order, as scalar fmaf would) -- the outer
//    product of the pages' matmul_l1_reg ("Register Tiling"), grown to a
//    128 x 256 block tile and an 8 x 16 microtile. The k-block loop is fully
//    unrolled so the next k group's shared loads overlap this one's FMAs.
//  * Conflict-free shared memory: A rows are 128 bytes with the 16-byte chunk
//    index XOR-ed by (row % 8); a warp's A loads touch rows r .. r+3 (distinct
//    mod 8), so its four distinct 16-byte chunks land in distinct banks. B
//    rows are read as 8 contiguous float4 per warp (128 bytes). This is the
//    bank-conflict avoidance of "Kernel 优化指南", "Bank Conflict 避免", done by
//    swizzling instead of padding. Stored transposes keep this property with
//    their own thread mapping (Lay).
//  * Epilogue: 16-byte stores when C permits ("向量化加载"), guarded scalar
//    stores otherwise; each warp store covers 4 rows x 128 contiguous bytes.
#include "kernels.h"
#include "ptx.cuh"

namespace gemm14 {
namespace {

using S = SgemmShape;
// Two fp32 values in one 64-bit register (low half = first value).
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
// d = a * b + d on both halves, each an IEEE fp32 fma (round to nearest).
__device__ __forceinline__ void fma2(uint64_t& d, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

struct SgemmSmem {
  uint64_t full[S::STAGES];
  uint64_t empty[S::STAGES];
  uint64_t bt_ready[2];  // B stored N x K: transposed buffer b holds the current stage
  int abort_flag;
  SkTable sched;  // this CTA's segments, decoded once
  // The loaders' position in the schedule (touched once per k-block, kept out
  // of registers): slot 0 for the TMA thread, one per thread for cp.async.
  SegmentCursor cursor[S::THREADS];
};

static_assert(sizeof(SgemmSmem) <= 512 + 20 * S::THREADS, "smem reserve for barriers and cursors");

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Byte offset of A element (m, k) inside an A stage: 128-byte rows, 16-byte
// chunks XOR-swizzled by (m % 8) -- the layout TMA's 128-byte swizzle writes.
__device__ __forceinline__ uint32_t a_tile_offset(int m, int k) {
  return static_cast<uint32_t>(m * 128 + ((((k >> 2) ^ (m & 7)) & 7) << 4) + (k & 3) * 4);
}

// Output tile index -> (row tile, column tile): row tiles vary fastest, so
// CTAs working at the same time share B panels.
struct TileGrid {
  int tiles_m;
  __device__ __forceinline__ void coords(int tile, int& tm, int& tn) const {
    tm = tile % tiles_m;
    tn = tile / tiles_m;
  }
};

// Loads of flat iteration j (output tile `tile`, k-block kb) into stage j % STAGES.
template <bool kTma, bool kGeneral, int kLay>
__device__ __forceinline__ void issue_stage(uint32_t j, int tile, int kb, const TileGrid& grid,
                                            uint8_t* tiles, SgemmSmem& sm,
                                            const CUtensorMap* map_a, const CUtensorMap* map_b,
                                            const GemmArgs& args) {
  // Failure-detection tests: the first stage is never loaded, so every wait
  // for it must expire and report a timeout.
  if (args.fault == kFaultSkipFirstStage && j == 0) return;
  int tm, tn;
  grid.coords(tile, tm, tn);
  const uint32_t s = j % S::stages(kLay);
  uint8_t* a_st = tiles + s * S::STAGE_BYTES;
  if (kTma) {
    // called by thread 0 only
    mbar_arrive_expect_tx(&sm.full[s], S::STAGE_BYTES);
    // A stored K x M: box 128 m x 32 k; B stored N x K: box 32 k x 256 n.
    if (kLay & 1) tma_load_2d(a_st, map_a, tm * S::BM, kb * S::BK, &sm.full[s]);
    else tma_load_2d(a_st, map_a, kb * S::BK, tm * S::BM, &sm.full[s]);
    if (kLay & 2) tma_load_2d(a_st + S::A_STAGE_BYTES, map_b, kb * S::BK, tn * S::BN, &sm.full[s]);
    else tma_load_2d(a_st + S::A_STAGE_BYTES, map_b, tn * S::BN, kb * S::BK, &sm.full[s]);
  } else {
    // called by all threads: 4096 A + 8192 B elements, 48 per thread. Each
    // thread's copies step through memory by a fixed stride and through
    // shared memory by a fixed offset, so the addresses are kept incrementally
    // (a few instructions a copy).
    const float* A = static_cast<const float*>(args.A);
    const float* B = static_cast<const float*>(args.B);
    const uint32_t a_sm = smem_u32(a_st);
    const uint32_t b_sm = a_sm + S::A_STAGE_BYTES;
    const int t = threadIdx.x;
    if (!(kGeneral && args.transa)) {
      // k = the thread's lane within the block: a warp reads 128 contiguous
      // bytes of a row; rows r0, r0 + 8, ... (same swizzle: r % 8 is fixed)
      const int kl = t & 31, r0 = t >> 5;
      const int k = kb * S::BK + kl;
      const int m = tm * S::BM + r0;
      const int rows_in = k < args.K ? args.M - m : 0;  // copies i with 8 i < rows_in
      const int64_t step = static_cast<int64_t>(S::THREADS / 32) * args.lda;
      int64_t off = static_cast<int64_t>(m) * args.lda + k;
      const uint32_t d0 = a_sm + a_tile_offset(r0, kl);
#pragma unroll
      for (int i = 0; i < S::BM / (S::THREADS / 32); ++i, off += step) {
        const bool in = (S::THREADS / 32) * i < rows_in;
        cp_async_4(d0 + i * (S::THREADS / 32) * 128, in ? A + off : A, in ? 4u : 0u);
      }
    } else {
      // A stored K x M: 128 threads read 512 contiguous bytes (128 m) of a k
      // row; the swizzle spreads their 4-byte stores over 8 banks.
      const int ml = t & (S::BM - 1), kr0 = t / S::BM;
      const int m = tm * S::BM + ml;
      const int k = kb * S::BK + kr0;
      const int k_in = m < args.M ? args.K - k : 0;  // copies i with 2 i < k_in
      constexpr int KSTEP = S::THREADS / S::BM;
      const int64_t step = static_cast<int64_t>(KSTEP) * args.lda;
      int64_t off = static_cast<int64_t>(k) * args.lda + m;
#pragma unroll
      for (int i = 0; i < S::BK / KSTEP; ++i, off += step) {
        const bool in = KSTEP * i < k_in;
        cp_async_4(a_sm + a_tile_offset(ml, kr0 + KSTEP * i), in ? A + off : A, in ? 4u : 0u);
      }
    }
    {
      // 256 threads = 256 columns of one k row. B stored N x K: thread n
      // reads its row's 32 consecutive k (one 128-byte line, kept in L1
      // across the loop); the shared-memory stores stay conflict-free.
      const int nl = t;
      const int n = tn * S::BN + nl;
      const bool tb = kGeneral && args.transb;
      const int64_t k_stride = tb ? 1 : args.ldb;
      const int k0 = kb * S::BK;
      const int k_in = n < args.N ? args.K - k0 : 0;  // copies kr < k_in
      int64_t off = (tb ? static_cast<int64_t>(n) * args.ldb : n) + k0 * k_stride;
#pragma unroll
      for (int kr = 0; kr < S::BK; ++kr, off += k_stride) {
        const bool in = kr < k_in;
        cp_async_4(b_sm + static_cast<uint32_t>(kr * S::BN + nl) * 4, in ? B + off : B,
                   in ? 4u : 0u);
      }
    }
    cp_async_mbar_arrive_noinc(&sm.full[s]);
  }
}

// Shared-memory layouts of the TMA loader for stored transposes. kLay bit 0:
// A is M-major ([32 k][128 m], 512-byte rows, as TMA writes A stored K x M);
// bit 1: B arrives K-major ([256 n][32 k], 128-byte rows with the 128-byte
// swizzle, as TMA writes B stored N x K) and is transposed in shared memory
// into the [k][n] layout of B stored K x N before the FMAs read it. The
// thread mapping follows A's layout so that shared loads stay 16 bytes wide
// and conflict-free:
//   rows    M-major A: warp_m*32 + tr*8 + i (8 contiguous rows per thread),
//           else warp_m*32 + tr + 4i;
//   columns warp_n*128 + 4tc + 32(j/4) + j%4.
// Accumulator pair p of row i holds columns j = 2p and 2p + 1.
template <int kLay>
struct Lay {
  static constexpr bool AM = (kLay & 1) != 0;
  static __device__ __forceinline__ int row(int warp_m, int tr, int i) {
    return AM ? warp_m * 32 + tr * 8 + i : warp_m * 32 + tr + 4 * i;
  }
  static __device__ __forceinline__ int col(int warp_n, int tc, int j) {
    return warp_n * 128 + tc * 4 + 32 * (j >> 2) + (j & 3);
  }
};

__device__ __forceinline__ float comp4(const float4& v, int q) {
  return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

// Four k (group kg of a 32-deep k-block) of the 8 x 16 register tile from a
// stage in layout kLay: per k, 8 A values (two 16-byte loads for M-major A,
// else from 16-byte loads along k), 8 column pairs of B (four 16-byte loads
// along n), and 64 packed fp32x2 FMAs.
template <int kLay>
__device__ __forceinline__ void fma_kgroup(uint32_t a_base, uint32_t b_base, int kg, int warp_m,
                                           int warp_n, int tr, int tc, uint64_t (&acc2)[8][8]) {
  using LY = Lay<kLay>;
  // M-major A: af[2kk + h] = rows 4h .. 4h+3 of this thread at k = 4kg + kk;
  // else af[i] = row i at k = 4kg .. 4kg+3.
  float4 af[8];
  if (LY::AM) {
    const uint32_t a0 = a_base + static_cast<uint32_t>((warp_m * 32 + tr * 8) * 4);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      af[2 * kk] = lds128(a0 + static_cast<uint32_t>((4 * kg + kk) * 512));
      af[2 * kk + 1] = lds128(a0 + static_cast<uint32_t>((4 * kg + kk) * 512 + 16));
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = LY::row(warp_m, tr, i);
      af[i] = lds128(a_base + static_cast<uint32_t>(r * 128 + (((kg ^ r) & 7) << 4)));
    }
  }
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    uint64_t bp[8];
    const uint32_t b0 = b_base + static_cast<uint32_t>((4 * kg + kk) * (S::BN * 4) +
                                                       (warp_n * 128 + tc * 4) * 4);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const float4 v = lds128(b0 + static_cast<uint32_t>(128 * jj));
      bp[2 * jj] = pack2(v.x, v.y);
      bp[2 * jj + 1] = pack2(v.z, v.w);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float av = LY::AM ? comp4(af[2 * kk + (i >> 2)], i & 3) : comp4(af[i], kk);
      const uint64_t a2 = pack2(av, av);
#pragma unroll
      for (int p = 0; p < 8; ++p) fma2(acc2[i][p], a2, bp[p]);
    }
  }
}

// One k-block: A from the stage, B ([k][n], 1 KB rows) at b_base.
template <int kLay>
__device__ __forceinline__ void fma_kblock(const uint8_t* stage, uint32_t b_base, int warp_m,
                                           int warp_n, int tr, int tc, uint64_t (&acc2)[8][8]) {
  const uint32_t a_base = smem_u32(stage);
  // fully unrolled: the next k group's shared loads overlap this one's FMAs
  // (5.7 % faster than unrolling by 2, no spills)
#pragma unroll
  for (int kg = 0; kg < S::BK / 4; ++kg)
    fma_kgroup<kLay>(a_base, b_base, kg, warp_m, warp_n, tr, tc, acc2);
}

// B stored N x K as TMA lands it ([256 n][32 k], 128-byte rows, 16-byte chunk
// c of row n at chunk c XOR (n % 8)) into bt as [32 k][256 n], the layout of
// B stored K x N. Thread t moves row n = t: eight 16-byte loads (a quarter
// warp reads 8 rows' distinct chunks) and 32 4-byte stores (a warp writes
// 128 contiguous bytes of a k row).
__device__ __forceinline__ void transpose_b(uint32_t b_st, uint32_t bt) {
  const int n = threadIdx.x;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float4 v[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
      v[c] = lds128(b_st + static_cast<uint32_t>(n * 128 + ((((4 * h + c) ^ n) & 7) << 4)));
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int k = 4 * (4 * h + c) + q;
        const float x = comp4(v[c], q);
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(bt + static_cast<uint32_t>((k * S::BN + n) * 4)),
                     "f"(x)
                     : "memory");
      }
  }
}

// kSK: the stream-K schedule (segments, workspace partials); without it the
// schedule is plain data-parallel (tiles w, w+G, ... whole) and none of the
// stream-K machinery is compiled in. kGeneral: stored transposes (cp.async
// loader) and the alpha / beta epilogue are read from args; without it the
// kernel is compiled for untransposed operands and a plain store of C. kLay
// (TMA loader only): the stored transposes' shared-memory layouts, above.
template <bool kTma, bool kSK, bool kGeneral, int kLay>
__global__ void __launch_bounds__(S::THREADS, 1)
    sgemm_simt_kernel(const __grid_constant__ CUtensorMap map_a,
                      const __grid_constant__ CUtensorMap map_b, const GemmArgs args) {
  static_assert(kLay == 0 || kTma, "transposed layouts come from the TMA loader");
  constexpr int STG = S::stages(kLay);        // ring stages
  constexpr bool kBT = (kLay & 2) != 0;      // B transposed in shared memory
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = align1024(smem_raw);
  const uint32_t bt_base = smem_u32(tiles + STG * S::STAGE_BYTES);  // two [k][n] buffers (kBT)
  SgemmSmem& sm = *reinterpret_cast<SgemmSmem*>(tiles + STG * S::STAGE_BYTES +
                                                (kBT ? 2 * S::BT_BYTES : 0));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int M = args.M, N = args.N;
  const int w = blockIdx.x;  // this CTA's worker index in the schedule
  const TileGrid tgrid{(M + S::BM - 1) / S::BM};
  const uint32_t n_iter = static_cast<uint32_t>(args.sk.iterations(w));
  const WaitCtx wc{args.err, &sm.abort_flag, args.wait_limit_ns, 0u};
  const bool producer = kTma ? threadIdx.x == 0 : true;
  uint32_t issued = 0;  // iterations whose loads this thread has issued

  if (threadIdx.x == 0) {
    for (int s = 0; s < STG; ++s) {
      mbar_init(&sm.full[s], kTma ? 1 : S::THREADS);
      mbar_init(&sm.empty[s], S::WARPS);
    }
    for (int b = 0; b < 2; ++b) mbar_init(&sm.bt_ready[b], S::THREADS);
    sm.abort_flag = 0;
    if (kSK) {
      sm.sched.fill(args.sk, w);
      if (sm.sched.n_sk > kMaxSk) {  // cannot happen for schedules make_stream_k builds
        atomicOr(args.err, kDevErrBadConfig);
        sm.abort_flag = 1;
      }
    }
    fence_barrier_init();
    if (kTma) {
      tma_prefetch_desc(&map_a);
      tma_prefetch_desc(&map_b);
    }
  }
  __syncthreads();
  // Set-up touched only shared memory and the parameters (and the error
  // word's commuting OR); global memory is used from here on.
  grid_dependency_wait();
  grid_launch_dependents();
  const int G = args.sk.G, L = args.sk.L;
  const int n_seg = kSK ? (sm.abort_flag ? 0 : sm.sched.segments()) : args.sk.dp_count(w);

  // The loaders walk the iterations in order. Data-parallel: iteration j is
  // k-block j % L of tile w + (j / L) * G. Stream-K: a cursor over the
  // decoded segments, kept in shared memory (touched once per k-block).
  // Data-parallel: two registers (tile, k-block). Stream-K: a cursor over the
  // decoded segments in shared memory (it would cost registers in the loop).
  SegmentCursor& pcur = sm.cursor[kTma ? 0 : threadIdx.x];
  int dp_tile = w, dp_kb = 0;
  auto load = [&](uint32_t j) {
    if (kSK) {
      issue_stage<kTma, kGeneral, kLay>(j, pcur.tile, pcur.kb, tgrid, tiles, sm, &map_a, &map_b, args);
      pcur.next<true>(sm.sched, G);
    } else {
      issue_stage<kTma, kGeneral, kLay>(j, dp_tile, dp_kb, tgrid, tiles, sm, &map_a, &map_b, args);
      if (++dp_kb == L) {
        dp_kb = 0;
        dp_tile += G;
      }
    }
  };

  // Prologue: fill the ring (fresh stages need no empty-wait).
  if (producer && n_seg > 0) {
    if (kSK) pcur.start<true>(sm.sched, w, n_seg, L);
    for (; issued < n_iter && issued < static_cast<uint32_t>(STG); ++issued) load(issued);
  }

  // This thread's rows: warp_m*32 + tr + 4*i (i < 8); columns:
  // warp_n*128 + tc*4 + 32*jj + q (jj, q < 4).
  const int warp_m = warp & 3;  // 4 warps along m (32 rows each)
  const int warp_n = warp >> 2; // 2 warps along n (128 columns each)
  const int tr = lane >> 3;     // 4 thread rows per warp
  const int tc = lane & 7;      // 8 thread columns per warp

  uint32_t it = 0;
  bool ok = true;
  for (int seg = 0; seg < n_seg && ok; ++seg) {
    int tile, kb0, kb1, kind, tm, tn;
    if (kSK) {
      sm.sched.get(seg, tile, kb0, kb1, kind);
    } else {
      tile = w + seg * G;
      kb0 = 0;
      kb1 = L;
      kind = kSegFull;
    }
    tgrid.coords(tile, tm, tn);
    // acc2[i][p] holds columns j = 2p and 2p + 1 (Lay<kLay>::col) of row i.
    uint64_t acc2[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc2[i][j] = 0ull;

    for (int kb = kb0; kb < kb1; ++kb, ++it) {
      const uint32_t s = it % STG, ph = (it / STG) & 1;
      if (!mbar_wait(&sm.full[s], ph, wc)) { ok = false; break; }
      uint8_t* stage = tiles + s * S::STAGE_BYTES;
      uint32_t b_base = smem_u32(stage) + S::A_STAGE_BYTES;
      if (kBT) {
        // Transpose this stage's B into buffer it % 2; every thread's part
        // is in before any thread reads it (a bounded wait, not a CTA
        // barrier: a thread that gave up on a wait leaves the loop). The
        // buffer's previous contents (iteration it - 2) were read before
        // each thread arrived here for iteration it - 1.
        const uint32_t bt = bt_base + (it & 1) * S::BT_BYTES;
        transpose_b(b_base, bt);
        mbar_arrive(&sm.bt_ready[it & 1]);
        if (!mbar_wait(&sm.bt_ready[it & 1], (it >> 1) & 1, wc)) { ok = false; break; }
        b_base = bt;
      }
      fma_kblock<kLay>(stage, b_base, warp_m, warp_n, tr, tc, acc2);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[s]);

      // Refill: once every warp is done with iteration it-1, its stage takes
      // iteration it-1+STG (one iteration of slack keeps warp 0 from waiting
      // on the slowest warp of the current iteration).
      if (producer && it >= 1 && issued < n_iter && issued == it - 1 + STG) {
        const uint32_t j = it - 1;
        if (!mbar_wait(&sm.empty[j % STG], (j / STG) & 1, wc)) {
          ok = false;
          break;
        }
        load(issued);
        ++issued;
      }
    }
    if (kSK) {
      // Stream-K segments end at a CTA barrier: a thread whose wait failed
      // has raised the abort flag and left the k loop, and all threads take
      // the decision to stop at the same point before the epilogues' barriers.
      __syncthreads();
      if (sm.abort_flag) ok = false;
    }
    if (!ok) break;

    // Stream-K. A PARTIAL stores its sums to workspace slot w (tile-local
    // element (r, c) at r * BN + c) and publishes flag w. A HEAD waits for the
    // later workers' flags and adds their slots w+1, ..., head_last, in that
    // order, into its own accumulators, then stores the tile like a FULL one.
    // Every worker runs the same thread mapping (Lay), so the element a thread
    // holds sits at the same place in each slot: the adds read the slots in
    // the accumulators' layout, and the sum is own + p(w+1) + p(w+2) + ...
    // as before, without a slot of the owner's own.
    if (kSK && kind == kSegPartial) {
      float* slot = args.partials + static_cast<size_t>(w) * (S::BM * S::BN);
#ifdef GEMM14_DEVICE_CHECKS
      // the bounds checks of a slot access (args.sk.G slots of BM x BN); the
      // product build compiles none of them (this kernel's registers are tight)
      auto slot_ok = [&](const float* p, int s, int width) {
        return dev_check(slot_span_ok(p - args.partials, s, S::BM * S::BN,
                                      static_cast<int64_t>(args.sk.G), width),
                         args.err);
      };
#endif
      {
        using LY = Lay<kLay>;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float* srow = slot + LY::row(warp_m, tr, i) * S::BN;
#pragma unroll
          for (int p = 0; p < 8; p += 2) {
            const float2 lo = unpack2(acc2[i][p]), hi = unpack2(acc2[i][p + 1]);
#ifdef GEMM14_DEVICE_CHECKS
            if (!slot_ok(srow + LY::col(warp_n, tc, 2 * p), w, 1) ||
                !slot_ok(srow + LY::col(warp_n, tc, 2 * p + 3), w, 1))
              continue;
#endif
            // columns 2p .. 2p+3 are consecutive
            __stcg(reinterpret_cast<float4*>(srow + LY::col(warp_n, tc, 2 * p)),
                   make_float4(lo.x, lo.y, hi.x, hi.y));
          }
        }
      }
      __syncthreads();
      if (threadIdx.x == 0 && dev_check(index_ok(w, args.sk.G), args.err))
        flag_publish(args.flags + w, args.epoch);
      continue;
    }
    if (kSK && kind == kSegHead) {
      const int last = sm.sched.head_last;
      if (threadIdx.x == 0)
        for (int c = w + 1; c <= last; ++c) {
          if (!dev_check(index_ok(c, args.sk.G), args.err)) break;
          // (inline: the accumulators are live across the wait)
          if (!flag_wait_inline(args.flags + c, args.epoch, wc)) break;  // raises abort on expiry
          flag_clear(args.flags + c);
        }
      __syncthreads();  // the flags were seen before any thread reads a slot
      if (sm.abort_flag) { ok = false; break; }
      using LY = Lay<kLay>;
#pragma unroll 1
      for (int c = w + 1; c <= last; ++c) {
        const float* slot = args.partials + static_cast<size_t>(c) * (S::BM * S::BN);
        // two rows of the thread's 8 x 16 block per round: their 8 (or 32)
        // loads in flight together
#pragma unroll
        for (int i0 = 0; i0 < 8; i0 += 2) {
          float v[2][16];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float* srow = slot + LY::row(warp_m, tr, i0 + h) * S::BN;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const float* q = srow + LY::col(warp_n, tc, 4 * jj);
#ifdef GEMM14_DEVICE_CHECKS
              if (!dev_check(slot_span_ok(q - args.partials, c, S::BM * S::BN, args.sk.G, 4),
                             args.err)) {
                v[h][4 * jj] = v[h][4 * jj + 1] = v[h][4 * jj + 2] = v[h][4 * jj + 3] = 0.f;
                continue;
              }
#endif
              const float4 t = __ldcg(reinterpret_cast<const float4*>(q));
              v[h][4 * jj] = t.x;
              v[h][4 * jj + 1] = t.y;
              v[h][4 * jj + 2] = t.z;
              v[h][4 * jj + 3] = t.w;
            }
          }
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int p = 0; p < 8; ++p) {
              const float2 a = unpack2(acc2[i0 + h][p]);
              acc2[i0 + h][p] = pack2(a.x + v[h][2 * p], a.y + v[h][2 * p + 1]);
            }
          // the next rounds' loads stay behind this one's adds (a compiler
          // barrier: without it all 32 loads are hoisted, and their registers
          // on top of the accumulators spill)
          asm volatile("" ::: "memory");
        }
      }
      // the HEAD's tile goes to C below, as a FULL tile's
    }
    // Epilogue: rows beyond M and columns beyond N are not written.
    {
      using LY = Lay<kLay>;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int row = tm * S::BM + LY::row(warp_m, tr, i);
        if (row >= M) continue;
        float* crow = args.C + static_cast<int64_t>(row) * args.ldc;
        float v[16];
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const float2 t = unpack2(acc2[i][p]);
          v[2 * p] = t.x;
          v[2 * p + 1] = t.y;
        }
        {
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int col = tn * S::BN + LY::col(warp_n, tc, 4 * jj);
            if (args.vec_store && col + 3 < N) {
              epi_store4<kGeneral>(args, crow + col,
                                   make_float4(v[4 * jj], v[4 * jj + 1], v[4 * jj + 2], v[4 * jj + 3]));
            } else {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                if (col + q < N) epi_store1<kGeneral>(args, crow + col + q, v[4 * jj + q]);
            }
          }
        }
      }
    }
  }

  // A CTA that gave up on a wait may still have copies in flight into its own
  // shared memory: drain them (bounded) before the CTA exits.
  __syncthreads();
  if (sm.abort_flag) {
    if (kTma) {
      if (threadIdx.x == 0) {
        const uint32_t first = issued > STG ? issued - STG : 0;
        for (uint32_t j = first; j < issued; ++j)
          if (!(args.fault == kFaultSkipFirstStage && j == 0))
            mbar_wait_timed(&sm.full[j % STG], (j / STG) & 1, 100000000ull);
      }
    } else {
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
  }
}

template <bool kTma, bool kSK, bool kGeneral, int kLay>
cudaError_t launch_variant(const CUtensorMap* map_a, const CUtensorMap* map_b,
                           const GemmArgs& args, int grid, cudaStream_t stream) {
  static DeviceOnce configured;
  const cudaError_t e = set_smem_once(configured, sgemm_simt_kernel<kTma, kSK, kGeneral, kLay>,
                                      S::smem_bytes(kLay));
  if (e != cudaSuccess) return e;
  CUtensorMap dummy{};
  return launch_kernel(sgemm_simt_kernel<kTma, kSK, kGeneral, kLay>, dim3(grid), dim3(S::THREADS),
                       S::smem_bytes(kLay), stream, map_a ? *map_a : dummy,
                       map_b ? *map_b : dummy, args);
}

template <bool kTma, bool kSK>
cudaError_t launch_epi(const CUtensorMap* map_a, const CUtensorMap* map_b, const GemmArgs& args,
                       int grid, cudaStream_t stream) {
  if constexpr (kTma) {
    if (args.transa || args.transb) {
      // the TMA loader reads stored transposes in their own layouts
      const int lay = (args.transa ? 1 : 0) | (args.transb ? 2 : 0);
      if (lay == 1) return launch_variant<true, kSK, true, 1>(map_a, map_b, args, grid, stream);
      if (lay == 2) return launch_variant<true, kSK, true, 2>(map_a, map_b, args, grid, stream);
      return launch_variant<true, kSK, true, 3>(map_a, map_b, args, grid, stream);
    }
  }
  if (args.transa || args.transb || args.epi != kEpiStore)
    return launch_variant<kTma, kSK, true, 0>(map_a, map_b, args, grid, stream);
  return launch_variant<kTma, kSK, false, 0>(map_a, map_b, args, grid, stream);
}

template <bool kTma>
cudaError_t launch(const CUtensorMap* map_a, const CUtensorMap* map_b, const GemmArgs& args,
                   int grid, cudaStream_t stream) {
  if (args.sk.dp_tiles < args.sk.tiles)
    return launch_epi<kTma, true>(map_a, map_b, args, grid, stream);
  return launch_epi<kTma, false>(map_a, map_b, args, grid, stream);
}

}  // namespace

cudaError_t launch_sgemm_tma(const CUtensorMap& map_a, const CUtensorMap& map_b,
                             const GemmArgs& args, int grid, cudaStream_t stream) {
  return launch<true>(&map_a, &map_b, args, grid, stream);
}

cudaError_t launch_sgemm_cpasync(const GemmArgs& args, int grid, cudaStream_t stream) {
  return launch<false>(nullptr, nullptr, args, grid, stream);
}

}  // namespace gemm14
