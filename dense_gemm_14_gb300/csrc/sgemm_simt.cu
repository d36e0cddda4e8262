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
//    swizzle; B: 256 n x 32 k). When an operand breaks TMA's 16-byte rules all
//    256 threads fill the very same shared-memory layout with 4-byte cp.async
//    copies instead. Either way out-of-range elements are zero-filled: the
//    guarded zero-fill of the pages' tiled kernels ("矩阵乘法中的分块与数据复用",
//    matmul_l1 and matmul_l1_reg).
//  * Register tiling: each thread owns an 8 x 16 block of C and per k does
//    8 x 16 FFMAs from 8 A values and 16 B values -- the outer product of the
//    pages' matmul_l1_reg ("Register Tiling"), grown to a 128 x 256 block tile
//    and an 8 x 16 microtile so that there are ~21 FFMAs per shared-memory
//    load instruction.
//  * Conflict-free shared memory: A rows are 128 bytes with the 16-byte chunk
//    index XOR-ed by (row % 8); a warp's A loads touch rows r .. r+3 (distinct
//    mod 8), so its four distinct 16-byte chunks land in distinct banks. B
//    rows are read as 8 contiguous float4 per warp (128 bytes). This is the
//    bank-conflict avoidance of "Kernel 优化指南", "Bank Conflict 避免", done by
//    swizzling instead of padding.
//  * Epilogue: 16-byte stores when C permits ("向量化加载"), guarded scalar
//    stores otherwise; each warp store covers 4 rows x 128 contiguous bytes.
#include "kernels.h"
#include "ptx.cuh"

// Schedule parameters of the inner loop (defaults are the measured best):
//   SGEMM_AK      k values per A-fragment load: 4 (float4) or 2 (float2)
//   SGEMM_UNROLL  unroll factor of the loop over A fragments in a k-block
//   SGEMM_B_OUTER 0: FFMAs ordered row-major over the 8 x 16 block (A value
//                 reused across 16 FFMAs); 1: column-major (B value reused)
#ifndef SGEMM_AK
#define SGEMM_AK 4
#endif
#ifndef SGEMM_UNROLL
#define SGEMM_UNROLL 8
#endif
#ifndef SGEMM_B_OUTER
#define SGEMM_B_OUTER 0
#endif
//   SGEMM_FFMA2   1: packed fp32x2 FMAs (fma.rn.f32x2, two IEEE fp32 FMAs per
//                 instruction, same rounding as fmaf); 0: scalar fmaf
#ifndef SGEMM_FFMA2
#define SGEMM_FFMA2 1
#endif
//   SGEMM_PACK_FIRST 1: duplicate all 8 A values of a k step into pairs
//                 before its packed FMAs; 0: each just before its 8 FMAs
#ifndef SGEMM_PACK_FIRST
#define SGEMM_PACK_FIRST 0
#endif
#define GEMM14_PRAGMA(x) _Pragma(#x)
#define GEMM14_UNROLL(n) GEMM14_PRAGMA(unroll n)

namespace gemm14 {
namespace {

using S = SgemmShape;
constexpr int kAK = SGEMM_AK;
static_assert(kAK == 2 || kAK == 4, "A fragments are float2 or float4");

template <int AK> struct AFrag;
template <> struct AFrag<4> {
  using T = float4;
  static __device__ __forceinline__ float get(const float4& v, int kk) {
    return kk == 0 ? v.x : kk == 1 ? v.y : kk == 2 ? v.z : v.w;
  }
};
template <> struct AFrag<2> {
  using T = float2;
  static __device__ __forceinline__ float get(const float2& v, int kk) {
    return kk == 0 ? v.x : v.y;
  }
};

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
template <bool kTma, bool kGeneral>
__device__ __forceinline__ void issue_stage(uint32_t j, int tile, int kb, const TileGrid& grid,
                                            uint8_t* tiles, SgemmSmem& sm,
                                            const CUtensorMap* map_a, const CUtensorMap* map_b,
                                            const GemmArgs& args) {
  // Failure-detection tests: the first stage is never loaded, so every wait
  // for it must expire and report a timeout.
  if (args.fault == kFaultSkipFirstStage && j == 0) return;
  int tm, tn;
  grid.coords(tile, tm, tn);
  const uint32_t s = j % S::STAGES;
  uint8_t* a_st = tiles + s * S::STAGE_BYTES;
  if (kTma) {
    // called by thread 0 only
    mbar_arrive_expect_tx(&sm.full[s], S::STAGE_BYTES);
    tma_load_2d(a_st, map_a, kb * S::BK, tm * S::BM, &sm.full[s]);
    tma_load_2d(a_st + S::A_STAGE_BYTES, map_b, tn * S::BN, kb * S::BK, &sm.full[s]);
  } else {
    // called by all threads: 4096 A + 8192 B elements, 48 per thread
    const float* A = static_cast<const float*>(args.A);
    const float* B = static_cast<const float*>(args.B);
    const uint32_t a_sm = smem_u32(a_st);
    const uint32_t b_sm = a_sm + S::A_STAGE_BYTES;
    const int t = threadIdx.x;
    if (!(kGeneral && args.transa)) {
      const int kl = t & 31;           // k within the block: a warp reads 128 contiguous bytes
      const int k = kb * S::BK + kl;
      const bool k_ok = k < args.K;
#pragma unroll 4
      for (int r = t >> 5; r < S::BM; r += S::THREADS / 32) {
        const int m = tm * S::BM + r;
        const bool in = k_ok && m < args.M;
        cp_async_4(a_sm + a_tile_offset(r, kl),
                   in ? A + static_cast<int64_t>(m) * args.lda + k : A, in ? 4u : 0u);
      }
    } else {
      // A stored K x M: 128 threads read 512 contiguous bytes (128 m) of a k
      // row; the swizzle spreads their 4-byte stores over 8 banks.
      const int ml = t & (S::BM - 1);
      const int m = tm * S::BM + ml;
      const bool m_ok = m < args.M;
#pragma unroll 4
      for (int kr = t / S::BM; kr < S::BK; kr += S::THREADS / S::BM) {
        const int k = kb * S::BK + kr;
        const bool in = m_ok && k < args.K;
        cp_async_4(a_sm + a_tile_offset(ml, kr),
                   in ? A + static_cast<int64_t>(k) * args.lda + m : A, in ? 4u : 0u);
      }
    }
    {
      // 256 threads = 256 columns of one k row. B stored N x K: thread n
      // reads its row's 32 consecutive k (one 128-byte line, kept in L1
      // across the loop); the shared-memory stores stay conflict-free.
      const int nl = t;
      const int n = tn * S::BN + nl;
      const bool n_ok = n < args.N;
      const bool tb = kGeneral && args.transb;
      const int64_t k_stride = tb ? 1 : args.ldb;
      const float* b_col = B + (tb ? static_cast<int64_t>(n) * args.ldb : n);
#pragma unroll 4
      for (int kr = 0; kr < S::BK; ++kr) {
        const int k = kb * S::BK + kr;
        const bool in = n_ok && k < args.K;
        cp_async_4(b_sm + static_cast<uint32_t>(kr * S::BN + nl) * 4,
                   in ? b_col + static_cast<int64_t>(k) * k_stride : B, in ? 4u : 0u);
      }
    }
    cp_async_mbar_arrive_noinc(&sm.full[s]);
  }
}

// kSK: the stream-K schedule (segments, workspace partials); without it the
// schedule is plain data-parallel (tiles w, w+G, ... whole) and none of the
// stream-K machinery is compiled in. kGeneral: stored transposes (cp.async
// loader) and the alpha / beta epilogue are read from args; without it the
// kernel is compiled for untransposed operands and a plain store of C.
template <bool kTma, bool kSK, bool kGeneral>
__global__ void __launch_bounds__(S::THREADS, 1)
    sgemm_simt_kernel(const __grid_constant__ CUtensorMap map_a,
                      const __grid_constant__ CUtensorMap map_b, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = align1024(smem_raw);
  SgemmSmem& sm = *reinterpret_cast<SgemmSmem*>(tiles + S::STAGES * S::STAGE_BYTES);

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
    for (int s = 0; s < S::STAGES; ++s) {
      mbar_init(&sm.full[s], kTma ? 1 : S::THREADS);
      mbar_init(&sm.empty[s], S::WARPS);
    }
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
      issue_stage<kTma, kGeneral>(j, pcur.tile, pcur.kb, tgrid, tiles, sm, &map_a, &map_b, args);
      pcur.next<true>(sm.sched, G);
    } else {
      issue_stage<kTma, kGeneral>(j, dp_tile, dp_kb, tgrid, tiles, sm, &map_a, &map_b, args);
      if (++dp_kb == L) {
        dp_kb = 0;
        dp_tile += G;
      }
    }
  };

  // Prologue: fill the ring (fresh stages need no empty-wait).
  if (producer && n_seg > 0) {
    if (kSK) pcur.start<true>(sm.sched, w, n_seg, L);
    for (; issued < n_iter && issued < static_cast<uint32_t>(S::STAGES); ++issued) load(issued);
  }

  // This thread's rows: warp_m*32 + tr + 4*i (i < 8); columns:
  // warp_n*128 + tc*4 + 32*jj + q (jj, q < 4).
  const int warp_m = warp & 3;  // 4 warps along m (32 rows each)
  const int warp_n = warp >> 2; // 2 warps along n (128 columns each)
  const int tr = lane >> 3;     // 4 thread rows per warp
  const int tc = lane & 7;      // 8 thread columns per warp
  const uint32_t a_thread = static_cast<uint32_t>((warp_m * 32 + tr) * 128);
  const uint32_t b_thread = static_cast<uint32_t>((warp_n * 128 + tc * 4) * 4);

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
#if SGEMM_FFMA2
    // acc2[i][2*jj + h] holds columns 4*jj + 2*h and 4*jj + 2*h + 1 of row i.
    uint64_t acc2[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc2[i][j] = 0ull;
#else
    float acc[8][16];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[i][j] = 0.f;
#endif

    for (int kb = kb0; kb < kb1; ++kb, ++it) {
      const uint32_t s = it % S::STAGES, ph = (it / S::STAGES) & 1;
      if (!mbar_wait(&sm.full[s], ph, wc)) { ok = false; break; }
      const uint8_t* a_st = tiles + s * S::STAGE_BYTES + a_thread;
      const uint8_t* b_st = tiles + s * S::STAGE_BYTES + S::A_STAGE_BYTES + b_thread;
      GEMM14_UNROLL(SGEMM_UNROLL)
      for (int kg = 0; kg < S::BK / kAK; ++kg) {
        // A values for k = kAK*kg .. kAK*kg + kAK-1 of this thread's 8 rows:
        // 16-byte chunk (kAK*kg)/4, XOR-swizzled by (row % 8) = tr + 4*(i % 2).
        const int k0 = kg * kAK;
        const uint32_t x0 = static_cast<uint32_t>((((k0 >> 2) ^ tr) << 4) + (k0 & 3) * 4);
        const uint32_t x1 = x0 ^ 64u;  // rows with (row % 8) >= 4
        typename AFrag<kAK>::T a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          a[i] = *reinterpret_cast<const typename AFrag<kAK>::T*>(a_st + 512 * i +
                                                                 ((i & 1) ? x1 : x0));
#if SGEMM_FFMA2
#pragma unroll
        for (int kk = 0; kk < kAK; ++kk) {
          ulonglong2 b[4];  // (cols 4jj, 4jj+1), (cols 4jj+2, 4jj+3)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
            b[jj] = *reinterpret_cast<const ulonglong2*>(b_st + (k0 + kk) * (S::BN * 4) +
                                                         128 * jj);
#if SGEMM_PACK_FIRST || SGEMM_B_OUTER
          uint64_t a2[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float av = AFrag<kAK>::get(a[i], kk);
            a2[i] = pack2(av, av);
          }
#if SGEMM_B_OUTER
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int i = 0; i < 8; ++i) fma2(acc2[i][2 * jj + h], a2[i], h ? b[jj].y : b[jj].x);
#else
#pragma unroll
          for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              fma2(acc2[i][2 * jj + 0], a2[i], b[jj].x);
              fma2(acc2[i][2 * jj + 1], a2[i], b[jj].y);
            }
#endif
#else
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float av = AFrag<kAK>::get(a[i], kk);
            const uint64_t a2 = pack2(av, av);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              fma2(acc2[i][2 * jj + 0], a2, b[jj].x);
              fma2(acc2[i][2 * jj + 1], a2, b[jj].y);
            }
          }
#endif
        }
#else
#pragma unroll
        for (int kk = 0; kk < kAK; ++kk) {
          float4 b[4];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
            b[jj] = *reinterpret_cast<const float4*>(b_st + (k0 + kk) * (S::BN * 4) + 128 * jj);
#if SGEMM_B_OUTER
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float bv = q == 0 ? b[jj].x : q == 1 ? b[jj].y : q == 2 ? b[jj].z : b[jj].w;
#pragma unroll
              for (int i = 0; i < 8; ++i)
                acc[i][jj * 4 + q] = fmaf(AFrag<kAK>::get(a[i], kk), bv, acc[i][jj * 4 + q]);
            }
          }
#else
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float av = AFrag<kAK>::get(a[i], kk);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              acc[i][jj * 4 + 0] = fmaf(av, b[jj].x, acc[i][jj * 4 + 0]);
              acc[i][jj * 4 + 1] = fmaf(av, b[jj].y, acc[i][jj * 4 + 1]);
              acc[i][jj * 4 + 2] = fmaf(av, b[jj].z, acc[i][jj * 4 + 2]);
              acc[i][jj * 4 + 3] = fmaf(av, b[jj].w, acc[i][jj * 4 + 3]);
            }
          }
#endif
        }
#endif
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[s]);

      // Refill: once every warp is done with iteration it-1, its stage takes
      // iteration it-1+STAGES (one iteration of slack keeps warp 0 from
      // waiting on the slowest warp of the current iteration).
      if (producer && it >= 1 && issued < n_iter && issued == it - 1 + S::STAGES) {
        const uint32_t j = it - 1;
        if (!mbar_wait(&sm.empty[j % S::STAGES], (j / S::STAGES) & 1, wc)) {
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

    // Stream-K: PARTIAL and HEAD segments leave their sums in workspace slot
    // w (tile-local element (r, c) at r * BN + c). A PARTIAL then publishes
    // flag w. A HEAD waits for the later workers' flags and reduces the slots
    // w, w+1, ..., head_last in that order into C, a plain loop over the tile
    // with the accumulators no longer live.
    const int r_loc = warp_m * 32 + tr;   // + 4 i
    const int c_loc = warp_n * 128 + tc * 4;  // + 32 jj
    if (kSK && kind != kSegFull) {
      // PARTIAL -> slot w; HEAD -> slot G + w (a worker may hold both, and a
      // PARTIAL must survive until its owner has read it).
      float* slot = args.partials +
                    static_cast<size_t>(kind == kSegHead ? args.sk.G + w : w) * (S::BM * S::BN);
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          float4 v;
#if SGEMM_FFMA2
          const float2 lo = unpack2(acc2[i][2 * jj]), hi = unpack2(acc2[i][2 * jj + 1]);
          v = make_float4(lo.x, lo.y, hi.x, hi.y);
#else
          v = make_float4(acc[i][jj * 4], acc[i][jj * 4 + 1], acc[i][jj * 4 + 2], acc[i][jj * 4 + 3]);
#endif
          __stcg(reinterpret_cast<float4*>(slot + (r_loc + 4 * i) * S::BN + c_loc + 32 * jj), v);
        }
      if (kind == kSegPartial) {
        __syncthreads();
        if (threadIdx.x == 0) flag_publish(args.flags + w, args.epoch);
        continue;
      }
      const int last = sm.sched.head_last;
      if (threadIdx.x == 0)
        for (int c = w + 1; c <= last; ++c)
          if (!flag_wait(args.flags + c, args.epoch, wc)) break;  // raises abort on expiry
      __syncthreads();  // also orders this CTA's own slot stores before the reads
      if (sm.abort_flag) { ok = false; break; }
      // float4 q of the tile (q = thread + 256 u): row q / 64, columns
      // 4 (q % 64) .. +3 -- a warp covers 512 contiguous bytes of a row.
      // Eight float4 per thread are in flight per slot to hide L2 latency.
      constexpr int kPer = S::BM * S::BN / 4 / S::THREADS;  // 32
#pragma unroll 1
      for (int u0 = 0; u0 < kPer; u0 += 8) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          v[u] = __ldcg(reinterpret_cast<const float4*>(slot) + threadIdx.x + (u0 + u) * S::THREADS);
#pragma unroll 1
        for (int c = w + 1; c <= last; ++c) {
          const float4* src = reinterpret_cast<const float4*>(
              args.partials + static_cast<size_t>(c) * (S::BM * S::BN));
          float4 p[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) p[u] = __ldcg(src + threadIdx.x + (u0 + u) * S::THREADS);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            v[u].x += p[u].x; v[u].y += p[u].y; v[u].z += p[u].z; v[u].w += p[u].w;
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int q = threadIdx.x + (u0 + u) * S::THREADS;
          const int r = q / (S::BN / 4), c4 = (q % (S::BN / 4)) * 4;
          const int row = tm * S::BM + r, col = tn * S::BN + c4;
          if (row >= M) continue;
          float* crow = args.C + static_cast<int64_t>(row) * args.ldc;
          if (args.vec_store && col + 3 < N) {
            epi_store4<kGeneral>(args, crow + col, v[u]);
          } else {
            if (col < N) epi_store1<kGeneral>(args, crow + col, v[u].x);
            if (col + 1 < N) epi_store1<kGeneral>(args, crow + col + 1, v[u].y);
            if (col + 2 < N) epi_store1<kGeneral>(args, crow + col + 2, v[u].z);
            if (col + 3 < N) epi_store1<kGeneral>(args, crow + col + 3, v[u].w);
          }
        }
      }
      continue;
    }

    // Epilogue: rows beyond M and columns beyond N are not written.
    const int row0 = tm * S::BM + r_loc;
    const int col0 = tn * S::BN + c_loc;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = row0 + 4 * i;
      if (row >= M) continue;
      float* crow = args.C + static_cast<int64_t>(row) * args.ldc;
#if SGEMM_FFMA2
      float acc_row[16];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 v = unpack2(acc2[i][j]);
        acc_row[2 * j] = v.x;
        acc_row[2 * j + 1] = v.y;
      }
#else
      const float* acc_row = acc[i];
#endif
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int col = col0 + 32 * jj;
        if (args.vec_store && col + 3 < N) {
          epi_store4<kGeneral>(args, crow + col,
                     make_float4(acc_row[jj * 4 + 0], acc_row[jj * 4 + 1], acc_row[jj * 4 + 2],
                                 acc_row[jj * 4 + 3]));
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (col + q < N) epi_store1<kGeneral>(args, crow + col + q, acc_row[jj * 4 + q]);
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
        const uint32_t first = issued > S::STAGES ? issued - S::STAGES : 0;
        for (uint32_t j = first; j < issued; ++j)
          if (!(args.fault == kFaultSkipFirstStage && j == 0))
            mbar_wait_timed(&sm.full[j % S::STAGES], (j / S::STAGES) & 1, 100000000ull);
      }
    } else {
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
  }
}

template <bool kTma, bool kSK, bool kGeneral>
cudaError_t launch_variant(const CUtensorMap* map_a, const CUtensorMap* map_b,
                           const GemmArgs& args, int grid, cudaStream_t stream) {
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(sgemm_simt_kernel<kTma, kSK, kGeneral>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  CUtensorMap dummy{};
  sgemm_simt_kernel<kTma, kSK, kGeneral><<<grid, S::THREADS, S::SMEM_BYTES, stream>>>(
      map_a ? *map_a : dummy, map_b ? *map_b : dummy, args);
  return cudaGetLastError();
}

template <bool kTma, bool kSK>
cudaError_t launch_epi(const CUtensorMap* map_a, const CUtensorMap* map_b, const GemmArgs& args,
                       int grid, cudaStream_t stream) {
  if (args.transa || args.transb || args.epi != kEpiStore)
    return launch_variant<kTma, kSK, true>(map_a, map_b, args, grid, stream);
  return launch_variant<kTma, kSK, false>(map_a, map_b, args, grid, stream);
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
