// hgemm_tc.cu -- bf16 / fp16 inputs, fp32 accumulate and output, on the
// 5th-generation tensor cores (tcgen05), C = A * B, all row-major.
//
// The pages' tensor-core kernel (WMMA 16x16x16 with half inputs and a float
// accumulator, "Kernel 优化指南", "Level 4: Tensor Cores (WMMA)") and their
// account of wgmma (gpu-hpc-book ch.06 "高级 cuda 特性 —— 从矩阵乘法(gemm)说起",
// "Tensor Cores" / "wgmma": asynchronous D = A*B + D with operands in shared
// memory fed by TMA) are the prior art; on sm_103a the same product is one
// tcgen05.mma issued by a single thread with the accumulator in tensor memory.
//
// Structure (one CTA per SM, persistent over output tiles of BM x BN, BM =
// 128, or 64 for products whose 128-row tiles leave SMs idle):
//   warp 0      producer: TMA loads of A (BM m x 64 k, K-major, 128-byte
//               swizzle) and B (BN/64 boxes of 64 n x 64 k, N-major, 128-byte
//               swizzle) into an S-stage ring (full/empty mbarriers); for
//               operands TMA cannot address, warp 0 and 7 more warps (6 ..)
//               fill the same layout with plain loads and stores;
//   warp 1      allocates 2*BN TMEM columns (two accumulators) and one lane
//               issues 4 x tcgen05.mma (K = 16 each) per 64-deep k-block;
//               tcgen05.commit frees the smem stage and, at the end of a
//               tile, publishes the accumulator;
//   warps 2..5  epilogue: tcgen05.ld 32 lanes x 32 columns at a time, fp32
//               stores to C (16-byte vectors when C allows, guarded edges);
//               while they drain accumulator b the MMA warp fills 1-b.
//               An M = 128 accumulator holds row r in TMEM lane r; an M = 64
//               one holds row r in lane 32 (r / 16) + r % 16, so each
//               epilogue warp finds its 16 rows in the first 16 lanes of its
//               quarter (the other 16 hold nothing of the product).
// Tiles are visited in groups of 16 row-tiles so that the CTAs running at the
// same time share A and B panels in L2.
#include "kernels.h"
#include "ptx.cuh"

namespace gemm14 {
namespace {

using H = HgemmShape;
constexpr int kGroupM = 16;

template <int BM, int BN>
struct TcSmem {
  static constexpr int STAGES = H::stages(BN, BM);
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint64_t partial_stored;  // stream-K: the 4 epilogue warps stored this CTA's partial
  uint64_t flags_ready;     // stream-K: the later workers' partials are published
  uint32_t tmem_base;
  int abort_flag;
  SkTable sched;  // this CTA's segments, decoded once
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Grouped raster: tile t -> (tm, tn), row-tiles in groups of kGroupM.
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int& tm, int& tn) {
  const int per_group = kGroupM * tiles_n;
  const int g = t / per_group;
  const int first_m = g * kGroupM;
  const int gm = min(tiles_m - first_m, kGroupM);
  const int r = t - g * per_group;
  tm = first_m + r % gm;
  tn = r / gm;
}

// Software loader for operands that break TMA's 16-byte rules (any 2-byte
// aligned base and pitch). A row segment is the 64 elements of one 128-byte
// row of the 128-byte swizzled layout TMA would produce. Loader warps copy
// the 16-byte-aligned global chunks that cover a segment straight into shared
// memory with cp.async.cg (no register holds data in flight, L1 is bypassed,
// and several stages are in flight at once), zero-filling bytes past the
// row's last element. When the segment starts sh bytes past a 16-byte
// boundary, it spans nine chunks: the first eight land in the row's eight
// swizzled slots, the ninth in a side buffer, and once they have landed the
// warp shifts the row left by sh bytes in place. sh is the same for every
// segment a loader warp handles (its rows are 8 apart and its k or column
// blocks 64 elements apart). No byte past a row's last element is read; bytes
// before a segment's first element are read only inside the operand (the
// chunk that holds the operand's first element, when that sits past a
// 16-byte boundary, is read element by element).
constexpr int kSoftWarps = H::SOFT_WARPS;  // warps 6 .. 13, two per scheduler; each fills every 8-th row

__device__ __align__(16) uint32_t g_zero_chunk[4];  // source of zero-byte copies

__device__ __forceinline__ void cp_async_16(uint32_t smem_dst, const void* src,
                                            uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds128u(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void sts128u(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// A bounded wait like mbar_wait whose polls let the thread sleep until the
// phase completes (or about kSleepHintNs pass): for the roles of the
// software-loader variants that wait long (the epilogue for a tile's whole
// main loop, the MMA warp for the loader warps), so that their polling takes
// no issue slots from the loader warps on the same schedulers.
constexpr uint32_t kSleepHintNs = 20000;

__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSleepHintNs)
      : "memory");
  return done != 0;
}

static __device__ __noinline__ bool mbar_wait_sleep_slow(uint64_t* bar, uint32_t parity,
                                                         const WaitCtx& w) {
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (*w.abort_flag) return false;
    if (globaltimer_ns() - t0 > w.limit_ns) {
      atomicOr(w.err, kDevErrTimeout);
      *w.abort_flag = 1;
      return false;
    }
  }
}

// mbar_wait for the TMA variants, the sleeping wait for the others.
template <bool kSleep>
__device__ __forceinline__ bool role_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  return kSleep ? mbar_wait_sleep_slow(bar, parity, w) : mbar_wait_slow<false>(bar, parity, w);
}

// Copy of one 16-byte chunk at global byte address cs into shared memory at
// d: the bytes below the row end re (zeros above). Bytes below the operand's
// base are not read (their slots are shifted out later).
__device__ __forceinline__ void copy_chunk(uint32_t d, uintptr_t cs, uintptr_t base,
                                           uintptr_t re, bool row_ok) {
  if (row_ok && cs < base) {
#pragma unroll 1
    for (int p = 0; p < 16; p += 2) {
      const uintptr_t a = cs + p;
      sts16(d + p, a >= base && a < re ? __ldg(reinterpret_cast<const uint16_t*>(a))
                                       : static_cast<uint16_t>(0));
    }
    return;
  }
  const uint32_t bytes =
      !row_ok || cs >= re ? 0u : re - cs >= 16 ? 16u : static_cast<uint32_t>(re - cs);
  cp_async_16(d, bytes ? reinterpret_cast<const void*>(cs) : g_zero_chunk, bytes);
}

// Bytes sh .. sh + 15 of the 32 bytes X, Y, sh = 4 Q + fs / 8 (fs 0 or 16).
template <int Q>
__device__ __forceinline__ uint4 shift_chunk(const uint4& X, const uint4& Y, uint32_t fs) {
  const uint32_t w[8] = {X.x, X.y, X.z, X.w, Y.x, Y.y, Y.z, Y.w};
  return make_uint4(__funnelshift_r(w[Q], w[Q + 1], fs), __funnelshift_r(w[Q + 1], w[Q + 2], fs),
                    __funnelshift_r(w[Q + 2], w[Q + 3], fs),
                    __funnelshift_r(w[Q + 3], w[Q + 4], fs));
}

// One operand's share of a stage for loader warp `part`. K-major (KMAJ): E
// tile rows from r0 (matrix rows r0 + part + 8 s) by 64 k from c0, segment s
// in smem row part + 8 s. MN-major: E / 64 boxes of 64 columns by 64 k rows
// (8 KB each); segment s is k row r0 + part + 8 (s % 8) of box s / 8,
// columns c0 + 64 (s / 8) ...
// Lane l copies chunk j = l % 8 of segments 4 t + l / 8, t = 0 .. NSEG / 4 - 1:
// relative to the lane's first segment, iteration t is rows_t(t) matrix rows,
// cols_t(t) elements and smem_t(t) shared bytes further on.
template <bool KMAJ, int E>
struct SoftOperand {
  static constexpr int NSEG = E / kSoftWarps;
  static constexpr int T = NSEG / 4;
  static constexpr int COLS = KMAJ ? 64 : E;  // elements of a stage's row span
  __device__ __forceinline__ static constexpr int rows_t(int t) { return KMAJ ? 32 * t : 32 * (t & 1); }
  __device__ __forceinline__ static constexpr int cols_t(int t) { return KMAJ ? 0 : 64 * (t >> 1); }
  __device__ __forceinline__ static constexpr uint32_t smem_t(int t) {
    return KMAJ ? 4096u * t : 4096u * (t & 1) + 8192u * (t >> 1);
  }
  // segment s of the side chunks: rows and columns past the warp's first
  __device__ __forceinline__ static int rows_s(int s) { return KMAJ ? 8 * s : 8 * (s & 7); }
  __device__ __forceinline__ static int cols_s(int s) { return KMAJ ? 0 : 64 * (s >> 3); }

  const uint16_t* src;
  int64_t ld;
  int r0, c0, nrows, ncols, part;
  uint32_t dst;  // shared address of the operand tile

  // Global byte address of the warp's first segment's first element.
  __device__ __forceinline__ uintptr_t first() const {
    return reinterpret_cast<uintptr_t>(src) +
           2 * static_cast<uintptr_t>(static_cast<int64_t>(r0 + part) * ld + c0);
  }
  __device__ __forceinline__ int shift() const { return static_cast<int>(first() & 15); }

  // Every row of the warp's segments is in the matrix, every chunk they need
  // lies in its row, and none starts below the operand's base.
  __device__ __forceinline__ bool interior(int sh) const {
    const int last_row = r0 + part + (KMAJ ? 8 * (NSEG - 1) : 56);
    return last_row < nrows && 2 * (c0 + COLS) - sh + (sh ? 16 : 0) <= 2 * ncols &&
           first() - sh >= reinterpret_cast<uintptr_t>(src);
  }

  __device__ __forceinline__ void issue(uint32_t side, int lane) const {
    const int sh = shift();
    const int j = lane & 7, s4 = lane >> 3;
    const uint32_t d = dst + (part + kSoftWarps * s4) * 128 + ((j ^ part) << 4);
    const uintptr_t rstep = 2 * static_cast<uintptr_t>(ld);
    if (interior(sh)) {
      // Whole 16-byte chunks, no bounds to check.
      const uintptr_t p = first() - sh + 16 * j + (kSoftWarps * s4) * rstep;
#pragma unroll
      for (int t = 0; t < T; ++t)
        cp_async_16(d + smem_t(t),
                    reinterpret_cast<const void*>(p + rows_t(t) * rstep + 2 * cols_t(t)), 16);
      if (sh) {
#pragma unroll
        for (int u = 0; u < (NSEG + 31) / 32; ++u) {
          const int s = 32 * u + lane;
          if (s < NSEG)
            cp_async_16(side + 128 * s,
                        reinterpret_cast<const void*>(first() - sh + 128 + rows_s(s) * rstep +
                                                      2 * cols_s(s)),
                        16);
        }
      }
      return;
    }
    // Edge of the matrix: chunk by chunk, bounded by the row's end.
    const uintptr_t base = reinterpret_cast<uintptr_t>(src);
    const int row1 = r0 + part + kSoftWarps * s4;
    const uintptr_t rs1 = base + 2 * static_cast<uintptr_t>(static_cast<int64_t>(row1) * ld);
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const int row = row1 + rows_t(t);
      const uintptr_t rs = rs1 + rows_t(t) * rstep;
      const uintptr_t cs = ((rs + 2 * static_cast<uintptr_t>(c0 + cols_t(t))) & ~uintptr_t(15)) + 16 * j;
      copy_chunk(d + smem_t(t), cs, base, rs + 2 * static_cast<uintptr_t>(ncols), row < nrows);
    }
    if (sh) {
#pragma unroll
      for (int u = 0; u < (NSEG + 31) / 32; ++u) {
        const int s = 32 * u + lane;
        if (s < NSEG) {
          const int row = r0 + part + rows_s(s);
          const uintptr_t rs = base + 2 * static_cast<uintptr_t>(static_cast<int64_t>(row) * ld);
          const uintptr_t cs = ((rs + 2 * static_cast<uintptr_t>(c0 + cols_s(s))) & ~uintptr_t(15)) + 128;
          copy_chunk(side + 128 * s, cs, base, rs + 2 * static_cast<uintptr_t>(ncols), row < nrows);
        }
      }
    }
  }

  // Chunks of RB iterations are read before any is rewritten, so that their
  // shared-memory latencies overlap.
  template <int Q>
  __device__ __forceinline__ void realign_q(uint32_t side, int lane, uint32_t fs) const {
    constexpr int RB = T < 8 ? T : 8;
    const int j = lane & 7, s4 = lane >> 3;
    const uint32_t rowb = dst + (part + kSoftWarps * s4) * 128;
    const uint32_t dx = rowb + ((j ^ part) << 4);
    const uint32_t dy = rowb + (((j + 1) ^ part) << 4);
    const uint32_t ds = side + 128 * s4;
#pragma unroll
    for (int t0 = 0; t0 < T; t0 += RB) {
      uint4 X[RB], Y[RB];
#pragma unroll
      for (int u = 0; u < RB; ++u) {
        X[u] = lds128u(dx + smem_t(t0 + u));
        Y[u] = lds128u(j < 7 ? dy + smem_t(t0 + u) : ds + 512 * (t0 + u));
      }
      __syncwarp();  // every lane has read its chunks before any is overwritten
#pragma unroll
      for (int u = 0; u < RB; ++u) sts128u(dx + smem_t(t0 + u), shift_chunk<Q>(X[u], Y[u], fs));
    }
  }

  // After every lane's copies of the stage have landed (and a __syncwarp).
  __device__ __forceinline__ void realign(uint32_t side, int lane) const {
    const int sh = shift();
    const uint32_t fs = 8u * static_cast<uint32_t>(sh & 3);
    switch (sh >> 2) {
      case 0: if (sh) realign_q<0>(side, lane, fs); break;
      case 1: realign_q<1>(side, lane, fs); break;
      case 2: realign_q<2>(side, lane, fs); break;
      default: realign_q<3>(side, lane, fs); break;
    }
  }
};

// Loader warp `part`'s share of one stage: the operands of kSoft (bit 0: A,
// bit 1: B; TMA loads the other). A stored M x K is K-major, stored K x M
// (transa) MN-major; B stored K x N is MN-major, stored N x K (transb)
// K-major. side: the stage's side buffer, one 128-byte row per segment index
// ((BM + BN) / 8 rows: A's segments, then B's), in which warp `part` owns the
// 16 bytes at 16 part; so a segment's ninth chunk sits in the one bank group
// the other seven lanes of its quarter-warp do not read in the realignment.
template <int BM, int BN, int kSoft>
struct SoftStage {
  static constexpr int A_BYTES = BM * H::BK * 2;
  static constexpr int SIDE_BYTES = (BM + BN) / kSoftWarps * 128;  // one stage, all warps
  template <class F>
  __device__ __forceinline__ static void each(const GemmArgs& args, uint32_t a_st, int tm, int tn,
                                              int kb, int part, uint32_t side, F&& f) {
    const uint16_t* A = static_cast<const uint16_t*>(args.A);
    const uint16_t* B = static_cast<const uint16_t*>(args.B);
    const uint32_t b_st = a_st + A_BYTES;
    const uint32_t side_b = side + BM / kSoftWarps * 128;
    const int k0 = kb * H::BK;
    if (kSoft & 1) {
      if (args.transa)
        f(SoftOperand<false, BM>{A, args.lda, k0, tm * BM, args.K, args.M, part, a_st}, side);
      else
        f(SoftOperand<true, BM>{A, args.lda, tm * BM, k0, args.M, args.K, part, a_st}, side);
    }
    if (kSoft & 2) {
      if (args.transb)
        f(SoftOperand<true, BN>{B, args.ldb, tn * BN, k0, args.N, args.K, part, b_st}, side_b);
      else
        f(SoftOperand<false, BN>{B, args.ldb, k0, tn * BN, args.K, args.N, part, b_st}, side_b);
    }
  }
  __device__ __forceinline__ static void issue(const GemmArgs& args, uint32_t a_st, int tm, int tn,
                                               int kb, int lane, int part, uint32_t side) {
    each(args, a_st, tm, tn, kb, part, side,
         [&](const auto& op, uint32_t sd) { op.issue(sd, lane); });
  }
  __device__ __forceinline__ static void realign(const GemmArgs& args, uint32_t a_st, int tm,
                                                 int tn, int kb, int lane, int part,
                                                 uint32_t side) {
    each(args, a_st, tm, tn, kb, part, side,
         [&](const auto& op, uint32_t sd) { op.realign(sd, lane); });
  }
};

// Stream-K fixup: a tile's owner reads the partial sums of its later workers
// kPre at a time. Workspace slot cw holds worker cw's BM x BN partial tile,
// row-major; this thread's row is r_loc and its chunk the 32 columns from
// 32 c. Loads of n (<= kPre) consecutive workers from cw0, all issued before
// any is used.
constexpr int kPre = 4;

// (Slot w holds worker w's BM x BN partial sums; args.sk.G slots. A load the
// bounds checks reject reads as zeros.)
template <int BM, int BN, int NP>
__device__ __forceinline__ void load_partials(float4 (&p)[NP][8], const GemmArgs& args, int cw0,
                                              int n, int r_loc, int c) {
#pragma unroll
  for (int j = 0; j < NP; ++j) {
    if (j < n) {
      const int64_t off = (static_cast<int64_t>(cw0 + j) * BM + r_loc) * BN + c * 32;
      const bool ok = dev_check(slot_span_ok(off, cw0 + j, BM * BN, args.sk.G, 32), args.err);
      const float* src = args.partials + off;
#pragma unroll
      for (int v = 0; v < 8; ++v)
        p[j][v] = ok ? __ldcg(reinterpret_cast<const float4*>(src + 4 * v))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// r += p[0] + ... + p[n-1], one worker after another (a fixed order).
template <int NP>
__device__ __forceinline__ void add_partials(uint32_t (&r)[32], const float4 (&p)[NP][8], int n) {
#pragma unroll
  for (int j = 0; j < NP; ++j) {
    if (j < n) {
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        r[4 * v + 0] = __float_as_uint(__uint_as_float(r[4 * v + 0]) + p[j][v].x);
        r[4 * v + 1] = __float_as_uint(__uint_as_float(r[4 * v + 1]) + p[j][v].y);
        r[4 * v + 2] = __float_as_uint(__uint_as_float(r[4 * v + 2]) + p[j][v].z);
        r[4 * v + 3] = __float_as_uint(__uint_as_float(r[4 * v + 3]) + p[j][v].w);
      }
    }
  }
}

// kSK: the stream-K schedule (segments, workspace partials); without it the
// schedule is plain data-parallel and none of the stream-K code is compiled in.
// kGeneral: stored transposes and the alpha / beta epilogue are read from
// args; without it the kernel is compiled for untransposed operands and a
// plain store of C (the software-loader variants are always general).
// kSoft: the operands the software loader copies (bit 0: A, bit 1: B); TMA
// loads the others. Threads of a variant: the six warps of the roles, plus the
// software loader's eight warps (6 .. 13) when kSoft is not 0 (warp 0, TMA's
// producer, then loads only the operands TMA can read, or idles).
template <int kSoft>
constexpr int tc_threads() { return kSoft == 0 ? H::THREADS : H::SOFT_THREADS; }

template <int BM, int BN, int kSoft, bool kSK, bool kGeneral>
__global__ void __launch_bounds__(tc_threads<kSoft>(), 1)
    hgemm_tc_kernel(const __grid_constant__ CUtensorMap map_a,
                    const __grid_constant__ CUtensorMap map_b,
                    const __grid_constant__ CUtensorMap map_c, const GemmArgs args,
                    const uint32_t idesc) {
  const int transa = kGeneral ? args.transa : 0;
  const int transb = kGeneral ? args.transb : 0;
  static_assert(BM == 64 || BM == 128, "tile rows");
  static_assert(kSoft == 0 || kGeneral, "software-loader variants are general");
  constexpr bool kTma = kSoft == 0;             // every operand by TMA
  constexpr bool kTmaPart = kSoft != 3;         // warp 0 issues TMA loads
  // bytes a stage's TMA loads bring (the operands the software loader leaves)
  constexpr uint32_t TMA_BYTES = ((kSoft & 1) ? 0u : uint32_t(BM * H::BK * 2)) +
                                 ((kSoft & 2) ? 0u : uint32_t(H::BK * BN * 2));
  constexpr int STAGES = H::stages(BN, BM);
  constexpr int A_BYTES = BM * H::BK * 2;      // 16 KB (BM 128) or 8 KB (BM 64)
  constexpr int B_BYTES = H::BK * BN * 2;      // BN/64 boxes of 8 KB
  constexpr int OUT_BUF_BYTES = H::out_buf_bytes(BM);
  constexpr int ROWS_PER_WARP = BM / 4;        // rows each epilogue warp stores
  constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr uint32_t TMEM_COLS = 2 * BN;

  static_assert(sizeof(TcSmem<BM, BN>) <= H::SMEM_RESERVE, "barrier block exceeds its reserve");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = align1024(smem_raw);
  uint8_t* out_stage = tiles + STAGES * STAGE_BYTES;  // epilogue staging for C
  TcSmem<BM, BN>& sm = *reinterpret_cast<TcSmem<BM, BN>*>(out_stage + H::out_bytes(BM));
  // Plain variant with a 16-byte-aligned C: the epilogue writes C with TMA
  // stores of 32 x 32 blocks staged in shared memory.
  const bool tma_c = !kGeneral && args.vec_store;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int M = args.M, N = args.N;
  const int tiles_m = (M + BM - 1) / BM;
  const int tiles_n = (N + BN - 1) / BN;
  const int w = blockIdx.x;  // this CTA's worker index in the schedule
  const WaitCtx wc{args.err, &sm.abort_flag, args.wait_limit_ns, 0u};
  uint32_t prod_it = 0;
  bool mma_issued = false;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // one TMA arrival (with the stage's bytes) and/or every loader thread's
      mbar_init(&sm.full[s], (kTmaPart ? 1 : 0) + (kSoft ? 32 * kSoftWarps : 0));
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], 4);
    }
    mbar_init(&sm.drain, 1);
    mbar_init(&sm.partial_stored, 4);
    mbar_init(&sm.flags_ready, 1);
    sm.abort_flag = 0;
    if (kSK) {
      sm.sched.fill(args.sk, w);
      if (sm.sched.n_sk > kMaxSk) {  // cannot happen for schedules make_stream_k builds
        atomicOr(args.err, kDevErrBadConfig);
        sm.abort_flag = 1;
      }
    }
    fence_barrier_init();
    if (!(kSoft & 1)) tma_prefetch_desc(&map_a);
    if (!(kSoft & 2)) tma_prefetch_desc(&map_b);
    if (tma_c) tma_prefetch_desc(&map_c);
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // Everything above touched only shared memory, TMEM and the kernel's
  // parameters (and, on a bad schedule, OR-ed a bit into the error word, which
  // commutes with an earlier grid's ORs); from here on global memory is read
  // and written.
  grid_dependency_wait();
  grid_launch_dependents();
  const uint32_t tmem_base = sm.tmem_base;
  const int G = args.sk.G, L = args.sk.L;
  const int n_seg = kSK ? (sm.abort_flag ? 0 : sm.sched.segments()) : args.sk.dp_count(w);
  // Segment i: data-parallel tile w + i * G whole, or the decoded stream-K table.
  auto segment = [&](int i, int& tile, int& kb0, int& kb1, int& kind) {
    if (kSK) {
      sm.sched.get(i, tile, kb0, kb1, kind);
    } else {
      tile = w + i * G;
      kb0 = 0;
      kb1 = L;
      kind = kSegFull;
    }
  };

  if ((kTmaPart && warp == 0) || (kSoft && warp >= 6)) {
    // ------------------------------------------------------------ producer
    // Segment by segment; a segment's tile coordinates are computed once.
    // Software loader: warps 6 .. 13 each fill their share of every stage's
    // kSoft operands, DEPTH stages in flight; warp 0 loads the others by TMA
    // (or idles when kSoft covers both).
    if (kSoft && warp >= 6) {
      using SS = SoftStage<BM, BN, kSoft>;
      // Stages a loader warp keeps in flight: all but the one the MMA reads,
      // as far as the side buffers fit in the epilogue staging they reuse.
      constexpr int DEPTH = (STAGES - 1) * SS::SIDE_BYTES <= H::out_bytes(BM)
                                ? STAGES - 1
                                : H::out_bytes(BM) / SS::SIDE_BYTES;
      static_assert(DEPTH >= 2, "software loader depth");
      const int part = warp - 6;
      const uint32_t tiles_u = smem_u32(tiles);
      // The software-loader variants are general (no TMA-store epilogue): the
      // epilogue staging holds the side chunks of the stages in flight.
      const uint32_t side_u = smem_u32(out_stage) + 16 * part;
      constexpr uint32_t SIDE_STAGE = SS::SIDE_BYTES;
      // Stages in flight, oldest first: tile (tm, tn) and k block (< 0: the
      // stage is not loaded and not announced).
      int q_tm[DEPTH] = {}, q_tn[DEPTH] = {}, q_kb[DEPTH] = {};
      int q_n = 0;
      uint32_t done_it = 0;
      // The oldest stage's copies have landed (every lane waited, then the
      // warp synchronised): realign, fence the generic-proxy writes for
      // tcgen05.mma, announce.
      auto complete_oldest = [&]() {
        const uint32_t s = done_it % STAGES;
        if (q_kb[0] >= 0) {
          SS::realign(args, tiles_u + s * STAGE_BYTES, q_tm[0], q_tn[0], q_kb[0], lane, part,
                      side_u + (done_it % DEPTH) * SIDE_STAGE);
          fence_proxy_async_smem();
          mbar_arrive(&sm.full[s]);
        }
#pragma unroll
        for (int j = 0; j + 1 < DEPTH; ++j) {
          q_tm[j] = q_tm[j + 1];
          q_tn[j] = q_tn[j + 1];
          q_kb[j] = q_kb[j + 1];
        }
        --q_n;
        ++done_it;
      };
      bool ok = true;
      for (int seg = 0; seg < n_seg && ok; ++seg) {
        int tile, kb0, kb1, kind, tm, tn;
        segment(seg, tile, kb0, kb1, kind);
        tile_coords(tile, tiles_m, tiles_n, tm, tn);
        for (int kb = kb0; kb < kb1; ++kb, ++prod_it) {
          const uint32_t s = prod_it % STAGES, ph = (prod_it / STAGES) & 1;
          int got = 1;
          if (lane == 0) got = mbar_wait(&sm.empty[s], ph ^ 1, wc) ? 1 : 0;
          got = __shfl_sync(0xffffffffu, got, 0);
          if (!got) { ok = false; break; }
          // Failure-detection tests: the first stage is never loaded.
          const bool skip = args.fault == kFaultSkipFirstStage && prod_it == 0;
          if (!skip)
            SS::issue(args, tiles_u + s * STAGE_BYTES, tm, tn, kb, lane, part,
                      side_u + (prod_it % DEPTH) * SIDE_STAGE);
          cp_async_commit();
#pragma unroll
          for (int j = 0; j < DEPTH; ++j) {
            if (j == q_n) {
              q_tm[j] = tm;
              q_tn[j] = tn;
              q_kb[j] = skip ? -1 : kb;
            }
          }
          if (++q_n == DEPTH) {
            cp_async_wait<DEPTH - 1>();
            __syncwarp();
            complete_oldest();
          }
        }
      }
      cp_async_wait<0>();
      __syncwarp();
      while (q_n > 0) complete_oldest();
    } else if (lane == 0) {
      bool ok = true;
      for (int seg = 0; seg < n_seg && ok; ++seg) {
        int tile, kb0, kb1, kind, tm, tn;
        segment(seg, tile, kb0, kb1, kind);
        tile_coords(tile, tiles_m, tiles_n, tm, tn);
        for (int kb = kb0; kb < kb1; ++kb, ++prod_it) {
          const uint32_t s = prod_it % STAGES, ph = (prod_it / STAGES) & 1;
          if (!mbar_wait(&sm.empty[s], ph ^ 1, wc)) { ok = false; break; }
          // Failure-detection tests: the first stage is never loaded.
          if (args.fault == kFaultSkipFirstStage && prod_it == 0) continue;
          uint8_t* a_st = tiles + s * STAGE_BYTES;
          uint8_t* b_st = a_st + A_BYTES;
          mbar_arrive_expect_tx(&sm.full[s], TMA_BYTES);
          // A: one box of 64 k x BM m, or (stored K x M) BM / 64 boxes of 64 m x 64 k.
          if (kSoft & 1) {
            // the software loader's
          } else if (!transa) {
            tma_load_2d(a_st, &map_a, kb * H::BK, tm * BM, &sm.full[s]);
          } else {
#pragma unroll
            for (int c = 0; c < BM / 64; ++c)
              tma_load_2d(a_st + c * (64 * H::BK * 2), &map_a, tm * BM + c * 64, kb * H::BK,
                          &sm.full[s]);
          }
          // B: BN / 64 boxes of 64 n x 64 k, or (stored N x K) one box of 64 k x BN n.
          if (kSoft & 2) {
            // the software loader's
          } else if (!transb) {
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_2d(b_st + c * (64 * H::BK * 2), &map_b, tn * BN + c * 64, kb * H::BK,
                          &sm.full[s]);
          } else {
            tma_load_2d(b_st, &map_b, kb * H::BK, tn * BN, &sm.full[s]);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const OperandDesc a_op = operand_desc(transa == 0);
      const OperandDesc b_op = operand_desc(transb != 0);
      bool ok = true;
      uint32_t it = 0;
      for (int seg = 0; seg < n_seg && ok; ++seg) {
        int tile, kb0, kb1, kind;
        segment(seg, tile, kb0, kb1, kind);
        const int b = seg & 1;
        const uint32_t aph = (seg >> 1) & 1;
        if (!role_wait<kSoft != 0>(&sm.acc_empty[b], aph ^ 1, wc)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!role_wait<kSoft != 0>(&sm.full[s], ph, wc)) { ok = false; break; }
          tc_fence_after_sync();
          const uint32_t a_addr = smem_u32(tiles + s * STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < H::BK / 16; ++kk) {
            const uint64_t a_desc = smem_desc_sw128(a_addr + kk * a_op.step, a_op.lbo, 1024);
            const uint64_t b_desc = smem_desc_sw128(b_addr + kk * b_op.step, b_op.lbo, 1024);
            tc_mma_f16(d_tmem, a_desc, b_desc, idesc, kb > kb0 || kk != 0);
          }
          mma_issued = true;
          tc_commit(&sm.empty[s]);
        }
        if (!ok) break;
        tc_commit(&sm.acc_full[b]);
      }
    }
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    // This thread's row within the tile: lane l of the quarter for BM 128;
    // for BM 64 lanes 0..15 hold rows 16 q + l and lanes 16..31 no row (they
    // take part in the warp-wide TMEM loads and the staging, but load and
    // store no data of their own).
    const bool has_row = BM == 128 || lane < 16;
    const int r_loc = q * ROWS_PER_WARP + (BM == 128 ? lane : (lane & 15));
    uint8_t* out_buf = out_stage + q * 2 * OUT_BUF_BYTES;
    int ob = 0;
    for (int seg = 0; seg < n_seg; ++seg) {
      int tile, kb0, kb1, kind, tm, tn;
      segment(seg, tile, kb0, kb1, kind);
      tile_coords(tile, tiles_m, tiles_n, tm, tn);
      const int b = seg & 1;
      const uint32_t aph = (seg >> 1) & 1;
      // One lane waits; the warp then proceeds converged (tcgen05.ld is .sync.aligned).
      int got = 1;
      if (lane == 0) got = role_wait<kSoft != 0>(&sm.acc_full[b], aph, wc) ? 1 : 0;
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      if (kSK && kind == kSegHead) {
        // Wait for every later worker holding part of this tile (one lane of
        // warp 2 polls their flags; the other warps wait on flags_ready).
        // A worker has at most one HEAD segment: the barrier's first phase.
        if (warp == 2 && lane == 0) {
          bool all = true;
          for (int c = w + 1; c <= sm.sched.head_last && all; ++c) {
            if (!dev_check(index_ok(c, args.sk.G), args.err)) break;
            all = flag_wait(args.flags + c, args.epoch, wc);
            if (all) flag_clear(args.flags + c);
          }
          if (all) mbar_arrive(&sm.flags_ready);
        }
        if (lane == 0) got = mbar_wait(&sm.flags_ready, 0, wc) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) break;
      }
      tc_fence_after_sync();
      const int row = tm * BM + r_loc;
      float* crow = args.C + static_cast<int64_t>(row) * args.ldc;
      float* prow = args.partials + (static_cast<size_t>(w) * BM + r_loc) * BN;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(b * BN);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        // HEAD: fetch the first (up to) kPre contributors' partials of this
        // chunk before the TMEM read, all loads in flight at once, so that
        // their latencies overlap each other and the TMEM read's.
        // (the software-loader variants, whose 448 threads allow 146 registers
        // each, prefetch one partial at a time)
        constexpr int NP = kTma ? kPre : 1;
        float4 pre[NP][8];
        const int n_pre =
            (kSK && kind == kSegHead && has_row) ? min(NP, sm.sched.head_last - w) : 0;
        if (kSK) load_partials<BM, BN, NP>(pre, args, w + 1, n_pre, r_loc, c);
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c * 32, r);
        tc_wait_ld();
        if (kSK && kind == kSegPartial) {
          // Stream-K: partial sums of this tile go to workspace slot w.
          if (!has_row ||
              !dev_check(slot_span_ok(prow + c * 32 - args.partials, w, BM * BN, args.sk.G, 32),
                         args.err))
            continue;
#pragma unroll
          for (int v = 0; v < 8; ++v)
            __stcg(reinterpret_cast<float4*>(prow + c * 32 + 4 * v),
                   make_float4(__uint_as_float(r[4 * v + 0]), __uint_as_float(r[4 * v + 1]),
                               __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3])));
          continue;
        }
        if (kSK && kind == kSegHead) {
          // Add the later workers' partial sums, in worker order: the
          // prefetched group, then further groups of kPre (loads first).
          add_partials<NP>(r, pre, n_pre);
          for (int cw0 = w + 1 + NP; has_row && cw0 <= sm.sched.head_last; cw0 += NP) {
            const int n = min(NP, sm.sched.head_last - cw0 + 1);
            load_partials<BM, BN, NP>(pre, args, cw0, n, r_loc, c);
            add_partials<NP>(r, pre, n);
          }
        }
        const int col0 = tn * BN + c * 32;
        // A TMA store clips a row at 16-byte granularity, not per element: a
        // chunk that runs past a column count N that is not a multiple of 4
        // would write up to 3 floats past column N - 1 (into the pitch's
        // padding), so that chunk takes the guarded direct stores.
        if (tma_c && (col0 + 32 <= N || (N & 3) == 0)) {
          // Row i of the 32 x 32 block goes to staging row i with its eight
          // 16-byte chunks permuted by i mod 8 (the 128-byte swizzle of
          // map_c); the TMA store leaves out rows >= M (and columns >= N,
          // as above). The buffer's store of two chunks ago has been read
          // out first.
          uint8_t* buf = out_buf + ob * OUT_BUF_BYTES;
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
          const uint32_t rb = smem_u32(buf) + static_cast<uint32_t>(lane * 128);
          if (has_row) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                               rb + static_cast<uint32_t>(((v ^ lane) & 7) << 4)),
                           "r"(r[4 * v + 0]), "r"(r[4 * v + 1]), "r"(r[4 * v + 2]),
                           "r"(r[4 * v + 3])
                           : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&map_c, buf, col0, tm * BM + q * ROWS_PER_WARP);
            bulk_commit();
          }
          ob ^= 1;
        } else if (has_row && row < M) {
          if (args.vec_store && col0 + 32 <= N) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              epi_store4<kGeneral>(args, crow + col0 + 4 * v,
                         make_float4(__uint_as_float(r[4 * v + 0]), __uint_as_float(r[4 * v + 1]),
                                     __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3])));
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (col0 + j < N) epi_store1<kGeneral>(args, crow + col0 + j, __uint_as_float(r[j]));
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.acc_empty[b]);
      if (kSK && kind == kSegPartial) {
        // All four warps' partial stores precede the flag. A worker has at
        // most one PARTIAL segment: the barrier's first phase.
        if (lane == 0) mbar_arrive(&sm.partial_stored);
        if (warp == 2 && lane == 0 && mbar_wait(&sm.partial_stored, 0, wc) &&
            dev_check(index_ok(w, args.sk.G), args.err))
          flag_publish(args.flags + w, args.epoch);
      }
    }
    // The TMA stores have finished (their reads of the staging buffers, and
    // their writes) before the CTA may exit.
    if (tma_c && lane == 0) bulk_wait_all();
  }

  // On abort: let issued MMAs and TMA loads finish (bounded) before TMEM is
  // freed and the CTA's shared memory is released.
  __syncthreads();
  if (sm.abort_flag) {
    if (warp == 1 && lane == 0 && mma_issued) {
      tc_commit(&sm.drain);
      mbar_wait_timed(&sm.drain, 0, 100000000ull);
    }
    if (kTmaPart && warp == 0 && lane == 0) {
      const uint32_t first = prod_it > STAGES ? prod_it - STAGES : 0;
      for (uint32_t j = first; j < prod_it; ++j)
        if (!(args.fault == kFaultSkipFirstStage && j == 0))
          mbar_wait_timed(&sm.full[j % STAGES], (j / STAGES) & 1, 100000000ull);
    }
    __syncthreads();
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int BM, int BN, int kSoft, bool kSK, bool kGeneral>
cudaError_t launch_variant(const CUtensorMap* map_a, const CUtensorMap* map_b,
                           const CUtensorMap* map_c, const GemmArgs& args, uint32_t idesc,
                           int grid, cudaStream_t stream) {
  static DeviceOnce configured;
  const cudaError_t e = set_smem_once(configured, hgemm_tc_kernel<BM, BN, kSoft, kSK, kGeneral>,
                                      H::smem_bytes(BN, BM));
  if (e != cudaSuccess) return e;
  CUtensorMap dummy{};
  return launch_kernel(hgemm_tc_kernel<BM, BN, kSoft, kSK, kGeneral>, dim3(grid),
                       dim3(tc_threads<kSoft>()), H::smem_bytes(BN, BM), stream,
                       map_a ? *map_a : dummy, map_b ? *map_b : dummy, map_c ? *map_c : dummy,
                       args, idesc);
}

template <int BM, int BN, int kSoft, bool kSK>
cudaError_t launch_epi(const CUtensorMap* map_a, const CUtensorMap* map_b,
                       const CUtensorMap* map_c, const GemmArgs& args, uint32_t idesc, int grid,
                       cudaStream_t stream) {
  if (kSoft || args.transa || args.transb || args.epi != kEpiStore)
    return launch_variant<BM, BN, kSoft, kSK, true>(map_a, map_b, map_c, args, idesc, grid,
                                                    stream);
  return launch_variant<BM, BN, kSoft, kSK, kSoft != 0>(map_a, map_b, map_c, args, idesc, grid,
                                                        stream);
}

// One operand by software and the other by TMA is compiled for the
// data-parallel schedule only: a split product whose operand TMA cannot read
// (its workspace too small to re-pitch it) loads both by software.
template <int BM, int BN, int kSoft>
cudaError_t launch_bn(const CUtensorMap* map_a, const CUtensorMap* map_b,
                      const CUtensorMap* map_c, const GemmArgs& args, uint32_t idesc, int grid,
                      cudaStream_t stream) {
  if (args.sk.dp_tiles < args.sk.tiles)
    return launch_epi<BM, BN, kSoft == 0 ? 0 : 3, true>(map_a, map_b, map_c, args, idesc, grid,
                                                        stream);
  return launch_epi<BM, BN, kSoft, false>(map_a, map_b, map_c, args, idesc, grid, stream);
}

template <int BM, int kSoft>
cudaError_t launch_bm(int bn, const CUtensorMap* map_a, const CUtensorMap* map_b,
                      const CUtensorMap* map_c, const GemmArgs& args, uint32_t idesc, int grid,
                      cudaStream_t stream) {
  switch (bn) {
    case 64: return launch_bn<BM, 64, kSoft>(map_a, map_b, map_c, args, idesc, grid, stream);
    case 128: return launch_bn<BM, 128, kSoft>(map_a, map_b, map_c, args, idesc, grid, stream);
    case 256: return launch_bn<BM, 256, kSoft>(map_a, map_b, map_c, args, idesc, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int kSoft>
cudaError_t launch_any(int bm, int bn, const CUtensorMap* map_a, const CUtensorMap* map_b,
                       const CUtensorMap* map_c, const GemmArgs& args, uint32_t idesc, int grid,
                       cudaStream_t stream) {
  switch (bm) {
    case 64: return launch_bm<64, kSoft>(bn, map_a, map_b, map_c, args, idesc, grid, stream);
    case 128: return launch_bm<128, kSoft>(bn, map_a, map_b, map_c, args, idesc, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_hgemm_tc(int bm, int bn, const CUtensorMap& map_a, const CUtensorMap& map_b,
                            const CUtensorMap& map_c, const GemmArgs& args, uint32_t idesc,
                            int grid, cudaStream_t stream) {
  return launch_any<0>(bm, bn, &map_a, &map_b, &map_c, args, idesc, grid, stream);
}

cudaError_t launch_hgemm_tc_soft(int bm, int bn, int soft, const CUtensorMap* map_a,
                                 const CUtensorMap* map_b, const GemmArgs& args, uint32_t idesc,
                                 int grid, cudaStream_t stream) {
  switch (soft) {
    case 1: return launch_any<1>(bm, bn, nullptr, map_b, nullptr, args, idesc, grid, stream);
    case 2: return launch_any<2>(bm, bn, map_a, nullptr, nullptr, args, idesc, grid, stream);
    case 3: return launch_any<3>(bm, bn, nullptr, nullptr, nullptr, args, idesc, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gemm14
