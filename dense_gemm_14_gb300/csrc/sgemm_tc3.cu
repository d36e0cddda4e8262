// sgemm_tc3.cu -- fp32 inputs on the 5th-generation tensor cores: tcgen05
// kind::tf32 on CTA pairs, fp32 accumulation in TMEM, C = A * B (and the
// extended product of the epilogue modes and stored transposes).
//
// TF32 is the pages' tensor-core format for fp32 data (gpu-hpc-book ch.06
// "高级 cuda 特性 —— 从矩阵乘法(gemm)说起", "Tensor Cores": 8 exponent bits as
// fp32, 10 fraction bits, taking fp32 inputs). The tensor cores read an fp32
// operand as tf32 by dropping its 13 low fraction bits, hi(x); one such
// product carries up to 2^-9 relative error, too much for the fp32 bound, so
// the kernel also runs the split-precision scheme known as 3xTF32 (Ootomo and
// Yokota, "Recovering single precision accuracy from Tensor Cores while
// surpassing the FP32 theoretical peak performance", 2022): lo(x) = x - hi(x)
// is exact in fp32, and
//     A B ~= hi(A) hi(B) + hi(A) lo(B) + lo(A) hi(B),
// dropping lo(A) lo(B) and the tensor cores' truncation of the lo parts (each
// below 2^-20 relative): at most 3 * 2^-20 |A||B| in all.
//
// Roles per CTA (cluster of two, persistent over 256 x 256 pair tiles; each
// CTA holds 128 rows of A and 128 columns of B; 384 threads for TF32, 320 for
// 3xTF32, which has no announcers):
//   warp 0      producer: TMA of this CTA's fp32 A and B tiles of a 32-deep
//               k-block, in the storage's own layout, into a raw ring;
//   warp 1      TMEM (2 x 256 columns per CTA); in the leader one lane issues
//               per k-block 4 slices x (1 or 3) pair MMAs M 256, N 256, K 8;
//   warps 2..5  epilogue: each CTA's 128 accumulator rows from TMEM to C;
//   warps 6..9  converters: write what the MMAs need beyond the raw tiles into
//               an operand ring. 3xTF32: 2 stages of the lo tiles and a
//               K-major copy of an operand stored MN-major. TF32: 4 stages of
//               K-major copies of both operands wherever one of them needs a
//               copy, so that no raw stage waits for the MMAs; 3 raw stages.
//               They release each stage to their CTA's announcer;
//   warps 10,11 announcers (TF32), each taking every other k-block: forward
//               each completed stage to the leader's barrier (one cluster-scope
//               release arrival per CTA and stage, about 0.6 us, kept off the
//               converters' path); the leader's MMAs read the stage once both
//               CTAs' arrived. For 3xTF32, whose MMAs outlast the arrival,
//               the converter warps arrive on the leader's barrier themselves.
// Every MMA operand is K-major with the 128-byte swizzle, the one layout every
// tcgen05 kind takes. A raw tile that TMA already wrote K-major (A stored
// M x K, B stored N x K) is an MMA operand as it stands (3xTF32, and TF32 with
// both operands stored so); its raw stage is then freed by the MMAs' commit
// as well as by the converters.
// Every wait is bounded, a CTA that gives up raises its peer's abort flag,
// and both CTAs meet at a cluster barrier before TMEM is freed.
#include "kernels.h"
#include "ptx.cuh"

namespace gemm14 {
namespace {

using T = Tf32Shape;

// Shared-memory plan of one storage variant (kTA: A stored K x M; kTB: B
// stored N x K). The operand stage holds, in this order, a K-major copy of A
// (if A is stored K x M), lo(A), a K-major copy of B (if B is stored K x N)
// and lo(B); the raw ring takes what is left of the ring budget.
template <bool kTA, bool kTB>
struct Tf32Plan {
  static constexpr bool A_RAW = !kTA;  // the raw A tile is K-major: the MMAs read it
  static constexpr bool B_RAW = kTB;
  static constexpr int A_HI = 0;
  static constexpr int A_LO = (A_RAW ? 0 : 1) * T::TILE;
  static constexpr int B_HI = A_LO + T::TILE;
  static constexpr int B_LO = B_HI + (B_RAW ? 0 : 1) * T::TILE;
  static constexpr int OP_STAGE = B_LO + T::TILE;
  // TF32 (one term) needs only K-major copies. Where one operand needs a
  // copy, both are copied (A at 0, B at TILE): the converters then free every
  // raw stage without waiting for the MMAs, and four operand stages cover the
  // MMAs' latency. The TF32 rings: 3 raw stages and 4 operand stages (both
  // operands as stored K-major: no copies, the 3xTF32 raw ring).
  static constexpr bool COPY_TF32 = !(A_RAW && B_RAW);
  static constexpr int OP1_STAGE = COPY_TF32 ? 2 * T::TILE : 0;
  static constexpr int RAW_STAGES_TF32 = COPY_TF32 ? 3 : 0;  // 0: RAW_STAGES
  static_assert(RAW_STAGES_TF32 * T::RAW_STAGE + T::OP_STAGES_TF32 * OP1_STAGE <= T::RING_BYTES,
                "TF32 rings");
  static constexpr int RAW_STAGES_FIT = (T::RING_BYTES - T::OP_STAGES * OP_STAGE) / T::RAW_STAGE;
  static constexpr int RAW_STAGES =
      RAW_STAGES_FIT < T::MAX_RAW_STAGES ? RAW_STAGES_FIT : T::MAX_RAW_STAGES;
  static_assert(RAW_STAGES >= 3, "raw ring depth");
  static_assert(RAW_STAGES * T::RAW_STAGE + T::OP_STAGES * OP_STAGE <= T::RING_BYTES, "rings");
};

// The ring geometry of one mode (kThree: 3xTF32), fixed at compile time in
// the roles' loops; the kernel picks the mode once per role.
template <class L, bool kThree>
struct Tf32Mode {
  static constexpr bool THREE = kThree;
  // the MMAs read hi(A) / hi(B) from the raw stage where TMA wrote it K-major
  static constexpr bool A_RAW = L::A_RAW && (kThree || !L::COPY_TF32);
  static constexpr bool B_RAW = L::B_RAW && (kThree || !L::COPY_TF32);
  static constexpr bool MMA_READS_RAW = A_RAW || B_RAW;
  static constexpr uint32_t RS =
      (kThree || !L::COPY_TF32) ? L::RAW_STAGES : L::RAW_STAGES_TF32;
  static constexpr uint32_t OP_LOG = kThree ? 1u : 2u;  // operand stages: 2 or 4
  static constexpr uint32_t OP_MASK = (1u << OP_LOG) - 1u;
  static constexpr uint32_t OP_BYTES = kThree ? L::OP_STAGE : L::OP1_STAGE;
  static constexpr uint32_t B_HI = kThree ? L::B_HI : T::TILE;
};

struct Tf32Smem {
  uint64_t raw_full[T::MAX_RAW_STAGES];   // each CTA: its TMA bytes of a raw stage landed
  uint64_t raw_empty[T::MAX_RAW_STAGES];  // each CTA: converters (and MMAs) are done with it
  // operand stages: T::OP_STAGES for 3xTF32, T::OP_STAGES_TF32 for TF32
  uint64_t op_full[T::OP_STAGES_TF32];    // leader: both CTAs forwarded an operand stage
  uint64_t conv_done[T::OP_STAGES_TF32];  // each CTA: its 4 converter warps wrote an operand stage
  uint64_t op_empty[T::OP_STAGES_TF32];   // each CTA: the pair MMAs finished reading it
  uint64_t acc_full[2];                   // each CTA: accumulator b holds a finished tile
  uint64_t acc_empty[2];                  // leader: all 8 epilogue warps drained accumulator b
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Tf32Smem) <= 512, "barrier block");

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void pair_tile_coords(int t, int tiles_m, int tiles_n, int& tm,
                                                 int& tn) {
  constexpr int kGroupM = 8;
  const int per_group = kGroupM * tiles_n;
  const int g = t / per_group;
  const int first_m = g * kGroupM;
  const int gm = min(tiles_m - first_m, kGroupM);
  const int r = t - g * per_group;
  tm = first_m + r % gm;
  tn = r / gm;
}

__device__ __forceinline__ void sts128(uint32_t addr, float4 v) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ float lds32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// lo(x) = x - hi(x), hi(x) = x with its 13 low fraction bits cleared (exact).
__device__ __forceinline__ float lo_tf32(float x) {
  return x - __uint_as_float(__float_as_uint(x) & 0xffffe000u);
}

// Byte offset of the 16-byte chunk c (k = 4c .. 4c+3) of row r in a K-major
// operand tile: 128-byte rows, chunk index XOR-ed with (r % 8) -- the layout
// TMA's 128-byte swizzle writes and the MMA descriptors below describe.
__device__ __forceinline__ uint32_t kmajor_chunk(int r, int c) {
  return static_cast<uint32_t>(r * 128 + (((c ^ r) & 7) << 4));
}

// Row r of a raw K-major tile (as TMA's 128-byte swizzle wrote it): the 32
// values of the row, chunk c in v[c].
__device__ __forceinline__ void load_kmajor(uint32_t raw, int r, float4 (&v)[8]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) v[c] = lds128(raw + kmajor_chunk(r, c));
}

// Column r of a raw MN-major tile (32 k rows of 128 fp32, unswizzled, as TMA
// wrote it): a warp reads 32 consecutive floats of one k row per load.
__device__ __forceinline__ void load_mnmajor(uint32_t raw, int r, float4 (&v)[8]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    v[c].x = lds32(raw + static_cast<uint32_t>(((4 * c + 0) * 128 + r) * 4));
    v[c].y = lds32(raw + static_cast<uint32_t>(((4 * c + 1) * 128 + r) * 4));
    v[c].z = lds32(raw + static_cast<uint32_t>(((4 * c + 2) * 128 + r) * 4));
    v[c].w = lds32(raw + static_cast<uint32_t>(((4 * c + 3) * 128 + r) * 4));
  }
}

// Row r of a K-major operand tile: the values as they are (the tensor cores
// drop their low bits), or their lo parts.
__device__ __forceinline__ void store_row(uint32_t tile, int r, const float4 (&v)[8]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) sts128(tile + kmajor_chunk(r, c), v[c]);
}
__device__ __forceinline__ void store_lo_row(uint32_t tile, int r, const float4 (&v)[8]) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    sts128(tile + kmajor_chunk(r, c),
           make_float4(lo_tf32(v[c].x), lo_tf32(v[c].y), lo_tf32(v[c].z), lo_tf32(v[c].w)));
}

// kTA / kTB: A stored K x M / B stored N x K. kGeneral: the alpha / beta
// epilogue read from args (else a plain store).
template <bool kTA, bool kTB, bool kGeneral>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(T::THREADS, 1)
    sgemm_tf32_pair_kernel(const __grid_constant__ CUtensorMap map_a,
                           const __grid_constant__ CUtensorMap map_b, const GemmArgs args,
                           const uint32_t idesc, const int terms) {
  using L = Tf32Plan<kTA, kTB>;
  using Three = Tf32Mode<L, true>;
  using One = Tf32Mode<L, false>;
  const bool three = terms == 3;
  // ring geometry of the mode, for set-up and teardown (the roles' loops
  // take it from Tf32Mode at compile time)
  const bool mma_reads_raw = three ? Three::MMA_READS_RAW : One::MMA_READS_RAW;
  const uint32_t rs = three ? Three::RS : One::RS;
  const uint32_t op_stages = three ? T::OP_STAGES : T::OP_STAGES_TF32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t* raw_ring = base;
  Tf32Smem& sm = *reinterpret_cast<Tf32Smem*>(base + T::RING_BYTES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(cluster_count_x());
  const int M = args.M, N = args.N, K = args.K;
  const int tiles_m = (M + T::BM - 1) / T::BM;
  const int tiles_n = (N + T::BN - 1) / T::BN;
  const int num_tiles = tiles_m * tiles_n;
  const int kblocks = (K + T::BK - 1) / T::BK;
  const WaitCtx wc{args.err, &sm.abort_flag, args.wait_limit_ns,
                   mapa_shared(smem_u32(&sm.abort_flag), rank ^ 1u)};
  uint32_t prod_it = 0;
  bool mma_issued = false;

  if (threadIdx.x == 0) {
    for (int s = 0; s < static_cast<int>(rs); ++s) {
      mbar_init(&sm.raw_full[s], 1);
      mbar_init(&sm.raw_empty[s], mma_reads_raw ? 5 : 4);
    }
    for (int s = 0; s < static_cast<int>(op_stages); ++s) {
      // 3xTF32: the 8 converter warps of both CTAs arrive themselves; TF32:
      // the two CTAs' announcers
      mbar_init(&sm.op_full[s], three ? 8 : 2);
      mbar_init(&sm.conv_done[s], 128);
      mbar_init(&sm.op_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], 8);
    }
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b);
  }
  // Both CTAs' barriers exist before either CTA signals the other's.
  cluster_sync();
  if (warp == 1) {
    tmem_alloc_pair(&sm.tmem_base, T::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // Set-up touched only shared memory, TMEM and the parameters; global memory
  // is used from here on.
  grid_dependency_wait();
  grid_launch_dependents();
  const uint32_t tmem_base = sm.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    auto run = [&](auto mode) {
      using Md = decltype(mode);
      if (lane == 0) {
        bool ok = true;
        uint32_t next_s = 0, next_ph = 0;  // raw stage and phase of prod_it
        for (int t = cid; t < num_tiles && ok; t += ncl) {
          int tm, tn;
          pair_tile_coords(t, tiles_m, tiles_n, tm, tn);
          const int m0 = tm * T::BM + static_cast<int>(rank) * 128;
          const int n0 = tn * T::BN + static_cast<int>(rank) * 128;
          for (int kb = 0; kb < kblocks; ++kb, ++prod_it) {
            const uint32_t s = next_s, ph = next_ph;
            if (!mbar_wait(&sm.raw_empty[s], ph ^ 1, wc)) { ok = false; break; }
            if (++next_s == Md::RS) { next_s = 0; next_ph ^= 1; }
            // Failure-detection tests: the first stage is never loaded.
            if (args.fault == kFaultSkipFirstStage && prod_it == 0) continue;
            uint8_t* ra = raw_ring + s * T::RAW_STAGE;
            uint8_t* rb = ra + T::TILE;
            mbar_arrive_expect_tx(&sm.raw_full[s], T::RAW_STAGE);
            if (kTA) tma_load_2d(ra, &map_a, m0, kb * T::BK, &sm.raw_full[s]);
            else tma_load_2d(ra, &map_a, kb * T::BK, m0, &sm.raw_full[s]);
            if (kTB) tma_load_2d(rb, &map_b, kb * T::BK, n0, &sm.raw_full[s]);
            else tma_load_2d(rb, &map_b, n0, kb * T::BK, &sm.raw_full[s]);
          }
        }
      }
    };
    if (three) run(Three{});
    else run(One{});
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    auto run = [&](auto mode) {
      using Md = decltype(mode);
      uint8_t* const op_ring_md = base + Md::RS * T::RAW_STAGE;
      if (leader && lane == 0) {
        bool ok = true;
        uint32_t it = 0, s = 0;  // s: raw stage of it
        int local = 0;
        for (int t = cid; t < num_tiles && ok; t += ncl, ++local) {
          const int b = local & 1;
          const uint32_t aph = (local >> 1) & 1;
          if (!mbar_wait_cluster(&sm.acc_empty[b], aph ^ 1, wc)) break;
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * T::BN);
          for (int kb = 0; kb < kblocks; ++kb, ++it, s = s + 1 == Md::RS ? 0 : s + 1) {
            const uint32_t o = it & Md::OP_MASK, oph = (it >> Md::OP_LOG) & 1;
            // Both CTAs' converters have seen raw stage s full and written
            // operand stage o.
            if (!mbar_wait_cluster(&sm.op_full[o], oph, wc)) { ok = false; break; }
            tc_fence_after_sync();
            const uint32_t raw = smem_u32(raw_ring + s * T::RAW_STAGE);
            const uint32_t op = smem_u32(op_ring_md + o * Md::OP_BYTES);
            const uint32_t a_hi = Md::A_RAW ? raw : op + L::A_HI;
            const uint32_t b_hi = Md::B_RAW ? raw + T::TILE : op + Md::B_HI;
#pragma unroll
            for (int kk = 0; kk < T::BK / 8; ++kk) {
              // K-major, 128-byte rows, 8-row groups 1024 B apart; a K = 8 slice
              // of tf32 is 32 bytes further along the rows.
              const uint32_t off = static_cast<uint32_t>(kk * 32);
              const uint64_t ah = smem_desc_sw128(a_hi + off, 16, 1024);
              const uint64_t bh = smem_desc_sw128(b_hi + off, 16, 1024);
              tc_mma_tf32_pair(d_tmem, ah, bh, idesc, (kb | kk) != 0);
              if (Md::THREE) {
                tc_mma_tf32_pair(d_tmem, ah, smem_desc_sw128(op + L::B_LO + off, 16, 1024), idesc,
                                 true);
                tc_mma_tf32_pair(d_tmem, smem_desc_sw128(op + L::A_LO + off, 16, 1024), bh, idesc,
                                 true);
              }
            }
            mma_issued = true;
            tc_commit_pair_multicast(&sm.op_empty[o], 0x3);
            if (Md::MMA_READS_RAW) tc_commit_pair_multicast(&sm.raw_empty[s], 0x3);
          }
          if (!ok) break;
          tc_commit_pair_multicast(&sm.acc_full[b], 0x3);
        }
      }
    };
    if (three) run(Three{});
    else run(One{});
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const uint32_t acc_empty_leader0 = mapa_shared(smem_u32(&sm.acc_empty[0]), 0);
    const uint32_t acc_empty_leader1 = mapa_shared(smem_u32(&sm.acc_empty[1]), 0);
    int local = 0;
    for (int t = cid; t < num_tiles; t += ncl, ++local) {
      int tm, tn;
      pair_tile_coords(t, tiles_m, tiles_n, tm, tn);
      const int b = local & 1;
      const uint32_t aph = (local >> 1) & 1;
      int got = 1;
      if (lane == 0) got = mbar_wait(&sm.acc_full[b], aph, wc) ? 1 : 0;
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      tc_fence_after_sync();
      const int row = tm * T::BM + static_cast<int>(rank) * 128 + q * 32 + lane;
      float* crow = args.C + static_cast<int64_t>(row) * args.ldc;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(b * T::BN);
#pragma unroll 1
      for (int c = 0; c < T::BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c * 32, r);
        tc_wait_ld();
        const int col0 = tn * T::BN + c * 32;
        if (row < M) {
          if (args.vec_store && col0 + 32 <= N) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              epi_store4<kGeneral>(
                  args, crow + col0 + 4 * v,
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
      if (lane == 0) mbar_arrive_cluster(b ? acc_empty_leader1 : acc_empty_leader0);
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------ converters
    auto run = [&](auto mode) {
      using Md = decltype(mode);
      uint8_t* const op_ring_md = base + Md::RS * T::RAW_STAGE;
      // Thread r handles row r of A and row r of B^T. A raw stage is released
      // only after the values loaded from it are stored: the stores consume
      // the loaded registers, so the loads have read the stage before TMA may
      // refill it (released straight after the loads, it was refilled under
      // them).
      const int r = threadIdx.x - 6 * 32;
      constexpr bool need_a = !Md::A_RAW || Md::THREE;  // a K-major copy of A, or lo(A)
      constexpr bool need_b = !Md::B_RAW || Md::THREE;
      uint32_t it = 0, s = 0, ph = 0;  // s, ph: raw stage and phase of it
      bool ok = true;
      for (int t = cid; t < num_tiles && ok; t += ncl) {
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const uint32_t o = it & Md::OP_MASK, oph = (it >> Md::OP_LOG) & 1;
          int got = 1;
          if (lane == 0) got = mbar_wait(&sm.raw_full[s], ph, wc) ? 1 : 0;
          got = __shfl_sync(0xffffffffu, got, 0);
          if (!got) { ok = false; break; }
          const uint32_t ra = smem_u32(raw_ring + s * T::RAW_STAGE);
          const uint32_t rb = ra + T::TILE;
          float4 va[8], vb[8];
          if (need_a) {
            if (kTA) load_mnmajor(ra, r, va);
            else load_kmajor(ra, r, va);
          }
          if (need_b) {
            if (kTB) load_kmajor(rb, r, vb);
            else load_mnmajor(rb, r, vb);
          }
          if (lane == 0) got = mbar_wait(&sm.op_empty[o], oph ^ 1, wc) ? 1 : 0;
          got = __shfl_sync(0xffffffffu, got, 0);
          if (!got) { ok = false; break; }
          const uint32_t op = smem_u32(op_ring_md + o * Md::OP_BYTES);
          if (!Md::A_RAW) store_row(op + L::A_HI, r, va);
          if (Md::THREE) store_lo_row(op + L::A_LO, r, va);
          if (!Md::B_RAW) store_row(op + Md::B_HI, r, vb);
          if (Md::THREE) store_lo_row(op + L::B_LO, r, vb);
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.raw_empty[s]);
          // This thread's operand writes -> visible to the MMAs (async proxy).
          fence_proxy_async_smem();
          if (Md::THREE) {
            // the warp's writes are ordered before lane 0's release arrival on
            // the leader's barrier (the 3xTF32 MMAs take longer than the
            // arrival, which stays on this path)
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&sm.op_full[o]), 0));
          } else {
            // released to this CTA's announcer (CTA scope), which forwards the
            // stage to the leader at cluster scope off this warp's path
            mbar_arrive(&sm.conv_done[o]);
          }
          if (++s == Md::RS) { s = 0; ph ^= 1; }
        }
      }
    };
    if (three) run(Three{});
    else run(One{});
  } else {
    // ------------------------------------------------------------ announcer
    // Acquires each operand stage from this CTA's converters and releases it
    // to the leader's op_full barrier at cluster scope: the converters' writes
    // reach the leader's MMAs through this chain of release and acquire.
    // Warp 10 + a handles the k-blocks it with it % 2 == a (TF32; for 3xTF32
    // the converters arrive themselves).
    const uint32_t a = static_cast<uint32_t>(warp - 10);
    if (lane == 0 && !three) {
      const uint32_t uses = static_cast<uint32_t>((num_tiles - cid + ncl - 1) / ncl) *
                            static_cast<uint32_t>(kblocks);  // this CTA's k-blocks
      for (uint32_t it = a; it < uses; it += 2) {
        const uint32_t o = it & One::OP_MASK;
        if (!mbar_wait(&sm.conv_done[o], (it >> One::OP_LOG) & 1, wc)) break;
        mbar_arrive_cluster(mapa_shared(smem_u32(&sm.op_full[o]), 0));
      }
    }
  }

  // Teardown. On abort, the leader lets its issued MMAs finish and every CTA
  // lets its own raw loads land (bounded) before the pair meets.
  __syncthreads();
  if (sm.abort_flag) {
    if (leader && warp == 1 && lane == 0 && mma_issued) {
      tc_commit_pair_multicast(&sm.drain, 0x1);
      mbar_wait_timed(&sm.drain, 0, 100000000ull);
    }
    if (warp == 0 && lane == 0) {
      const uint32_t first = prod_it > rs ? prod_it - rs : 0;
      for (uint32_t j = first; j < prod_it; ++j)
        if (!(args.fault == kFaultSkipFirstStage && j == 0))
          mbar_wait_timed(&sm.raw_full[j % rs], (j / rs) & 1, 100000000ull);
    }
  }
  // Neither CTA frees TMEM or exits while the pair may still use it.
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, T::TMEM_COLS);
  }
}

template <bool kTA, bool kTB, bool kGeneral>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(sgemm_tf32_pair_kernel<kTA, kTB, kGeneral>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
}

template <bool kTA, bool kTB, bool kGeneral>
cudaError_t launch_one(const CUtensorMap& map_a, const CUtensorMap& map_b, const GemmArgs& args,
                       uint32_t idesc, int terms, int clusters, cudaStream_t stream) {
  // 3xTF32 runs without the announcer warps (its converters arrive on the
  // leader's barrier themselves)
  const int threads = T::threads(terms == 3);
  return launch_kernel(sgemm_tf32_pair_kernel<kTA, kTB, kGeneral>, dim3(2 * clusters),
                       dim3(threads), T::SMEM_BYTES, stream, map_a, map_b, args, idesc, terms);
}

template <bool kTA, bool kTB>
cudaError_t launch_epi(const CUtensorMap& map_a, const CUtensorMap& map_b, const GemmArgs& args,
                       uint32_t idesc, int terms, int clusters, cudaStream_t stream) {
  if (args.epi != kEpiStore)
    return launch_one<kTA, kTB, true>(map_a, map_b, args, idesc, terms, clusters, stream);
  return launch_one<kTA, kTB, false>(map_a, map_b, args, idesc, terms, clusters, stream);
}

}  // namespace

int tf32_pair_max_clusters() {
  static DeviceOnce cached;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= DeviceOnce::kDevices) return 0;
  // -1: the kernels' attributes could not be set (not kept: tried again)
  const int n = cached.get(
      dev,
      [] {
        if (set_smem<false, false, false>() || set_smem<false, false, true>() ||
            set_smem<true, false, false>() || set_smem<true, false, true>() ||
            set_smem<false, true, false>() || set_smem<false, true, true>() ||
            set_smem<true, true, false>() || set_smem<true, true, true>())
          return -1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(T::THREADS, 1, 1);
        cfg.dynamicSmemBytes = T::SMEM_BYTES;
        int k = 0;
        if (cudaOccupancyMaxActiveClusters(&k, sgemm_tf32_pair_kernel<false, false, false>,
                                           &cfg) != cudaSuccess)
          k = 0;
        return k;
      },
      [](int v) { return v >= 0; });
  return n > 0 ? n : 0;
}

cudaError_t launch_sgemm_tf32_pair(const CUtensorMap& map_a, const CUtensorMap& map_b,
                                   const GemmArgs& args, int terms, int clusters,
                                   cudaStream_t stream) {
  const uint32_t idesc = idesc_tf32_f32acc(T::BM, T::BN);
  if (args.transa) {
    if (args.transb) return launch_epi<true, true>(map_a, map_b, args, idesc, terms, clusters, stream);
    return launch_epi<true, false>(map_a, map_b, args, idesc, terms, clusters, stream);
  }
  if (args.transb) return launch_epi<false, true>(map_a, map_b, args, idesc, terms, clusters, stream);
  return launch_epi<false, false>(map_a, map_b, args, idesc, terms, clusters, stream);
}

}  // namespace gemm14
