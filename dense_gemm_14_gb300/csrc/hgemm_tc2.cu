// hgemm_tc2.cu -- bf16 / fp16 inputs, fp32 accumulate and output, on CTA
// pairs: tcgen05.mma.cta_group::2 computes a 256 x 256 output tile on two SMs.
//
// Why pairs: a one-SM 128 x 256 MMA reads 96 B/clk of operands from shared
// memory while TMA writes another 96 B/clk into it, more than one SM's shared
// memory serves; on a pair each SM holds its 128 rows of A and HALF of B
// (128 columns), the tensor cores exchange the B halves, and per SM the
// traffic drops to 64 + 64 B/clk. L2 -> SM traffic per output element drops
// by a third as well. (The pages' wgmma discussion, gpu-hpc-book ch.06
// "高级 cuda 特性 —— 从矩阵乘法(gemm)说起", "Tensor Cores" / "wgmma", is the
// prior art: asynchronous D = A*B + D with TMA-fed shared-memory operands.)
//
// Roles per CTA (192 threads, cluster of 2, persistent over pair tiles):
//   warp 0      producer: TMA loads of this CTA's A rows (128 m x 64 k) and
//               B columns (2 boxes of 64 n x 64 k) into a 6-stage ring; the
//               completion of BOTH CTAs' loads is counted on the leader's
//               full barrier (cta_group::2 TMA);
//   warp 1      both CTAs allocate the pair's TMEM (2 x 256 columns); in the
//               leader one lane issues the pair MMAs (M 256, N 256, K 16) and
//               commits to both CTAs' empty / accumulator barriers;
//   warps 2..5  epilogue in each CTA: its 128 rows of the accumulator from
//               its own TMEM to C; all eight epilogue warps release the
//               accumulator on the leader's barrier.
// Every wait is bounded; a CTA that gives up also raises its peer's abort
// flag. Both CTAs meet at a cluster barrier before TMEM is freed, so neither
// exits while the pair MMAs may still read its shared memory.
#include "kernels.h"
#include "ptx.cuh"

namespace gemm14 {
namespace {

using P = PairShape;

struct PairSmem {
  uint64_t full[P::STAGES];   // leader: both CTAs' bytes of a stage have landed
  uint64_t empty[P::STAGES];  // each CTA: the pair MMAs finished reading the stage
  uint64_t acc_full[2];       // each CTA: accumulator b holds a finished tile
  uint64_t acc_empty[2];      // leader: all 8 epilogue warps drained accumulator b
  uint64_t drain;
  uint64_t partial_stored;    // stream-K: this CTA's 4 epilogue warps stored its partial
  uint64_t flags_ready;       // stream-K: the later workers' partials are published
  uint32_t tmem_base;
  int abort_flag;
  SkTable sched;              // stream-K: this cluster's segments, decoded once
};
static_assert(sizeof(PairSmem) <= 256, "barrier block of the pair kernel");

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Grouped raster over pair tiles: groups of kGroupM row-tiles.
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

// kGeneral: stored transposes and the alpha / beta epilogue are read from
// args; without it the kernel is compiled for untransposed operands and a
// plain store of C (the common case, with nothing decided at run time).
// kSK: the stream-K schedule (streamk.cuh) with a cluster as the worker:
// both CTAs of a cluster walk the same segments; each CTA stores the partial
// sums of its 128 rows to its own workspace slot (worker w, rank r: slot
// 2w + r, flag 2w + r), and the owner of a split tile adds, per CTA, the same
// rank's partials of the later workers in worker order.
// kTf32: fp32 operands read as tf32 (tcgen05 kind::tf32, K = 8 per MMA), A
// stored M x K and B stored N x K, i.e. both K-major as TMA writes them: the
// same 128-byte rows, boxes and descriptors as 16-bit K-major operands, a
// k-block being 32 fp32 instead of 64 16-bit elements.
// kTf32 with args.k_terms == 3: the split-precision 3xTF32 product (Ootomo and
// Yokota, "Recovering single precision accuracy from Tensor Cores while
// surpassing the FP32 theoretical peak performance", 2022) from lo(A) and
// lo(B) written ahead of the call (map_a_lo, map_b_lo): the k sum runs over
// three terms of L k-blocks each, lo(A) hi(B), then hi(A) lo(B), then
// hi(A) hi(B) (small terms first), as if K were 3 K; only the producer's
// choice of tensor map and k coordinate tells them apart, so stream-K splits
// the 3 L k-blocks like any others.
template <bool kGeneral, bool kSK, bool kTf32>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(P::THREADS, 1)
    hgemm_tc2_kernel(const __grid_constant__ CUtensorMap map_a,
                     const __grid_constant__ CUtensorMap map_b,
                     const __grid_constant__ CUtensorMap map_c,
                     const __grid_constant__ CUtensorMap map_a_lo,
                     const __grid_constant__ CUtensorMap map_b_lo, const GemmArgs args,
                     const uint32_t idesc) {
  const int transa = kTf32 ? 0 : kGeneral ? args.transa : 0;
  const int transb = kTf32 ? 1 : kGeneral ? args.transb : 0;
  constexpr int BK = kTf32 ? 32 : P::BK;  // elements of a 128-byte k-block row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = align1024(smem_raw);
  uint8_t* out_stage = tiles + P::STAGES * P::STAGE_BYTES;  // epilogue staging for C
  PairSmem& sm = *reinterpret_cast<PairSmem*>(out_stage + P::OUT_BYTES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(cluster_count_x());
  const int M = args.M, N = args.N, K = args.K;
  const int tiles_m = (M + P::BM - 1) / P::BM;
  const int tiles_n = (N + P::BN - 1) / P::BN;
  const int num_tiles = tiles_m * tiles_n;
  const int kb_term = (K + BK - 1) / BK;  // k-blocks of one term of the sum
  const bool split3 = kTf32 && args.k_terms == 3;
  const int kblocks = split3 ? 3 * kb_term : kb_term;
  const WaitCtx wc{args.err, &sm.abort_flag, args.wait_limit_ns,
                   mapa_shared(smem_u32(&sm.abort_flag), rank ^ 1u)};
  uint32_t prod_it = 0;
  bool mma_issued = false;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P::STAGES; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], 8);
    }
    mbar_init(&sm.drain, 1);
    mbar_init(&sm.partial_stored, 4);
    mbar_init(&sm.flags_ready, 1);
    sm.abort_flag = 0;
    if (kSK) {
      sm.sched.fill(args.sk, cid);
      if (sm.sched.n_sk > kMaxSk) {  // cannot happen for schedules make_stream_k builds
        atomicOr(args.err, kDevErrBadConfig);
        sm.abort_flag = 1;
      }
    }
    fence_barrier_init();
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b);
    if (!kGeneral && args.vec_store) tma_prefetch_desc(&map_c);
    if (split3) {
      tma_prefetch_desc(&map_a_lo);
      tma_prefetch_desc(&map_b_lo);
    }
  }
  // Both CTAs' barriers exist before either CTA signals the other's.
  cluster_sync();
  if (warp == 1) {
    tmem_alloc_pair(&sm.tmem_base, P::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // Set-up touched only shared memory, TMEM and the parameters (and the error
  // word's commuting OR); global memory is used from here on.
  grid_dependency_wait();
  grid_launch_dependents();
  const uint32_t tmem_base = sm.tmem_base;
  // Both CTAs of a cluster decoded the same table: a pair that gave up at
  // set-up (abort) runs no segment in either CTA.
  const int n_seg = kSK ? (sm.abort_flag ? 0 : sm.sched.segments())
                        : (cid < num_tiles ? (num_tiles - 1 - cid) / ncl + 1 : 0);
  // Segment i: data-parallel tile cid + i * ncl whole, or the decoded table.
  auto segment = [&](int i, int& tile, int& kb0, int& kb1, int& kind) {
    if (kSK) {
      sm.sched.get(i, tile, kb0, kb1, kind);
    } else {
      tile = cid + i * ncl;
      kb0 = 0;
      kb1 = kblocks;
      kind = kSegFull;
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      for (int seg = 0; seg < n_seg && ok; ++seg) {
        int t, kb0, kb1, kind, tm, tn;
        segment(seg, t, kb0, kb1, kind);
        pair_tile_coords(t, tiles_m, tiles_n, tm, tn);
        for (int kb = kb0; kb < kb1; ++kb, ++prod_it) {
          const uint32_t s = prod_it % P::STAGES, ph = (prod_it / P::STAGES) & 1;
          if (!mbar_wait(&sm.empty[s], ph ^ 1, wc)) { ok = false; break; }
          // Failure-detection tests: the first stage is never loaded.
          if (args.fault == kFaultSkipFirstStage && prod_it == 0) continue;
          uint8_t* a_st = tiles + s * P::STAGE_BYTES;
          uint8_t* b_st = a_st + P::A_BYTES;
          const uint32_t full_leader = mapa_shared(smem_u32(&sm.full[s]), 0);
          if (leader) mbar_arrive_expect_tx(&sm.full[s], 2 * P::STAGE_BYTES);
          const int m0 = tm * P::BM + static_cast<int>(rank) * 128;
          const int n0 = tn * P::BN + static_cast<int>(rank) * 128;
          // 3xTF32: term t = kb / L reads lo(A) (t = 0) or lo(B) (t = 1) at
          // k-block kb - t L; the plain product reads map_a and map_b at kb.
          const CUtensorMap* ma = &map_a;
          const CUtensorMap* mb = &map_b;
          int kq = kb;
          if (split3) {
            const int t = kb / kb_term;
            kq = kb - t * kb_term;
            if (t == 0) ma = &map_a_lo;
            if (t == 1) mb = &map_b_lo;
          }
          // A: one box of 64 k x 128 m, or (stored K x M) two of 64 m x 64 k.
          if (!transa) {
            tma_load_2d_pair(a_st, ma, kq * BK, m0, full_leader);
          } else {
#pragma unroll
            for (int c = 0; c < 2; ++c)
              tma_load_2d_pair(a_st + c * (64 * P::BK * 2), &map_a, m0 + c * 64, kb * P::BK,
                               full_leader);
          }
          // B: two boxes of 64 n x 64 k, or (stored N x K) one of 64 k x 128 n.
          if (!transb) {
#pragma unroll
            for (int c = 0; c < 2; ++c)
              tma_load_2d_pair(b_st + c * (64 * P::BK * 2), &map_b, n0 + c * 64, kb * P::BK,
                               full_leader);
          } else {
            tma_load_2d_pair(b_st, mb, kq * BK, n0, full_leader);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (leader && lane == 0) {
      const OperandDesc a_op = operand_desc(transa == 0);
      const OperandDesc b_op = operand_desc(transb != 0);
      bool ok = true;
      uint32_t it = 0;
      for (int seg = 0; seg < n_seg && ok; ++seg) {
        int t, kb0, kb1, kind;
        segment(seg, t, kb0, kb1, kind);
        const int b = seg & 1;
        const uint32_t aph = (seg >> 1) & 1;
        if (!mbar_wait_cluster(&sm.acc_empty[b], aph ^ 1, wc)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * P::BN);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const uint32_t s = it % P::STAGES, ph = (it / P::STAGES) & 1;
          if (!mbar_wait(&sm.full[s], ph, wc)) { ok = false; break; }
          tc_fence_after_sync();
          const uint32_t a_addr = smem_u32(tiles + s * P::STAGE_BYTES);
          const uint32_t b_addr = a_addr + P::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < P::BK / 16; ++kk) {
            // Each CTA's 128 rows of A and 128 columns of B, in the same
            // layout in both CTAs.
            const uint64_t a_desc = smem_desc_sw128(a_addr + kk * a_op.step, a_op.lbo, 1024);
            const uint64_t b_desc = smem_desc_sw128(b_addr + kk * b_op.step, b_op.lbo, 1024);
            if (kTf32)
              tc_mma_tf32_pair(d_tmem, a_desc, b_desc, idesc, kb > kb0 || kk != 0);
            else
              tc_mma_f16_pair(d_tmem, a_desc, b_desc, idesc, kb > kb0 || kk != 0);
          }
          mma_issued = true;
          tc_commit_pair_multicast(&sm.empty[s], 0x3);
        }
        if (!ok) break;
        tc_commit_pair_multicast(&sm.acc_full[b], 0x3);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Thread = one row of the CTA's 128 (TMEM lane), 32 columns per chunk.
    // The plain variant with a 16-byte-aligned C stages each warp's 32 x 32
    // block in shared memory (128-byte swizzle: a row's 16-byte pieces spread
    // over all banks) and writes it with one TMA store; two buffers per warp
    // let the next chunk overlap the store. Otherwise each thread stores its
    // row segment directly (the alpha / beta modes read C there).
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r_loc = q * 32 + lane;  // this thread's row within the CTA's 128
    const uint32_t acc_empty_leader0 = mapa_shared(smem_u32(&sm.acc_empty[0]), 0);
    const uint32_t acc_empty_leader1 = mapa_shared(smem_u32(&sm.acc_empty[1]), 0);
    const int w = cid;
    const bool tma_c = !kGeneral && args.vec_store;
    uint8_t* out_buf = out_stage + q * 2 * P::OUT_BUF_BYTES;
    int ob = 0;
    // Stream-K slot of worker c for this CTA (128 rows x 256 fp32), laid out
    // chunk by chunk as [chunk][float4 v][row]: the 32 rows of a warp store
    // (and load) 512 contiguous bytes per instruction.
    auto slot4 = [&](int c, int chunk, int v) {
      return reinterpret_cast<float4*>(args.partials) +
             (static_cast<size_t>(2 * c + rank) * (P::BN / 32) + chunk) * 8 * 128 +
             static_cast<size_t>(v) * 128 + r_loc;
    };
    // the bounds checks of a slot access (2 args.sk.G slots of 8 x 8 x 128 float4)
    auto slot_ok = [&](int c, int chunk, int v) {
      const int64_t off = slot4(c, chunk, v) - reinterpret_cast<float4*>(args.partials);
      return dev_check(slot_span_ok(off, 2 * c + static_cast<int>(rank), (P::BN / 32) * 8 * 128,
                                    2 * static_cast<int64_t>(args.sk.G), 1),
                       args.err);
    };
    const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int seg = 0; seg < n_seg; ++seg) {
      int t, kb0, kb1, kind, tm, tn;
      segment(seg, t, kb0, kb1, kind);
      pair_tile_coords(t, tiles_m, tiles_n, tm, tn);
      const int b = seg & 1;
      const uint32_t aph = (seg >> 1) & 1;
      int got = 1;
      if (lane == 0) got = mbar_wait(&sm.acc_full[b], aph, wc) ? 1 : 0;
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      if (kSK && kind == kSegHead) {
        // Wait for the later workers holding the rest of this tile (one lane
        // of warp 2 polls their flags for this CTA's rank; the other warps
        // wait on flags_ready). A worker has at most one HEAD segment.
        if (warp == 2 && lane == 0) {
          bool all = true;
          for (int c = w + 1; c <= sm.sched.head_last && all; ++c) {
            if (!dev_check(index_ok(2 * c + rank, 2 * static_cast<int64_t>(args.sk.G)),
                           args.err))
              break;
            all = flag_wait(args.flags + 2 * c + rank, args.epoch, wc);
            if (all) flag_clear(args.flags + 2 * c + rank);
          }
          if (all) mbar_arrive(&sm.flags_ready);
        }
        if (lane == 0) got = mbar_wait(&sm.flags_ready, 0, wc) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) break;
      }
      tc_fence_after_sync();
      const int row0 = tm * P::BM + static_cast<int>(rank) * 128 + q * 32;  // the warp's rows
      const int row = row0 + lane;
      float* crow = args.C + static_cast<int64_t>(row) * args.ldc;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(b * P::BN);
#pragma unroll 1
      for (int c = 0; c < P::BN / 32; ++c) {
        // HEAD: fetch the first contributor's partial of this chunk before the
        // TMEM read so that the two latencies overlap.
        float4 pre[8];
        if (kSK && kind == kSegHead && sm.sched.head_last > w) {
#pragma unroll
          for (int v = 0; v < 8; ++v) pre[v] = slot_ok(w + 1, c, v) ? __ldcg(slot4(w + 1, c, v)) : zero4;
        }
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c * 32, r);
        tc_wait_ld();
        if (kSK && kind == kSegPartial) {
          // Stream-K: this CTA's partial sums of the tile go to its slot.
#pragma unroll
          for (int v = 0; v < 8; ++v)
            if (slot_ok(w, c, v))
              __stcg(slot4(w, c, v),
                   make_float4(__uint_as_float(r[4 * v + 0]), __uint_as_float(r[4 * v + 1]),
                               __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3])));
          continue;
        }
        if (kSK && kind == kSegHead) {
          // Add the later workers' partial sums, in worker order.
          for (int cw = w + 1; cw <= sm.sched.head_last; ++cw) {
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              const float4 p = cw == w + 1 ? pre[v]
                               : slot_ok(cw, c, v) ? __ldcg(slot4(cw, c, v)) : zero4;
              r[4 * v + 0] = __float_as_uint(__uint_as_float(r[4 * v + 0]) + p.x);
              r[4 * v + 1] = __float_as_uint(__uint_as_float(r[4 * v + 1]) + p.y);
              r[4 * v + 2] = __float_as_uint(__uint_as_float(r[4 * v + 2]) + p.z);
              r[4 * v + 3] = __float_as_uint(__uint_as_float(r[4 * v + 3]) + p.w);
            }
          }
        }
        const int col0 = tn * P::BN + c * 32;
        // A TMA store clips a row at 16-byte granularity, not per element: a
        // chunk that runs past a column count N that is not a multiple of 4
        // would write up to 3 floats past column N - 1 (into the pitch's
        // padding), so that chunk takes the guarded direct stores.
        if (tma_c && (col0 + 32 <= N || (N & 3) == 0)) {
          // The buffer's store of two chunks ago has been read out.
          uint8_t* buf = out_buf + ob * P::OUT_BUF_BYTES;
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
          const uint32_t rb = smem_u32(buf) + static_cast<uint32_t>(lane * 128);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                             rb + static_cast<uint32_t>(((v ^ lane) & 7) << 4)),
                         "r"(r[4 * v + 0]), "r"(r[4 * v + 1]), "r"(r[4 * v + 2]), "r"(r[4 * v + 3])
                         : "memory");
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&map_c, buf, col0, row0);
            bulk_commit();
          }
          ob ^= 1;
        } else if (row < M) {
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
      if (lane == 0) mbar_arrive_cluster(b ? acc_empty_leader1 : acc_empty_leader0);
      if (kSK && kind == kSegPartial) {
        // All four warps' partial stores precede the flag. A worker has at
        // most one PARTIAL segment: the barrier's first phase.
        if (lane == 0) mbar_arrive(&sm.partial_stored);
        if (warp == 2 && lane == 0 && mbar_wait(&sm.partial_stored, 0, wc) &&
            dev_check(index_ok(2 * w + rank, 2 * static_cast<int64_t>(args.sk.G)), args.err))
          flag_publish(args.flags + 2 * w + rank, args.epoch);
      }
    }
    // The TMA stores have finished (their reads of the staging buffers, and
    // their writes) before the CTA may exit.
    if (tma_c && lane == 0) bulk_wait_all();
  }

  // Teardown. On abort, the leader lets its issued MMAs and both CTAs' loads
  // (counted on its full barriers) finish, bounded, before the pair meets.
  __syncthreads();
  if (sm.abort_flag && leader) {
    if (warp == 1 && lane == 0 && mma_issued) {
      tc_commit_pair_multicast(&sm.drain, 0x1);
      mbar_wait_timed(&sm.drain, 0, 100000000ull);
    }
    if (warp == 0 && lane == 0) {
      const uint32_t first = prod_it > P::STAGES ? prod_it - P::STAGES : 0;
      for (uint32_t j = first; j < prod_it; ++j)
        if (!(args.fault == kFaultSkipFirstStage && j == 0))
          mbar_wait_timed(&sm.full[j % P::STAGES], (j / P::STAGES) & 1, 100000000ull);
    }
  }
  // Neither CTA frees TMEM or exits while the pair may still use it.
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, P::TMEM_COLS);
  }
}

template <bool kGeneral, bool kSK, bool kTf32>
cudaError_t set_pair_smem() {
  return cudaFuncSetAttribute(hgemm_tc2_kernel<kGeneral, kSK, kTf32>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, P::SMEM_BYTES);
}

template <bool kTf32>
cudaError_t set_pair_smem_all() {
  cudaError_t e;
  if ((e = set_pair_smem<false, false, kTf32>()) != cudaSuccess ||
      (e = set_pair_smem<true, false, kTf32>()) != cudaSuccess ||
      (e = set_pair_smem<false, true, kTf32>()) != cudaSuccess)
    return e;
  return set_pair_smem<true, true, kTf32>();
}

}  // namespace

int pair_max_clusters() {
  static DeviceOnce cached;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= DeviceOnce::kDevices) return 0;
  // -1: the kernels' attributes could not be set (not kept: tried again)
  const int n = cached.get(
      dev,
      [] {
        if (set_pair_smem_all<false>() != cudaSuccess || set_pair_smem_all<true>() != cudaSuccess)
          return -1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(P::THREADS, 1, 1);
        cfg.dynamicSmemBytes = P::SMEM_BYTES;
        int k = 0;
        if (cudaOccupancyMaxActiveClusters(&k, hgemm_tc2_kernel<false, false, false>, &cfg) !=
            cudaSuccess)
          k = 0;
        return k;
      },
      [](int v) { return v >= 0; });
  return n > 0 ? n : 0;
}

cudaError_t launch_hgemm_tc_pair(const CUtensorMap& map_a, const CUtensorMap& map_b,
                                 const CUtensorMap& map_c, const CUtensorMap& map_a_lo,
                                 const CUtensorMap& map_b_lo, const GemmArgs& args,
                                 uint32_t idesc, int clusters, bool tf32, cudaStream_t stream) {
  if (args.k_terms == 3 && !tf32) return cudaErrorInvalidValue;
  // tf32 operands are stored M x K and N x K, which the tf32 variants fix at
  // compile time: only the epilogue mode makes them general
  const bool general =
      (!tf32 && (args.transa || args.transb)) || args.epi != kEpiStore;
  const bool sk = args.sk.dp_tiles < args.sk.tiles;
  const dim3 grid(2 * clusters), block(P::THREADS);
  auto kernel =
      tf32 ? (sk ? (general ? hgemm_tc2_kernel<true, true, true> : hgemm_tc2_kernel<false, true, true>)
                 : (general ? hgemm_tc2_kernel<true, false, true>
                            : hgemm_tc2_kernel<false, false, true>))
           : (sk ? (general ? hgemm_tc2_kernel<true, true, false>
                            : hgemm_tc2_kernel<false, true, false>)
                 : (general ? hgemm_tc2_kernel<true, false, false>
                            : hgemm_tc2_kernel<false, false, false>));
  return launch_kernel(kernel, grid, block, P::SMEM_BYTES, stream, map_a, map_b, map_c,
                       map_a_lo, map_b_lo, args, idesc);
}

}  // namespace gemm14
