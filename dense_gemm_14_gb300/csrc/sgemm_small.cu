// sgemm_small.cu -- fp32 products with too few 128 x 256 output tiles to
// occupy the GPU (C = alpha op(A) op(B) + beta C, fp32 FFMA).
//
// The large fp32 kernel gives each SM a 128 x 256 tile, so a 256^3 product
// runs on 2 SMs, each working through 16.8 MFLOP alone. Here the tiles are
// 64 x 64 and, when that still leaves SMs idle, the k range of each tile is
// split over the CTAs of a thread-block cluster (2 to 8 CTAs): every CTA sums
// its own slice of k into registers, writes the 64 x 64 partial tile to its
// shared memory, and after a cluster barrier each CTA adds up one band of
// rows of all the cluster's partial tiles through distributed shared memory
// (ld.shared::cluster), rank 0's first, and stores that band of C. The sum
// is thus formed in a fixed order (deterministic run to run) without any
// workspace, atomics or second launch.
//
// Within a CTA: 128 threads, each with a 4 x 8 block of the tile summed with
// packed fp32x2 FMAs (fma.rn.f32x2: two IEEE fp32 FMAs per instruction, each
// accumulator summed over k in order); a 3-stage cp.async ring of 32-deep
// k-blocks (A tile 64 x 32, B tile 32 x 64, zero filled outside the
// matrices). This is the shared-memory tiling and
// register blocking of gpu-hpc-book ch.06 "高级 cuda 特性 —— 从矩阵乘法(gemm)
// 说起" ("矩阵乘法中的分块与数据复用", matmul_l1 and matmul_l1_reg) and the
// double buffering of "Kernel 优化指南" ("Level 3: Double Buffering"), sized for
// latency rather than throughput; the split of k over cooperating blocks
// follows the same chapter's "调度优化" point that a grid needs enough blocks
// to keep every SM busy.
#include "kernels.h"
#include "ptx.cuh"

namespace gemm14 {
namespace {

using Q = SmallShape;
constexpr int A_LD = Q::BK + 4;  // A stage: [BM][BK + 4] (rows of 144 bytes)
constexpr int B_LD = Q::BN + 4;  // B stage: [BK][BN + 4] (rows of 272 bytes)
constexpr int P_LD = Q::BN + 4;  // partial tile: [BM][BN + 4]
constexpr int A_STAGE = Q::BM * A_LD;  // floats
constexpr int B_STAGE = Q::BK * B_LD;
static_assert(Q::STAGES * (A_STAGE + B_STAGE) * 4 <= Q::SMEM_BYTES, "stage ring");
static_assert(Q::BM * P_LD * 4 <= Q::SMEM_BYTES, "partial tile");

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
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

// Loads k-block kb of tile (m0, n0) into stage s: A[m][k] (m < 64, k < 32)
// and B[k][n] (k < 32, n < 64). Elements outside op(A) / op(B) or past the
// CTA's k range end read as zero. kVec: A stored M x K and B stored K x N,
// both 16-byte aligned with pitches of multiples of 4 floats: 16-byte copies
// along k (A) and n (B), partly filled at the matrix edges; otherwise 4-byte
// copies, placed so that every storage lands in the same layout (and so
// sums in the same order).
template <bool kVec>
__device__ __forceinline__ void load_stage(float* st, const GemmArgs& a, int m0, int n0, int k0,
                                           int k_end) {
  const float* A = static_cast<const float*>(a.A);
  const float* B = static_cast<const float*>(a.B);
  float* As = st;
  float* Bs = st + A_STAGE;
  const int t = threadIdx.x;
  if (kVec) {
    // A: 64 rows x 8 chunks of 4 k; B: 32 rows x 16 chunks of 4 n
#pragma unroll
    for (int i = 0; i < 512 / Q::THREADS; ++i) {
      const int c = t + i * Q::THREADS;
      const int m = c >> 3, kc = (c & 7) * 4;
      const int gm = m0 + m, gk = k0 + kc;
      const int left = gm < a.M ? min(k_end - gk, 4) : 0;
      const uint32_t bytes = left > 0 ? 4u * left : 0u;
      cp_async_16(smem_u32(As + m * A_LD + kc), bytes ? A + static_cast<int64_t>(gm) * a.lda + gk : A,
                  bytes);
    }
#pragma unroll
    for (int i = 0; i < 512 / Q::THREADS; ++i) {
      const int c = t + i * Q::THREADS;
      const int k = c >> 4, nc = (c & 15) * 4;
      const int gk = k0 + k, gn = n0 + nc;
      const int left = gk < k_end ? min(a.N - gn, 4) : 0;
      const uint32_t bytes = left > 0 ? 4u * left : 0u;
      cp_async_16(smem_u32(Bs + k * B_LD + nc), bytes ? B + static_cast<int64_t>(gk) * a.ldb + gn : B,
                  bytes);
    }
  } else {
    // one element per copy; consecutive threads read consecutive addresses
    // of the stored matrix
    constexpr int R32 = Q::THREADS / 32, R64 = Q::THREADS / 64;  // rows per pass
#pragma unroll 4
    for (int i = 0; i < 2048 / Q::THREADS; ++i) {
      int m, k;
      if (!a.transa) {  // A[m * lda + k]: k fastest
        k = t & 31;
        m = (t >> 5) + R32 * i;
      } else {          // A[k * lda + m]: m fastest
        m = t & 63;
        k = (t >> 6) + R64 * i;
      }
      const int gm = m0 + m, gk = k0 + k;
      const bool in = gm < a.M && gk < k_end;
      const int64_t off = a.transa ? static_cast<int64_t>(gk) * a.lda + gm
                                   : static_cast<int64_t>(gm) * a.lda + gk;
      cp_async_4(smem_u32(As + m * A_LD + k), in ? A + off : A, in ? 4u : 0u);
    }
#pragma unroll 4
    for (int i = 0; i < 2048 / Q::THREADS; ++i) {
      int k, n;
      if (!a.transb) {  // B[k * ldb + n]: n fastest
        n = t & 63;
        k = (t >> 6) + R64 * i;
      } else {          // B[n * ldb + k]: k fastest
        k = t & 31;
        n = (t >> 5) + R32 * i;
      }
      const int gk = k0 + k, gn = n0 + n;
      const bool in = gn < a.N && gk < k_end;
      const int64_t off = a.transb ? static_cast<int64_t>(gn) * a.ldb + gk
                                   : static_cast<int64_t>(gk) * a.ldb + gn;
      cp_async_4(smem_u32(Bs + k * B_LD + n), in ? B + off : B, in ? 4u : 0u);
    }
  }
}

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

// Thread t of the CTA: warp w = t / 32 holds rows 16 w .. 16 w + 15; lane l
// holds rows 16 w + (l / 8) + 4 i (i < 4) and columns 4 (l % 8) + q and
// 32 + 4 (l % 8) + q (q < 4). acc2[i][p]: row i, columns pair p (p < 2: the
// first four columns, p >= 2: the second four).
__device__ __forceinline__ int small_row(int t, int i) {
  return 16 * (t >> 5) + ((t & 31) >> 3) + 4 * i;
}
__device__ __forceinline__ int small_col(int t, int h) { return 32 * h + 4 * (t & 7); }

// The thread's 4 x 8 block over one k-block, k in order: per 4 k, four
// 16-byte loads of A (4 k of each row) and two of B per k.
__device__ __forceinline__ void fma_block(const float* st, int t, uint64_t (&acc2)[4][4]) {
  const uint32_t a0 = smem_u32(st + small_row(t, 0) * A_LD);
  const uint32_t b0 = smem_u32(st + A_STAGE + small_col(t, 0));
#pragma unroll
  for (int k4 = 0; k4 < Q::BK; k4 += 4) {
    float4 a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = lds128(a0 + static_cast<uint32_t>((4 * i * A_LD + k4) * 4));
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint32_t bk = b0 + static_cast<uint32_t>((k4 + kk) * B_LD * 4);
      const float4 v0 = lds128(bk), v1 = lds128(bk + 128);
      const uint64_t bp[4] = {pack2(v0.x, v0.y), pack2(v0.z, v0.w), pack2(v1.x, v1.y),
                              pack2(v1.z, v1.w)};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
        const uint64_t a2 = pack2(av, av);
#pragma unroll
        for (int p = 0; p < 4; ++p) fma2(acc2[i][p], a2, bp[p]);
      }
    }
  }
}

constexpr int kMaxClusterSplit = 8;  // the plan splits a tile over at most 8 CTAs

__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t cluster_addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(cluster_addr)
               : "memory");
  return v;
}

// Writes s (4 consecutive columns from (row, col)) to C through the
// epilogue's update, vectorised when C allows and the 4 columns lie inside N.
__device__ __forceinline__ void store4(const GemmArgs& a, int row, int col, float4 s) {
  if (row >= a.M || col >= a.N) return;
  float* p = a.C + static_cast<int64_t>(row) * a.ldc + col;
  if (a.vec_store && col + 4 <= a.N) {
    epi_store4<true>(a, p, s);
  } else {
    const float v[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (col + j < a.N) epi_store1<true>(a, p + j, v[j]);
  }
}

// Grid: split x tiles CTAs, clusters of `split` consecutive CTAs (one tile
// each). Rank r of a cluster sums k-blocks [r * kb_per, (r + 1) * kb_per).
template <bool kVec>
__global__ void __launch_bounds__(Q::THREADS)
    sgemm_small_kernel(const GemmArgs args, const int split, const int kb_per) {
  extern __shared__ __align__(16) float smem[];
  const int t = threadIdx.x;
  const int tile = blockIdx.x / split;
  const int rank = split > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int tiles_m = (args.M + Q::BM - 1) / Q::BM;
  const int m0 = (tile % tiles_m) * Q::BM;
  const int n0 = (tile / tiles_m) * Q::BN;
  const int kb_begin = rank * kb_per;
  const int k_end = min(args.K, (kb_begin + kb_per) * Q::BK);
  const int nkb = max(0, min(kb_per, (args.K + Q::BK - 1) / Q::BK - kb_begin));
  uint64_t acc2[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc2[i][j] = 0ull;

  // Global memory is touched only after the previous grid on the stream is
  // complete (programmatic dependent launch).
  grid_dependency_wait();
  grid_launch_dependents();
#pragma unroll
  for (int s = 0; s < Q::STAGES - 1; ++s) {
    if (s < nkb)
      load_stage<kVec>(smem + s * (A_STAGE + B_STAGE), args, m0, n0, (kb_begin + s) * Q::BK,
                       k_end);
    cp_async_commit();
  }
#pragma unroll 1
  for (int i = 0; i < nkb; ++i) {
    cp_async_wait<Q::STAGES - 2>();
    __syncthreads();
    // the stage read in iteration i - 1 is free again: fill it with k-block i + STAGES - 1
    const int nx = i + Q::STAGES - 1;
    if (nx < nkb)
      load_stage<kVec>(smem + (nx % Q::STAGES) * (A_STAGE + B_STAGE), args, m0, n0,
                       (kb_begin + nx) * Q::BK, k_end);
    cp_async_commit();
    fma_block(smem + (i % Q::STAGES) * (A_STAGE + B_STAGE), t, acc2);
  }
  cp_async_wait<0>();

  // the thread's row i, columns 32 h + 4 (t % 8) .. + 3
  auto quad = [&](int i, int h) {
    const float2 lo = unpack2(acc2[i][2 * h]), hi = unpack2(acc2[i][2 * h + 1]);
    return make_float4(lo.x, lo.y, hi.x, hi.y);
  };
  if (split == 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h) store4(args, m0 + small_row(t, i), n0 + small_col(t, h), quad(i, h));
    return;
  }
  // Partial tile into this CTA's shared memory (the ring is no longer read).
  __syncthreads();
  float* P = smem;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int h = 0; h < 2; ++h)
      *reinterpret_cast<float4*>(P + small_row(t, i) * P_LD + small_col(t, h)) = quad(i, h);
  cluster_sync();  // every partial tile of the cluster is written and visible
  // Rank r adds up rows [r * rows, (r + 1) * rows) of the tile: one float4
  // of 4 columns per thread and step, ranks in order 0, 1, ...
  const int rows = Q::BM / split;
  const uint32_t p_local = smem_u32(P);
  for (int e = t; e < rows * (Q::BN / 4); e += Q::THREADS) {
    const int r = rank * rows + e / (Q::BN / 4);
    const int c = (e % (Q::BN / 4)) * 4;
    const uint32_t off = static_cast<uint32_t>((r * P_LD + c) * 4);
    // every rank's value is loaded before the first add, so that the remote
    // loads' latencies overlap; the sum still runs over ranks 0, 1, ...
    float4 v[kMaxClusterSplit];
#pragma unroll
    for (int q = 0; q < kMaxClusterSplit; ++q)
      if (q < split) v[q] = ld_dsmem_f4(mapa_shared(p_local + off, static_cast<uint32_t>(q)));
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < kMaxClusterSplit; ++q) {
      if (q < split) {
        s.x += v[q].x;
        s.y += v[q].y;
        s.z += v[q].z;
        s.w += v[q].w;
      }
    }
    store4(args, m0 + r, n0 + c, s);
  }
  // No CTA leaves while another still reads its partial tile. The values read
  // were all consumed above, so the arrival needs no release ordering.
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" :::
                   "memory");
}

template <bool kVec>
cudaError_t launch_small(const GemmArgs& args, int split, int kb_per, int tiles,
                         cudaStream_t stream) {
  static DeviceOnce configured;
  cudaError_t e = set_smem_once(configured, sgemm_small_kernel<kVec>, Q::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(split);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(split) * static_cast<unsigned>(tiles));
  cfg.blockDim = dim3(Q::THREADS);
  cfg.dynamicSmemBytes = Q::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, sgemm_small_kernel<kVec>, args, split, kb_per);
}

}  // namespace

cudaError_t launch_sgemm_small(const GemmArgs& args, bool vec_loads, int split, int tiles,
                               cudaStream_t stream) {
  if (split < 1 || split > 8 || (Q::BM % split) != 0 || tiles < 1) return cudaErrorInvalidValue;
  const int L = (args.K + Q::BK - 1) / Q::BK;
  const int kb_per = (L + split - 1) / split;
  return vec_loads ? launch_small<true>(args, split, kb_per, tiles, stream)
                   : launch_small<false>(args, split, kb_per, tiles, stream);
}

}  // namespace gemm14
