// kernels.h -- internal interface between the C-ABI layer (api.cu) and the
// kernel translation units. Nothing here crosses the library boundary.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <mutex>
#include <utility>

#include "checks.h"
#include "streamk.cuh"

namespace gemm14 {

// Launches kernel over grid x block threads with smem bytes of dynamic shared
// memory on stream, with programmatic stream serialisation: the grid may be
// launched while the previous grid on the stream still runs, and waits for it
// inside (grid_dependency_wait) before touching global memory. This hides the
// gap between back-to-back products (a few microseconds per launch).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// A value worked out once per device (a kernel's shared-memory attribute set,
// an occupancy query) and reused by later calls on that device. First calls
// from several host threads at once are serialised by the lock: one runs
// set_up(), the others then read its result. A result for which keep(v) is
// false (a failed set-up) is returned but not stored, so the next call on the
// device tries again.
class DeviceOnce {
 public:
  static constexpr int kDevices = 64;
  DeviceOnce() {
    for (auto& v : value_) v.store(kUnset, std::memory_order_relaxed);
  }
  template <typename SetUp, typename Keep>
  int get(int dev, SetUp&& set_up, Keep&& keep) {
    if (dev < 0 || dev >= kDevices) return set_up();
    int v = value_[dev].load(std::memory_order_acquire);
    if (v != kUnset) return v;
    std::lock_guard<std::mutex> lock(mutex_);
    v = value_[dev].load(std::memory_order_relaxed);
    if (v != kUnset) return v;
    v = set_up();
    if (keep(v)) value_[dev].store(v, std::memory_order_release);
    return v;
  }

 private:
  static constexpr int kUnset = INT_MIN;
  std::atomic<int> value_[kDevices];
  std::mutex mutex_;
};

// Sets `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device (see DeviceOnce; `once` is the kernel's own).
template <typename Kernel>
cudaError_t set_smem_once(DeviceOnce& once, Kernel kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return static_cast<cudaError_t>(once.get(
      dev,
      [&] {
        return static_cast<int>(
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
      },
      [](int r) { return r == static_cast<int>(cudaSuccess); }));
}

// How the epilogue writes an output element from its sum s:
//   kEpiStore  C = s                     (alpha = 1, beta = 0)
//   kEpiScale  C = alpha * s             (beta = 0: C is not read)
//   kEpiAccum  C = alpha * s + beta * C  (one fp32 fma on beta * C)
enum : int { kEpiStore = 0, kEpiScale = 1, kEpiAccum = 2 };

// Arguments shared by every kernel: sizes, operand pointers and the library's
// device error word (a plain device pointer, see api.cu).
// Operand storage: op(A) is M x K and op(B) is K x N. transa == 0: A is a
// row-major M x K matrix (element (i, k) at A[i * lda + k]); transa == 1: A is
// stored K x M (element (i, k) at A[k * lda + i]). Likewise transb == 0: B is
// K x N (B[k * ldb + j]); transb == 1: B is stored N x K (B[j * ldb + k]).
struct GemmArgs {
  int M, N, K;
  const void* A;
  int64_t lda;
  const void* B;
  int64_t ldb;
  float* C;
  int64_t ldc;
  int vec_store;  // C rows may take 16-byte stores (C 16-B aligned, ldc % 4 == 0)
  int transa, transb;
  int epi;              // kEpiStore / kEpiScale / kEpiAccum
  float alpha, beta;
  unsigned* err;
  unsigned long long wait_limit_ns;  // time limit of one mbarrier wait
  int fault;  // kFaultNone, or kFaultSkipFirstStage (failure-detection tests only)
  StreamK sk;          // work schedule; sk.G == number of workers launched
  float* partials;     // stream-K: tile-sized fp32 slots (see streamk_workspace_bytes), or null
  unsigned* flags;     // stream-K: G publication flags (hold the call's epoch)
  unsigned epoch;      // this call's nonzero epoch
  // Terms of the k sum (the pair kernel's tf32 variant): 0 or 1, the plain
  // product; 3, the split-precision 3xTF32 product from operands split ahead
  // of the call, lo(A) hi(B) + hi(A) lo(B) + hi(A) hi(B), run as 3 x the
  // k-blocks of one term (see launch_hgemm_tc_pair).
  int k_terms;
};

// The epilogue's update of one output element, and of four consecutive ones
// (p 16-byte aligned). kEpiAccum reads C; the others do not. kGeneral false:
// a plain store, with args.epi not consulted (kernels compiled for the
// kEpiStore case only).
// Both skip a store outside C's M x N block when the device-side bounds checks
// are compiled in (checks.h).
template <bool kGeneral>
__device__ __forceinline__ void epi_store1(const GemmArgs& a, float* p, float s) {
  if (!dev_check(c_span_ok(p - a.C, a.ldc, a.M, a.N, 1), a.err)) return;
  if (!kGeneral || a.epi == kEpiStore) *p = s;
  else if (a.epi == kEpiScale) *p = a.alpha * s;
  else *p = fmaf(a.alpha, s, a.beta * *p);
}
template <bool kGeneral>
__device__ __forceinline__ void epi_store4(const GemmArgs& a, float* p, float4 v) {
  if (!dev_check(c_span_ok(p - a.C, a.ldc, a.M, a.N, 4), a.err)) return;
  float4* q = reinterpret_cast<float4*>(p);
  if (!kGeneral || a.epi == kEpiStore) {
    *q = v;
  } else if (a.epi == kEpiScale) {
    *q = make_float4(a.alpha * v.x, a.alpha * v.y, a.alpha * v.z, a.alpha * v.w);
  } else {
    const float4 c = *q;
    *q = make_float4(fmaf(a.alpha, v.x, a.beta * c.x), fmaf(a.alpha, v.y, a.beta * c.y),
                     fmaf(a.alpha, v.z, a.beta * c.z), fmaf(a.alpha, v.w, a.beta * c.w));
  }
}

// Stream-K workspace layout on a GPU with `sms` SMs: first one flag word
// per SM (a region whose place and size never depend on the product, so a
// workspace reused for another shape never finds partial sums where a flag
// is expected), then `spw` tile slots of bm x bn floats per worker (slot w: a
// worker's PARTIAL).
inline size_t streamk_flag_bytes(int sms) {
  return ((static_cast<size_t>(sms) * sizeof(unsigned) + 255) / 256) * 256;
}
inline size_t streamk_workspace_bytes(int sms, int bm, int bn, int spw) {
  return streamk_flag_bytes(sms) + static_cast<size_t>(spw) * sms * bm * bn * sizeof(float);
}

// Fault modes a test may request for one call (see gemm14_debug_inject).
enum : int { kFaultNone = 0, kFaultSkipFirstStage = 1 };

// ---- fp32 SIMT kernel (sgemm_simt.cu)
struct SgemmShape {
  static constexpr int BM = 128, BN = 256, BK = 32, STAGES = 4;
  static constexpr int WARPS = 8;  // all compute; thread 0 also issues the TMA loads
  static constexpr int THREADS = WARPS * 32;
  static constexpr int A_STAGE_BYTES = BM * BK * 4;
  static constexpr int B_STAGE_BYTES = BK * BN * 4;
  static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
  // + barriers, schedule table and the loaders' cursors (20 B per thread) + align slack
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 512 + 20 * THREADS + 1024;
  // B stored N x K read by TMA (layout bit 1): each stage's B tile is
  // transposed in shared memory into one of two [k][n] buffers, and the ring
  // has one stage fewer to make room for them.
  static constexpr int BT_BYTES = BK * BN * 4;
  static constexpr int stages(int lay) { return (lay & 2) ? STAGES - 1 : STAGES; }
  static constexpr int smem_bytes(int lay) {
    return stages(lay) * STAGE_BYTES + ((lay & 2) ? 2 * BT_BYTES : 0) + 512 + 20 * THREADS + 1024;
  }
};

// Loader: TMA tensor maps (A box 32 x 128 with 128-byte swizzle, B box
// 256 x 32) or, when the operands break TMA's 16-byte rules, cp.async.
cudaError_t launch_sgemm_tma(const CUtensorMap& map_a, const CUtensorMap& map_b,
                             const GemmArgs& args, int grid, cudaStream_t stream);
cudaError_t launch_sgemm_cpasync(const GemmArgs& args, int grid, cudaStream_t stream);

// ---- fp32 products with few 128 x 256 tiles (sgemm_small.cu): 64 x 64 tiles,
// the k range of each split over a cluster of `split` CTAs (1, 2, 4 or 8)
// whose partial tiles are added through distributed shared memory.
struct SmallShape {
  static constexpr int BM = 64, BN = 64, BK = 32, STAGES = 3, THREADS = 128;
  // 3 stages of A [64][36] + B [32][68] floats
  static constexpr int SMEM_BYTES = STAGES * (BM * (BK + 4) + BK * (BN + 4)) * 4;
};
// vec_loads: A stored M x K and B stored K x N, 16-byte aligned, pitches
// multiples of 4 floats (16-byte copies); else 4-byte copies (any storage,
// pitch or alignment). tiles: 64 x 64 output tiles; the grid is split x tiles.
cudaError_t launch_sgemm_small(const GemmArgs& args, bool vec_loads, int split, int tiles,
                               cudaStream_t stream);

// ---- bf16 / fp16 tcgen05 kernel (hgemm_tc.cu): tiles of bm x bn on one SM,
// bm = 128 (M = 128 MMAs) or 64 (M = 64 MMAs, for products whose 128-row
// tiles would leave SMs idle).
struct HgemmShape {
  static constexpr int BM = 128, BK = 64;
  static constexpr int THREADS = 6 * 32;  // producer, MMA, 4 epilogue warps
  // + the software loader's warps when an operand breaks TMA's rules
  static constexpr int SOFT_WARPS = 8;
  static constexpr int SOFT_THREADS = THREADS + 32 * SOFT_WARPS;
  static constexpr int stages(int bn, int bm = 128) {
    return bm == 128 ? (bn == 256 ? 4 : bn == 128 ? 6 : 8) : (bn == 256 ? 4 : bn == 128 ? 8 : 12);
  }
  static constexpr int stage_bytes(int bn, int bm = 128) { return bm * BK * 2 + BK * bn * 2; }
  // epilogue staging for TMA stores of C: per epilogue warp two buffers of
  // bm / 4 rows x 32 fp32 columns (4 KB each for bm = 128)
  static constexpr int out_buf_bytes(int bm = 128) { return (bm / 4) * 32 * 4; }
  static constexpr int out_bytes(int bm = 128) { return 4 * 2 * out_buf_bytes(bm); }
  static constexpr int SMEM_RESERVE = 512;  // barriers and the stream-K table
  static constexpr int smem_bytes(int bn, int bm = 128) {
    return stages(bn, bm) * stage_bytes(bn, bm) + out_bytes(bm) + SMEM_RESERVE + 1024;
  }
};

// bm in {64, 128}, bn in {64, 128, 256}; idesc is the tcgen05 instruction
// descriptor (operand format and shape M = bm, N = bn); map_a boxes are 64 k x
// bm rows (A stored M x K) or 64 m x 64 k (stored K x M); map_b boxes are 64
// (n) x 64 (k). map_c: C as a 2-D fp32 tensor (box 32 columns x bm / 4 rows,
// 128-byte swizzle) for the TMA-store epilogue of the plain variant when C
// takes 16-byte stores.
cudaError_t launch_hgemm_tc(int bm, int bn, const CUtensorMap& map_a, const CUtensorMap& map_b,
                            const CUtensorMap& map_c, const GemmArgs& args, uint32_t idesc,
                            int grid, cudaStream_t stream);
// ---- bf16 / fp16 tcgen05 kernel on CTA pairs (hgemm_tc2.cu): 256 x 256 tiles
struct PairShape {
  static constexpr int BM = 256, BN = 256, BK = 64, STAGES = 6;
  static constexpr int THREADS = 6 * 32;
  static constexpr int A_BYTES = 128 * BK * 2;      // this CTA's 128 rows of A
  static constexpr int B_BYTES = BK * 128 * 2;      // this CTA's 128 columns of B
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // epilogue staging for TMA stores of C: per epilogue warp two buffers of
  // 32 rows x 32 fp32 columns (4 KB each)
  static constexpr int OUT_BUF_BYTES = 32 * 32 * 4;
  static constexpr int OUT_BYTES = 4 * 2 * OUT_BUF_BYTES;
  static constexpr int TMEM_COLS = 512;             // two 128-lane x 256-column accumulators
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + OUT_BYTES + 256 + 1024;
};

// Clusters of two that fit at once on the current device (0: the pair kernel
// cannot run). The first call per device also sets the kernel's smem limit.
int pair_max_clusters();
// map_c: C as a 2-D fp32 tensor (box 32 columns x 32 rows, 128-byte swizzle)
// for the TMA-store epilogue of the plain variant when C takes 16-byte stores
// (args.vec_store); otherwise unused.
// tf32: fp32 operands stored M x K and N x K read as tf32 (kind::tf32, a
// k-block of 32 elements; maps of fp32 boxes 32 k x 128 rows, 128-byte swizzle).
// With args.k_terms == 3 (tf32 only), map_a_lo and map_b_lo describe lo(A) and
// lo(B) (x minus x with its 13 low fraction bits cleared) in the same storage
// and boxes as map_a and map_b, which hold A and B themselves (the tensor
// cores read them as hi(A) and hi(B)); otherwise both are unused.
cudaError_t launch_hgemm_tc_pair(const CUtensorMap& map_a, const CUtensorMap& map_b,
                                 const CUtensorMap& map_c, const CUtensorMap& map_a_lo,
                                 const CUtensorMap& map_b_lo, const GemmArgs& args,
                                 uint32_t idesc, int clusters, bool tf32, cudaStream_t stream);

// Same kernel with the software loader for the operands TMA cannot address:
// soft bit 0 = A, bit 1 = B; the other operand (if any) comes by TMA through
// its map (map_a / map_b; the software operand's may be null).
cudaError_t launch_hgemm_tc_soft(int bm, int bn, int soft, const CUtensorMap* map_a,
                                 const CUtensorMap* map_b, const GemmArgs& args, uint32_t idesc,
                                 int grid, cudaStream_t stream);

// ---- fp32 inputs on the tensor cores (sgemm_tc3.cu): tcgen05 kind::tf32 on
// CTA pairs, 256 x 256 tiles. The tensor cores read an fp32 operand as tf32 by
// dropping its 13 low fraction bits: hi(x). terms = 1 computes hi(A) hi(B)
// (TF32); terms = 3 adds hi(A) lo(B) + lo(A) hi(B) with lo(x) = x - hi(x),
// written by converter warps ("3xTF32").
struct Tf32Shape {
  static constexpr int BM = 256, BN = 256, BK = 32;  // k-block: 32 fp32 = one 128-byte row
  static constexpr int OP_STAGES = 2;       // 3xTF32
  static constexpr int OP_STAGES_TF32 = 4;  // TF32: compact stages (copies only)
  static constexpr int MAX_RAW_STAGES = 5;
  // producer, MMA, 4 epilogue, 4 converter warps; TF32 adds two announcer
  // warps (each forwards every other k-block's operand stage)
  static constexpr int THREADS = 12 * 32;
  static constexpr int threads(bool three) { return three ? 10 * 32 : THREADS; }
  static constexpr int op_stages(bool three) { return three ? OP_STAGES : OP_STAGES_TF32; }
  static constexpr int TILE = 128 * BK * 4;       // one CTA's 128 rows x 32 k of fp32: 16 KB
  static constexpr int RAW_STAGE = 2 * TILE;      // A, B as loaded
  static constexpr int RING_BYTES = 224 * 1024;   // raw + operand rings
  static constexpr int TMEM_COLS = 512;
  static constexpr int SMEM_BYTES = RING_BYTES + 512 + 1024;
};

// Clusters of two the tf32 kernel fits at once on the current device (0: it
// cannot run). The first call per device also sets the kernels' smem limit.
int tf32_pair_max_clusters();
// map_a / map_b: A stored M x K: box 32 k x 128 m, 128-byte swizzle; stored
// K x M (transa): box 128 m x 32 k, no swizzle. B stored K x N: box 128 n x
// 32 k, no swizzle; stored N x K (transb): box 32 k x 128 n, 128-byte swizzle.
cudaError_t launch_sgemm_tf32_pair(const CUtensorMap& map_a, const CUtensorMap& map_b,
                                   const GemmArgs& args, int terms, int clusters,
                                   cudaStream_t stream);

// A rows x cols matrix to copy from row pitch ld_src to row pitch ld_dst
// (rows = 0: nothing).
struct RepitchJob {
  const void* src;
  int64_t ld_src;
  void* dst;
  int64_t ld_dst;
  int64_t rows, cols;
  int transpose;  // relayout only: the destination is the cols x rows transpose
  // relayout only: when set, lo(x) = x - (x with its 13 low fraction bits
  // cleared) of each element goes here, placed and pitched as in dst (which
  // may then be null: no copy of x itself)
  void* dst_lo;
};
// Both copies in one launch on `stream`, elements of elem_bytes (2 or 4) (copy.cu).
cudaError_t launch_repitch(const RepitchJob& j0, const RepitchJob& j1, int elem_bytes,
                           int sm_count, cudaStream_t stream);
// Both fp32 copies in one launch, each transposed when job.transpose, and each
// also (or only) split into its lo part when job.dst_lo (copy.cu).
cudaError_t launch_relayout(const RepitchJob& j0, const RepitchJob& j1, int sm_count,
                            cudaStream_t stream);

// ---- C = beta * C over an M x N block (epilogue.cu): the call when the
// product term vanishes (K == 0 or alpha == 0) and beta is not 0 or 1.
cudaError_t launch_scale_c(float* C, int64_t ldc, int M, int N, float beta, int sm_count,
                           cudaStream_t stream);

}  // namespace gemm14
