// api.cu -- the C ABI of libgemm14.so: argument validation, launch planning,
// TMA tensor-map encoding, device checks and error reporting.
// The contract of each entry point is documented in include/gemm14.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/gemm14.h"
#include "api_internal.h"
#include "plan.h"
#include "kernels.h"
#include "ptx.cuh"

namespace gemm14 {
namespace {

// The library's device error word: kernels OR kDevErr* bits into it when a
// bounded wait expires. Host code reaches it through the address cached per
// device below (a symbol's host-side name is not a device address).
__device__ unsigned g_device_error;

thread_local char t_last_error[256] = "";

// Stream-K publication flags hold the epoch of the call that wrote them; a
// call's epoch is never 0 and differs from the previous 2^32 - 1 calls'.
std::atomic<unsigned> g_epoch{0};
unsigned next_epoch() {
  unsigned e;
  do { e = ++g_epoch; } while (e == 0);
  return e;
}

// One-shot request from gemm14_debug_inject for the next call on this thread.
thread_local int t_fault = kFaultNone;
thread_local unsigned long long t_wait_limit_ns = 0;

void set_cuda_error(const char* what, cudaError_t e) {
  std::snprintf(t_last_error, sizeof t_last_error, "%s: %s (%d)", what, cudaGetErrorString(e),
                static_cast<int>(e));
}

void set_driver_error(const char* what, CUresult r) {
  std::snprintf(t_last_error, sizeof t_last_error, "%s: CUresult %d", what, static_cast<int>(r));
}

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int sm_count = 0;
  unsigned* err_word = nullptr;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mutex;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode_tiled = nullptr;
std::once_flag g_encode_once;

// Looks up the current device once: compute capability, SM count and the
// device address of the error word. Returns a gemm14_status.
int current_device(const DeviceInfo** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_cuda_error("cudaGetDevice", e);
    return GEMM14_ERR_UNSUPPORTED_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return GEMM14_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_devices_mutex);
  DeviceInfo& d = g_devices[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) {
      set_cuda_error("cudaDeviceGetAttribute", e);
      return GEMM14_ERR_CUDA;
    }
    d.supported = (major == 10 && minor == 3);
    d.sm_count = sms;
    if (d.supported) {
      void* p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_device_error)) != cudaSuccess) {
        set_cuda_error("cudaGetSymbolAddress(error word)", e);
        return GEMM14_ERR_CUDA;
      }
      d.err_word = static_cast<unsigned*>(p);
    }
    d.ready = true;
  }
  if (!d.supported) return GEMM14_ERR_UNSUPPORTED_DEVICE;
  *out = &d;
  return GEMM14_OK;
}

int encoder(EncodeTiledFn* fn) {
  std::call_once(g_encode_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                     cudaEnableDefault, &q);
    if (e == cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_encode_tiled = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!g_encode_tiled) {
    std::snprintf(t_last_error, sizeof t_last_error, "cuTensorMapEncodeTiled not available");
    return GEMM14_ERR_CUDA;
  }
  *fn = g_encode_tiled;
  return GEMM14_OK;
}

// 2-D row-major tensor map: `rows` x `cols` elements, row pitch ld elements,
// box = box_cols (inner) x box_rows, zero fill out of range.
int make_map(CUtensorMap* map, CUtensorMapDataType type, int elem_bytes, const void* base,
             int64_t rows, int64_t cols, int64_t ld, int box_cols, int box_rows,
             CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = nullptr;
  int st = encoder(&fn);
  if (st != GEMM14_OK) return st;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * elem_bytes};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, type, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_driver_error("cuTensorMapEncodeTiled", r);
    return GEMM14_ERR_CUDA;
  }
  return GEMM14_OK;
}

// Argument validation shared by the entry points and the planner. transa /
// transb select the stored shape of A (M x K, or K x M) and of B (K x N, or
// N x K); each must be 0 or 1.
int validate(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K, const void* A,
             int64_t lda, const void* B, int64_t ldb, const void* C, int64_t ldc) {
  if (dtype != GEMM14_DTYPE_F32 && dtype != GEMM14_DTYPE_BF16 && dtype != GEMM14_DTYPE_F16 &&
      !is_tf32_mode(dtype))
    return GEMM14_ERR_INVALID_ARG;
  if ((transa != 0 && transa != 1) || (transb != 0 && transb != 1)) return GEMM14_ERR_INVALID_ARG;
  const int64_t kMax = INT32_MAX;
  if (M < 0 || N < 0 || K < 0 || M > kMax || N > kMax || K > kMax) return GEMM14_ERR_INVALID_ARG;
  const int64_t a_cols = transa ? M : K, b_cols = transb ? K : N;
  if (lda < (a_cols > 1 ? a_cols : 1) || ldb < (b_cols > 1 ? b_cols : 1) ||
      ldc < (N > 1 ? N : 1))
    return GEMM14_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM14_OK;
  if (!C || !aligned(C, 4)) return GEMM14_ERR_INVALID_ARG;
  if (K == 0) return GEMM14_OK;
  const int eb = elem_bytes_of(dtype);
  if (!A || !B || !aligned(A, eb) || !aligned(B, eb)) return GEMM14_ERR_INVALID_ARG;
  // TMA strides must stay below 2^40 bytes.
  if (lda > (int64_t(1) << 36) || ldb > (int64_t(1) << 36)) return GEMM14_ERR_INVALID_ARG;
  return GEMM14_OK;
}
int validate(int dtype, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
             const void* B, int64_t ldb, const void* C, int64_t ldc) {
  return validate(dtype, 0, 0, M, N, K, A, lda, B, ldb, C, ldc);
}

bool debug_checks() {
  static const bool on = [] {
    const char* v = std::getenv("GEMM14_DEBUG");
    return v && v[0] && v[0] != '0';
  }();
  return on;
}

int finish(cudaError_t e, const char* what, cudaStream_t stream) {
  if (e != cudaSuccess) {
    set_cuda_error(what, e);
    return GEMM14_ERR_CUDA;
  }
  if (debug_checks()) return gemm14_check_device_error(stream);
  return GEMM14_OK;
}

// The schedule of a one-SM-per-tile launch: data-parallel over min(tiles, SMs)
// CTAs, or, with a large enough workspace, stream-K over all SMs.
void schedule(const gemm14_plan& plan, int64_t K, int sm_count, void* workspace,
              size_t workspace_bytes, GemmArgs& args, int& grid) {
  const int tiles = static_cast<int>(plan.tiles);
  const int L = static_cast<int>((K + plan.bk - 1) / plan.bk);
  const size_t need = workspace_need(plan, sm_count, K);
  const bool sk = workspace && need && workspace_bytes >= need;
  if (sk) {
    args.sk = make_stream_k(tiles, L, one_sm_split_workers(plan.kernel, tiles, L, sm_count),
                            true);
    // Flags first (a fixed region), then the slots; sk.G <= sm_count.
    args.flags = static_cast<unsigned*>(workspace);
    args.partials = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                             streamk_flag_bytes(sm_count));
    args.epoch = next_epoch();
    grid = args.sk.G;
  } else {
    grid = tiles < sm_count ? tiles : sm_count;
    args.sk = make_stream_k(tiles, L, grid, false);
    args.partials = nullptr;
    args.flags = nullptr;
    args.epoch = 0;
  }
}

// Tensor maps of the 16-bit kernels for a tile of bm rows x bn columns:
// A stored M x K: box 64 k x bm m; stored K x M: box 64 m x 64 k (bm / 64
// loads per stage). B stored K x N: box 64 n x 64 k (bn / 64 loads); stored
// N x K: box 64 k x bn n. All with the 128-byte swizzle.
// ma / mb may be null: that operand gets no map (the software loader reads it).
int make_maps_16(bool bf16, int transa, int transb, int64_t M, int64_t N, int64_t K,
                 const void* A, int64_t lda, const void* B, int64_t ldb, int bm, int bn,
                 CUtensorMap* ma, CUtensorMap* mb) {
  const CUtensorMapDataType tt =
      bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  int st = GEMM14_OK;
  if (ma)
    st = transa ? make_map(ma, tt, 2, A, K, M, lda, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B)
                : make_map(ma, tt, 2, A, M, K, lda, 64, bm, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != GEMM14_OK || !mb) return st;
  return transb ? make_map(mb, tt, 2, B, N, K, ldb, 64, bn, CU_TENSOR_MAP_SWIZZLE_128B)
                : make_map(mb, tt, 2, B, K, N, ldb, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
}

// The CTA-pair kernel (plan kernels 3 and 5): data-parallel over
// min(tiles, clusters) clusters, or, with a large enough workspace, stream-K
// over all co-resident clusters (workers).
int run_pair(const gemm14_plan& plan, GemmArgs& args, const CUtensorMap& ma,
             const CUtensorMap& mb, const CUtensorMap& ma_lo, const CUtensorMap& mb_lo,
             int pair_clusters, bool tf32, uint32_t idesc, int64_t K, int sm_count,
             void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  int clusters = static_cast<int>(plan.tiles < pair_clusters ? plan.tiles : pair_clusters);
  const int terms = args.k_terms == 3 ? 3 : 1;  // k-blocks of the split 3xTF32 sum
  const int L = static_cast<int>((K + plan.bk - 1) / plan.bk) * terms;
  const size_t need = workspace_need(plan, sm_count, K, terms);
  const int workers = pair_split_workers(plan.tiles, L, pair_clusters);
  if (workspace && need && workspace_bytes >= need && workers > 0) {
    if (plan.tiles >= 2 * static_cast<int64_t>(pair_clusters))
      // whole waves data-parallel, the last one and a half split
      args.sk = make_stream_k(static_cast<int>(plan.tiles), L, workers, true);
    else  // fewer than two waves: every tile split (dp_tiles = 0)
      args.sk = StreamK{static_cast<int>(plan.tiles), L, workers, 0};
    args.flags = static_cast<unsigned*>(workspace);
    args.partials = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                             streamk_flag_bytes(sm_count));
    args.epoch = next_epoch();
    clusters = args.sk.G;
  } else {
    args.sk = make_stream_k(static_cast<int>(plan.tiles), L, clusters, false);
  }
  // C for the TMA-store epilogue of the plain variants (plain stores into a
  // 16-byte-aligned C): box 32 columns x 32 rows of fp32, 128-byte swizzle.
  // The variant is plain exactly when launch_hgemm_tc_pair picks it.
  const bool general = (!tf32 && (args.transa || args.transb)) || args.epi != kEpiStore;
  CUtensorMap mc{};
  if (!general && plan.vec_store) {
    const int st = make_map(&mc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, args.C, args.M, args.N,
                            args.ldc, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != GEMM14_OK) return st;
  }
  return finish(launch_hgemm_tc_pair(ma, mb, mc, ma_lo, mb_lo, args, idesc, clusters, tf32,
                                     stream),
                "hgemm pair launch", stream);
}

int run_gemm(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K, float alpha,
             const void* A, int64_t lda, const void* B, int64_t ldb, float beta, float* C,
             int64_t ldc, void* workspace, size_t workspace_bytes, void* stream_ptr) {
  // A pending test request applies to this call only, whatever its outcome.
  const int fault = t_fault;
  const unsigned long long wait_limit_ns = t_wait_limit_ns ? t_wait_limit_ns : kWaitTimeoutNs;
  t_fault = kFaultNone;
  t_wait_limit_ns = 0;
  int st = validate(dtype, transa, transb, M, N, K, A, lda, B, ldb, C, ldc);
  if (st != GEMM14_OK) return st;
  if (workspace && !aligned(workspace, 16)) return GEMM14_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM14_OK;
  const DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev)) != GEMM14_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

  if (K == 0 || alpha == 0.0f) {
    // No product term (A and B are not read): C = beta * C.
    if (beta == 1.0f) return GEMM14_OK;
    if (beta == 0.0f) {
      cudaError_t e = cudaMemset2DAsync(C, static_cast<size_t>(ldc) * 4, 0,
                                        static_cast<size_t>(N) * 4, static_cast<size_t>(M),
                                        stream);
      return finish(e, "cudaMemset2DAsync", stream);
    }
    return finish(launch_scale_c(C, ldc, static_cast<int>(M), static_cast<int>(N), beta,
                                 dev->sm_count, stream),
                  "scale launch", stream);
  }

  // Operands TMA cannot read: with room in the workspace, copy them there with
  // 16-byte pitches first; the call then keeps the workspace's start (up to
  // the copies) for the stream-K schedule. 3xTF32 on the pair kernel also
  // writes lo(A) and lo(B) there (k_terms = 3; A and B are read as hi).
  int k_terms = 1;
  const void* A_lo = nullptr;
  const void* B_lo = nullptr;
  int64_t ld_lo = 0;
  if (workspace) {
    Repitch rp;
    plan_repitch(dtype, transa, transb, M, N, K, A, lda, B, ldb, C, ldc, dev->sm_count, &rp);
    if ((rp.a || rp.b || rp.split) && workspace_bytes >= rp.total) {
      char* ws = static_cast<char*>(workspace);
      RepitchJob ja{}, jb{};
      // source rows x cols as stored; the copy (and lo part) is that, or its
      // transpose. With the split a copy's pitch is ld_lo as well.
      if (rp.a || rp.split) {
        ja = RepitchJob{A, lda, rp.a ? ws + rp.a_off : nullptr, rp.split ? rp.ld_lo : rp.lda,
                        transa ? K : M, transa ? M : K, rp.a_t ? 1 : 0,
                        rp.split ? ws + rp.a_lo_off : nullptr};
        if (rp.a) {
          A = ws + rp.a_off;
          lda = rp.lda;
        }
      }
      if (rp.b || rp.split) {
        jb = RepitchJob{B, ldb, rp.b ? ws + rp.b_off : nullptr, rp.split ? rp.ld_lo : rp.ldb,
                        transb ? N : K, transb ? K : N, rp.b_t ? 1 : 0,
                        rp.split ? ws + rp.b_lo_off : nullptr};
        if (rp.b) {
          B = ws + rp.b_off;
          ldb = rp.ldb;
        }
      }
      transa = rp.transa;
      transb = rp.transb;
      const cudaError_t e =
          rp.a_t || rp.b_t || rp.split
              ? launch_relayout(ja, jb, dev->sm_count, stream)
              : launch_repitch(ja, jb, elem_bytes_of(dtype), dev->sm_count, stream);
      if (e != cudaSuccess) return finish(e, "re-pitch launch", stream);
      workspace_bytes = rp.a_off;
      if (rp.split) {
        k_terms = 3;
        A_lo = ws + rp.a_lo_off;
        B_lo = ws + rp.b_lo_off;
        ld_lo = rp.ld_lo;
        dtype = GEMM14_DTYPE_TF32;  // planned as TF32, run with 3 terms
      }
    }
  }

  // With a workspace, plan for a split; if the split that plan counts on
  // does not fit the workspace left (an fp32 product of few tiles), plan as
  // the call without a workspace.
  bool split_ok = workspace != nullptr;
  gemm14_plan plan;
  plan_for(dtype, transa, transb, M, N, K, A, lda, B, ldb, C, ldc, dev->sm_count, &plan, split_ok);
  if (split_ok && plan.kernel == 1 && workspace_bytes < workspace_need(plan, dev->sm_count, K)) {
    split_ok = false;
    plan_for(dtype, transa, transb, M, N, K, A, lda, B, ldb, C, ldc, dev->sm_count, &plan);
  }
  const int epi = beta != 0.0f ? kEpiAccum : alpha != 1.0f ? kEpiScale : kEpiStore;
  GemmArgs args{static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                A, lda, B, ldb, C, ldc, plan.vec_store, transa, transb, epi, alpha, beta,
                dev->err_word, wait_limit_ns, fault, StreamK{}, nullptr, nullptr, 0u, k_terms};
  int grid = plan.grid;

  if (plan.kernel == 5) {
    const int pair_clusters = pair_max_clusters();
    if (pair_clusters > 0) {
      // A stored M x K, B stored N x K: boxes of 32 k (128 bytes) x 128 rows
      // (and so lo(A), lo(B) in the workspace)
      CUtensorMap ma, mb, ma_lo{}, mb_lo{};
      const CUtensorMapDataType f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
      if ((st = make_map(&ma, f32, 4, A, M, K, lda, 32, 128, CU_TENSOR_MAP_SWIZZLE_128B)) !=
              GEMM14_OK ||
          (st = make_map(&mb, f32, 4, B, N, K, ldb, 32, 128, CU_TENSOR_MAP_SWIZZLE_128B)) !=
              GEMM14_OK)
        return st;
      if (k_terms == 3 &&
          ((st = make_map(&ma_lo, f32, 4, A_lo, M, K, ld_lo, 32, 128,
                          CU_TENSOR_MAP_SWIZZLE_128B)) != GEMM14_OK ||
           (st = make_map(&mb_lo, f32, 4, B_lo, N, K, ld_lo, 32, 128,
                          CU_TENSOR_MAP_SWIZZLE_128B)) != GEMM14_OK))
        return st;
      return run_pair(plan, args, ma, mb, ma_lo, mb_lo, pair_clusters, true,
                      idesc_tf32_f32acc(PairShape::BM, PairShape::BN), K, dev->sm_count,
                      workspace, workspace_bytes, stream);
    }
    // clusters of two do not fit: plan without the pair kernel (the split
    // operands' hi parts are A and B themselves: 3xTF32 on the converter kernel)
    g_pair_enabled.store(0);
    if (k_terms == 3) {
      dtype = GEMM14_DTYPE_F32_3XTF32;
      k_terms = 1;
      args.k_terms = 1;
    }
    plan_for(dtype, transa, transb, M, N, K, A, lda, B, ldb, C, ldc, dev->sm_count, &plan,
             split_ok);
    args.vec_store = plan.vec_store;
    grid = plan.grid;
  }
  if (plan.kernel == 4) {
    const int clusters_max = tf32_pair_max_clusters();
    if (clusters_max > 0) {
      CUtensorMap ma, mb;
      const CUtensorMapDataType f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
      st = transa ? make_map(&ma, f32, 4, A, K, M, lda, 128, Tf32Shape::BK,
                             CU_TENSOR_MAP_SWIZZLE_NONE)
                  : make_map(&ma, f32, 4, A, M, K, lda, Tf32Shape::BK, 128,
                             CU_TENSOR_MAP_SWIZZLE_128B);
      if (st != GEMM14_OK) return st;
      st = transb ? make_map(&mb, f32, 4, B, N, K, ldb, Tf32Shape::BK, 128,
                             CU_TENSOR_MAP_SWIZZLE_128B)
                  : make_map(&mb, f32, 4, B, K, N, ldb, 128, Tf32Shape::BK,
                             CU_TENSOR_MAP_SWIZZLE_NONE);
      if (st != GEMM14_OK) return st;
      const int64_t clusters = plan.tiles < clusters_max ? plan.tiles : clusters_max;
      const int terms = dtype == GEMM14_DTYPE_F32_3XTF32 ? 3 : 1;
      return finish(launch_sgemm_tf32_pair(ma, mb, args, terms, static_cast<int>(clusters), stream),
                    "tf32 pair launch", stream);
    }
    // clusters of the tf32 kernel do not fit: the fp32 SIMT kernel
    dtype = GEMM14_DTYPE_F32;
    plan_for(dtype, transa, transb, M, N, K, A, lda, B, ldb, C, ldc, dev->sm_count, &plan,
             split_ok);
    args.vec_store = plan.vec_store;
    grid = plan.grid;
  }
  if (is_tf32_mode(dtype)) dtype = GEMM14_DTYPE_F32;  // planned on the SIMT kernel

  if (dtype == GEMM14_DTYPE_F32 && plan.kernel == 6) {
    // few tiles: 64 x 64 tiles, k split over clusters (no workspace)
    const int tiles = static_cast<int>(plan.tiles);
    return finish(launch_sgemm_small(args, plan.loader == 1, plan.grid / tiles, tiles, stream),
                  "sgemm small launch", stream);
  }
  if (dtype == GEMM14_DTYPE_F32) {
    schedule(plan, K, dev->sm_count, workspace, workspace_bytes, args, grid);
    if (plan.loader == 2)
      return finish(launch_sgemm_cpasync(args, grid, stream), "sgemm launch", stream);
    // A stored M x K: box 32 k x 128 m, 128-byte swizzle; stored K x M: box
    // 128 m x 32 k. B stored K x N: box 256 n x 32 k; stored N x K: box
    // 32 k x 256 n, 128-byte swizzle.
    CUtensorMap ma, mb;
    const CUtensorMapDataType f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    st = transa ? make_map(&ma, f32, 4, A, K, M, lda, SgemmShape::BM, SgemmShape::BK,
                           CU_TENSOR_MAP_SWIZZLE_NONE)
                : make_map(&ma, f32, 4, A, M, K, lda, SgemmShape::BK, SgemmShape::BM,
                           CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != GEMM14_OK) return st;
    st = transb ? make_map(&mb, f32, 4, B, N, K, ldb, SgemmShape::BK, SgemmShape::BN,
                           CU_TENSOR_MAP_SWIZZLE_128B)
                : make_map(&mb, f32, 4, B, K, N, ldb, SgemmShape::BN, SgemmShape::BK,
                           CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != GEMM14_OK) return st;
    return finish(launch_sgemm_tma(ma, mb, args, grid, stream), "sgemm launch", stream);
  }

  const bool bf16 = dtype == GEMM14_DTYPE_BF16;
  int pair_clusters = 0;
  if (plan.kernel == 3) {
    pair_clusters = pair_max_clusters();
    if (pair_clusters <= 0) {
      // clusters of two do not fit: the one-SM kernel computes the same product
      g_pair_enabled.store(0);
    }
  }
  if (plan.kernel == 3 && pair_clusters > 0) {
    CUtensorMap ma, mb, unused{};
    // each CTA of a pair loads 128 rows of A and 128 columns of B
    if ((st = make_maps_16(bf16, transa, transb, M, N, K, A, lda, B, ldb, 128, 128, &ma, &mb)) !=
        GEMM14_OK)
      return st;
    return run_pair(plan, args, ma, mb, unused, unused, pair_clusters, false,
                    idesc_f16_f32acc(bf16, PairShape::BM, PairShape::BN, transa != 0, transb == 0),
                    K, dev->sm_count, workspace, workspace_bytes, stream);
  }
  if (plan.kernel == 3)
    plan_for(dtype, transa, transb, M, N, K, A, lda, B, ldb, C, ldc, dev->sm_count, &plan);
  schedule(plan, K, dev->sm_count, workspace, workspace_bytes, args, grid);
  const uint32_t idesc = idesc_f16_f32acc(bf16, plan.bm, plan.bn, transa != 0, transb == 0);
  if (plan.loader != 1) {
    // software loader for A (loader 3), B (4) or both (2); TMA for the other
    const int soft = plan.loader == 3 ? 1 : plan.loader == 4 ? 2 : 3;
    CUtensorMap ma{}, mb{};
    if (soft != 3 &&
        (st = make_maps_16(bf16, transa, transb, M, N, K, A, lda, B, ldb, plan.bm, plan.bn,
                           soft == 1 ? nullptr : &ma, soft == 2 ? nullptr : &mb)) != GEMM14_OK)
      return st;
    return finish(launch_hgemm_tc_soft(plan.bm, plan.bn, soft, &ma, &mb, args, idesc, grid,
                                       stream),
                  "hgemm launch", stream);
  }
  CUtensorMap ma, mb, mc{};
  if ((st = make_maps_16(bf16, transa, transb, M, N, K, A, lda, B, ldb, plan.bm, plan.bn, &ma,
                         &mb)) != GEMM14_OK)
    return st;
  // C for the TMA-store epilogue of the plain variant (untransposed operands,
  // plain store, 16-byte-aligned C), as for the pair kernel: boxes of 32
  // columns x the rows one epilogue warp holds (bm / 4).
  // The variant is plain exactly when launch_hgemm_tc picks it.
  if (!args.transa && !args.transb && args.epi == kEpiStore && plan.vec_store &&
      (st = make_map(&mc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, args.C, args.M, args.N, args.ldc,
                     32, plan.bm / 4, CU_TENSOR_MAP_SWIZZLE_128B)) != GEMM14_OK)
    return st;
  return finish(launch_hgemm_tc(plan.bm, plan.bn, ma, mb, mc, args, idesc, grid, stream),
                "hgemm launch", stream);
}

int run_gemm(int dtype, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
             const void* B, int64_t ldb, float* C, int64_t ldc, void* workspace,
             size_t workspace_bytes, void* stream_ptr) {
  return run_gemm(dtype, 0, 0, M, N, K, 1.0f, A, lda, B, ldb, 0.0f, C, ldc, workspace,
                  workspace_bytes, stream_ptr);
}

}  // namespace

// ---- the internal interface of api_internal.h (for the host-buffer runtime)
int product_on_stream(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K,
                      float alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
                      float beta, float* C, int64_t ldc, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream) {
  return run_gemm(dtype, transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, workspace,
                  workspace_bytes, stream);
}

int validate_product(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K,
                     const void* A, int64_t lda, const void* B, int64_t ldb, const void* C,
                     int64_t ldc) {
  return validate(dtype, transa, transb, M, N, K, A, lda, B, ldb, C, ldc);
}

size_t product_workspace_bytes(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K,
                               const void* A, int64_t lda, const void* B, int64_t ldb,
                               const void* C, int64_t ldc) {
  const DeviceInfo* dev = nullptr;
  if (current_device(&dev) != GEMM14_OK) return 0;
  // TF32 and 3xTF32 also get room for their K-major copies and lo parts (the
  // pair kernel runs them several times faster than the converter kernel);
  // the other products take the stream-K region only
  if (is_tf32_mode(dtype)) {
    Repitch rp;
    plan_repitch(dtype, transa, transb, M, N, K, A, lda, B, ldb, C, ldc, dev->sm_count, &rp);
    if (rp.a || rp.b || rp.split) return rp.total;
  }
  gemm14_plan plan;
  plan_for(dtype, transa, transb, M, N, K, A, lda, B, ldb, C, ldc, dev->sm_count, &plan, true);
  return workspace_need(plan, dev->sm_count, K);
}

int operand_bytes(int dtype) { return elem_bytes_of(dtype); }

double schedule_efficiency(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K) {
  const DeviceInfo* dev = nullptr;
  if (current_device(&dev) != GEMM14_OK || M <= 0 || N <= 0 || K <= 0) return 1.0;
  // Dense operands with 16-byte pitches at a 4 KB-aligned notional address:
  // the plan of such device copies (only alignment and sizes enter it).
  const int eb = elem_bytes_of(dtype);
  const int64_t q = 16 / eb;
  const int64_t lda = ((transa ? M : K) + q - 1) / q * q, ldb = ((transb ? K : N) + q - 1) / q * q;
  const int64_t ldc = (N + 3) / 4 * 4;
  const void* base = reinterpret_cast<const void*>(uintptr_t(1) << 12);
  gemm14_plan plan;
  plan_for(dtype, transa, transb, M, N, K, base, lda, base, ldb, base, ldc, dev->sm_count, &plan,
           true);
  if (plan.tiles <= 0 || workspace_need(plan, dev->sm_count, K) > 0) return 1.0;
  const int64_t slots =
      plan.kernel == 3 || plan.kernel == 5 ? dev->sm_count / 2 : dev->sm_count;
  if (slots <= 0) return 1.0;
  const int64_t waves = (plan.tiles + slots - 1) / slots;
  return static_cast<double>(plan.tiles) / static_cast<double>(waves * slots);
}

int current_device_index(int* device) {
  const DeviceInfo* dev = nullptr;
  const int st = current_device(&dev);
  if (st != GEMM14_OK) return st;
  cudaError_t e = cudaGetDevice(device);
  if (e != cudaSuccess) {
    set_cuda_error("cudaGetDevice", e);
    return GEMM14_ERR_CUDA;
  }
  return GEMM14_OK;
}

// The status a device error word stands for: a failed bounds check (checked
// builds) first, then any other recorded failure (an expired wait).
int status_of_error_word(unsigned word) {
  if (word & kDevErrBounds) return GEMM14_ERR_DEVICE_CHECK;
  return word ? GEMM14_ERR_TIMEOUT : GEMM14_OK;
}

int take_device_error() {
  const DeviceInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st != GEMM14_OK) return st;
  unsigned word = 0;
  cudaError_t e;
  if ((e = cudaMemcpy(&word, dev->err_word, sizeof word, cudaMemcpyDeviceToHost)) != cudaSuccess ||
      (e = cudaMemset(dev->err_word, 0, sizeof word)) != cudaSuccess) {
    set_cuda_error("reading the device error word", e);
    return GEMM14_ERR_CUDA;
  }
  return status_of_error_word(word);
}

void note_cuda_error(const char* what, cudaError_t e) { set_cuda_error(what, e); }

}  // namespace gemm14

using namespace gemm14;

extern "C" {

int gemm_f32(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B,
             int64_t ldb, float* C, int64_t ldc, void* stream) {
  return run_gemm(GEMM14_DTYPE_F32, M, N, K, A, lda, B, ldb, C, ldc, nullptr, 0, stream);
}

int gemm_bf16_f32acc(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                     const void* B, int64_t ldb, float* C, int64_t ldc, void* stream) {
  return run_gemm(GEMM14_DTYPE_BF16, M, N, K, A, lda, B, ldb, C, ldc, nullptr, 0, stream);
}

int gemm_f16_f32acc(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                    int64_t ldb, float* C, int64_t ldc, void* stream) {
  return run_gemm(GEMM14_DTYPE_F16, M, N, K, A, lda, B, ldb, C, ldc, nullptr, 0, stream);
}

int gemm_f32_ws(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B,
                int64_t ldb, float* C, int64_t ldc, void* workspace, size_t workspace_bytes,
                void* stream) {
  return run_gemm(GEMM14_DTYPE_F32, M, N, K, A, lda, B, ldb, C, ldc, workspace, workspace_bytes,
                  stream);
}

int gemm_bf16_f32acc_ws(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                        const void* B, int64_t ldb, float* C, int64_t ldc, void* workspace,
                        size_t workspace_bytes, void* stream) {
  return run_gemm(GEMM14_DTYPE_BF16, M, N, K, A, lda, B, ldb, C, ldc, workspace,
                  workspace_bytes, stream);
}

int gemm_f16_f32acc_ws(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                       const void* B, int64_t ldb, float* C, int64_t ldc, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return run_gemm(GEMM14_DTYPE_F16, M, N, K, A, lda, B, ldb, C, ldc, workspace, workspace_bytes,
                  stream);
}

int gemm_tf32_f32acc(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                     const float* B, int64_t ldb, float* C, int64_t ldc, void* stream) {
  return run_gemm(GEMM14_DTYPE_TF32, M, N, K, A, lda, B, ldb, C, ldc, nullptr, 0, stream);
}

int gemm_f32_3xtf32(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                    const float* B, int64_t ldb, float* C, int64_t ldc, void* stream) {
  return run_gemm(GEMM14_DTYPE_F32_3XTF32, M, N, K, A, lda, B, ldb, C, ldc, nullptr, 0, stream);
}

int gemm14_gemm_ex(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K,
                   float alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
                   float beta, float* C, int64_t ldc, void* workspace, size_t workspace_bytes,
                   void* stream) {
  return run_gemm(dtype, transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, workspace,
                  workspace_bytes, stream);
}

size_t gemm14_workspace_bytes(int dtype, int64_t M, int64_t N, int64_t K, int sm_count) {
  if (sm_count <= 0) {
    const DeviceInfo* dev = nullptr;
    if (current_device(&dev) != GEMM14_OK) return 0;
    sm_count = dev->sm_count;
  }
  // Pointers only matter for the loader choice; assume TMA-addressable operands.
  const void* p = reinterpret_cast<const void*>(uintptr_t(1) << 16);
  const int64_t lda = ((K + 7) / 8) * 8, ldb = ((N + 7) / 8) * 8;
  if (validate(dtype, M, N, K, p, lda > 0 ? lda : 1, p, ldb > 0 ? ldb : 1, p,
               N > 0 ? ldb : 1) != GEMM14_OK)
    return 0;
  gemm14_plan plan;
  plan_for(dtype, M, N, K, p, lda, p, ldb, p, ldb, sm_count, &plan, true);
  return workspace_need(plan, sm_count, K);
}

size_t gemm14_workspace_bytes_ex(int dtype, int transa, int transb, int64_t M, int64_t N,
                                 int64_t K, const void* A, int64_t lda, const void* B,
                                 int64_t ldb, const void* C, int64_t ldc, int sm_count) {
  if (sm_count <= 0) {
    const DeviceInfo* dev = nullptr;
    if (current_device(&dev) != GEMM14_OK) return 0;
    sm_count = dev->sm_count;
  }
  if (validate(dtype, transa, transb, M, N, K, A, lda, B, ldb, C, ldc) != GEMM14_OK) return 0;
  if (M == 0 || N == 0 || K == 0) return 0;
  Repitch rp;
  plan_repitch(dtype, transa, transb, M, N, K, A, lda, B, ldb, C, ldc, sm_count, &rp);
  if (rp.a || rp.b || rp.split) return rp.total;
  gemm14_plan plan;
  plan_for(dtype, transa, transb, M, N, K, A, lda, B, ldb, C, ldc, sm_count, &plan, true);
  return workspace_need(plan, sm_count, K);
}

const char* gemm14_status_string(int status) {
  switch (status) {
    case GEMM14_OK: return "ok";
    case GEMM14_ERR_INVALID_ARG: return "invalid argument";
    case GEMM14_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case GEMM14_ERR_CUDA: return "CUDA error";
    case GEMM14_ERR_TIMEOUT: return "device-side wait timed out";
    case GEMM14_ERR_DEVICE_CHECK: return "device-side bounds check failed (access skipped)";
    default: return "unknown status";
  }
}

const char* gemm14_last_error_string(void) { return t_last_error; }

int gemm14_check_device_error(void* stream_ptr) {
  const DeviceInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st != GEMM14_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    set_cuda_error("cudaStreamSynchronize", e);
    return GEMM14_ERR_CUDA;
  }
  unsigned word = 0;
  if ((e = cudaMemcpy(&word, dev->err_word, sizeof word, cudaMemcpyDeviceToHost)) != cudaSuccess ||
      (e = cudaMemset(dev->err_word, 0, sizeof word)) != cudaSuccess) {
    set_cuda_error("reading the device error word", e);
    return GEMM14_ERR_CUDA;
  }
  return status_of_error_word(word);
}

int gemm14_plan_gemm(int dtype, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                     const void* B, int64_t ldb, const void* C, int64_t ldc, int sm_count,
                     gemm14_plan* plan) {
  if (!plan) return GEMM14_ERR_INVALID_ARG;
  int st = validate(dtype, M, N, K, A, lda, B, ldb, C, ldc);
  if (st != GEMM14_OK) return st;
  plan_for(dtype, M, N, K, A, lda, B, ldb, C, ldc, sm_count, plan);
  return GEMM14_OK;
}

int gemm14_plan_gemm_ex(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K,
                        const void* A, int64_t lda, const void* B, int64_t ldb, const void* C,
                        int64_t ldc, int sm_count, gemm14_plan* plan) {
  if (!plan) return GEMM14_ERR_INVALID_ARG;
  int st = validate(dtype, transa, transb, M, N, K, A, lda, B, ldb, C, ldc);
  if (st != GEMM14_OK) return st;
  plan_for(dtype, transa, transb, M, N, K, A, lda, B, ldb, C, ldc, sm_count, plan);
  return GEMM14_OK;
}

int gemm14_set_pair_kernel(int enable) {
  const int previous = g_pair_enabled.load();
  g_pair_enabled.store(enable ? 1 : 0);
  return previous;
}

int gemm14_debug_inject(int fault, uint64_t wait_limit_ns) {
  if (fault != kFaultNone && fault != kFaultSkipFirstStage) return GEMM14_ERR_INVALID_ARG;
  t_fault = fault;
  t_wait_limit_ns = wait_limit_ns;
  return GEMM14_OK;
}

int gemm14_version(void) { return 200; }

}  // extern "C"

// ----------------------------------------------------------------------------
// The entry point that allocates nothing.
//
// Some callers may not allocate device memory at all: code that runs inside a
// framework whose pool has reserved the GPU's memory up front and owns every
// allocation, plug-ins and embedded libraries that are not allowed to touch
// the allocator, and latency-critical paths that cannot afford the implicit
// device synchronisation of cudaMalloc / cudaFree. Such a caller cannot set
// up the workspace of gemm_bf16_f32acc_ws. gemm_bf16_f32acc_noalloc gives it
// the same product with the workspace taken from a fixed array that lives in
// the library itself (reserved on every GPU that loads the library, for as
// long as the process runs).
namespace gemm14 {
namespace {

// Capacity of the built-in scratch: the largest split either 16-bit kernel
// makes (flags + one 128 x 256 fp32 slot per SM: 19.9 MB on 152 SMs) fits on
// any GPU with up to 159 SMs. Operand copies (re-pitching) also land here
// when they fit beside the split's region.
constexpr size_t kNoAllocScratchBytes = size_t(20) << 20;  // 20 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocScratch {
  bool ready = false;
  unsigned char* ptr = nullptr;  // device address of g_noalloc_scratch
};
NoAllocScratch g_noalloc[kMaxDevices];
std::mutex g_noalloc_mutex;

// Device address of the scratch on the current device, looked up once per
// device (the symbol's host-side name is not a device address), with its
// flag words cleared on that first use, on the caller's stream.
int noalloc_scratch(int sm_count, cudaStream_t stream, unsigned char** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    set_cuda_error("cudaGetDevice", e);
    return GEMM14_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoAllocScratch& s = g_noalloc[dev];
  if (!s.ready) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess) {
      set_cuda_error("cudaGetSymbolAddress(no-alloc scratch)", e);
      return GEMM14_ERR_CUDA;
    }
    if ((e = cudaMemsetAsync(p, 0, streamk_flag_bytes(sm_count), stream)) != cudaSuccess) {
      set_cuda_error("cudaMemsetAsync(no-alloc scratch flags)", e);
      return GEMM14_ERR_CUDA;
    }
    s.ptr = static_cast<unsigned char*>(p);
    s.ready = true;
  }
  *out = s.ptr;
  return GEMM14_OK;
}

}  // namespace
}  // namespace gemm14

extern "C" int gemm_bf16_f32acc_noalloc(int64_t M, int64_t N, int64_t K, const void* A,
                                        int64_t lda, const void* B, int64_t ldb, float* C,
                                        int64_t ldc, void* stream_ptr) {
  int st = validate(GEMM14_DTYPE_BF16, M, N, K, A, lda, B, ldb, C, ldc);
  if (st != GEMM14_OK) return st;
  if (M == 0 || N == 0 || K == 0)  // nothing to split: the plain path
    return run_gemm(GEMM14_DTYPE_BF16, M, N, K, A, lda, B, ldb, C, ldc, nullptr, 0, stream_ptr);
  const DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev)) != GEMM14_OK) return st;
  gemm14_plan plan;
  plan_for(GEMM14_DTYPE_BF16, M, N, K, A, lda, B, ldb, C, ldc, dev->sm_count, &plan);
  const size_t need = workspace_need(plan, dev->sm_count, K);
  if (need > kNoAllocScratchBytes) {
    std::snprintf(t_last_error, sizeof t_last_error,
                  "gemm_bf16_f32acc_noalloc: this product's split needs %zu bytes of scratch, "
                  "more than the %zu bytes built into the library; gemm_bf16_f32acc computes it "
                  "unsplit without scratch, gemm_bf16_f32acc_ws with a caller workspace",
                  need, kNoAllocScratchBytes);
    return GEMM14_ERR_INVALID_ARG;
  }
  if (need == 0)
    return run_gemm(GEMM14_DTYPE_BF16, M, N, K, A, lda, B, ldb, C, ldc, nullptr, 0, stream_ptr);
  unsigned char* scratch = nullptr;
  if ((st = noalloc_scratch(dev->sm_count, static_cast<cudaStream_t>(stream_ptr), &scratch)) !=
      GEMM14_OK)
    return st;
  return run_gemm(GEMM14_DTYPE_BF16, M, N, K, A, lda, B, ldb, C, ldc, scratch,
                  kNoAllocScratchBytes, stream_ptr);
}
