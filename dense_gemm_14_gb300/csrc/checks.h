// checks.h -- the predicates of the device-side bounds checks. A build with
// -DGEMM14_DEVICE_CHECKS (python -m dense_gemm_14_gb300.build --checked)
// tests every plain global store of C and every stream-K slot and flag access
// against them before it happens. A failed check records kDevErrBounds in the
// call's device error word (gemm14_check_device_error then returns
// GEMM14_ERR_DEVICE_CHECK) and skips the access, so that an index the
// kernel's arithmetic got wrong never reaches memory outside its buffer. TMA
// copies need no check: the tensor map bounds them in hardware. The product
// build compiles every check to the constant true.
//
// Plain C++ with no CUDA dependency, so that the host tests compile and check
// the predicates themselves.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define GEMM14_HD __host__ __device__
#else
#define GEMM14_HD
#endif

namespace gemm14 {

// `width` consecutive fp32 elements starting `off` elements past C's first
// element lie inside C's row-major M x N block of row pitch ldc (none of
// them in a row's padding, before C or past its last row).
GEMM14_HD inline bool c_span_ok(int64_t off, int64_t ldc, int64_t M, int64_t N, int width) {
  if (off < 0 || ldc <= 0 || width <= 0 || N > ldc) return false;
  const int64_t row = off / ldc;
  const int64_t col = off - row * ldc;
  return row < M && col + width <= N;
}

// `width` consecutive fp32 elements starting `off` elements into a stream-K
// slot region of n_slots slots of slot_elems elements each lie inside slot
// `slot` (a worker's partial sums never spill into another worker's slot).
GEMM14_HD inline bool slot_span_ok(int64_t off, int64_t slot, int64_t slot_elems,
                                   int64_t n_slots, int width) {
  if (slot < 0 || slot >= n_slots || slot_elems <= 0 || width <= 0) return false;
  return off >= slot * slot_elems && off + width <= (slot + 1) * slot_elems;
}

// Index i of an array of n entries (the stream-K flags).
GEMM14_HD inline bool index_ok(int64_t i, int64_t n) { return i >= 0 && i < n; }

// The device error word's bit for a failed check.
constexpr unsigned kDevErrBounds = 4u;

#if defined(__CUDACC__)
// With GEMM14_DEVICE_CHECKS a false `ok` records kDevErrBounds in *err and the
// caller skips the access; otherwise every check is true and its predicate,
// free of side effects, is dropped.
#ifdef GEMM14_DEVICE_CHECKS
__device__ __forceinline__ bool dev_check(bool ok, unsigned* err) {
  if (!ok) atomicOr(err, kDevErrBounds);
  return ok;
}
#else
__device__ __forceinline__ bool dev_check(bool, unsigned*) { return true; }
#endif
#endif

}  // namespace gemm14
