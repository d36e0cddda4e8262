// copy.cu -- re-pitching an operand that TMA cannot address (a base or a
// row pitch that is not a multiple of 16 bytes) into a caller workspace with a
// 16-byte pitch, so that the product runs on the TMA loaders instead of the
// element-wise ones; and, for tf32 products, transposing an fp32 operand into
// the K-major storage the tensor cores read straight from TMA, and, for
// split-precision 3xTF32 products, writing the lo part of each element. A
// memory-bound pass: each element is read once and written once or twice. The work items are segments of kUnroll x 32 consecutive elements of a
// row; a warp loads a whole segment (its lanes on consecutive elements, so
// reads and writes are coalesced whatever the source alignment) before it
// stores any of it, keeping kUnroll loads per lane in flight.
#include "kernels.h"
#include "ptx.cuh"

namespace gemm14 {
namespace {

constexpr int kUnroll = 8;

template <typename T>
__global__ void __launch_bounds__(256) repitch_kernel(const RepitchJob j0, const RepitchJob j1) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t seg = 32 * kUnroll;
  const int64_t per_row0 = (j0.cols + seg - 1) / seg, per_row1 = (j1.cols + seg - 1) / seg;
  const int64_t items0 = j0.rows * per_row0;
  const int64_t items = items0 + j1.rows * per_row1;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t it = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       it < items; it += warps) {
    const bool first = it < items0;
    const RepitchJob& j = first ? j0 : j1;
    const int64_t per_row = first ? per_row0 : per_row1;
    const int64_t i = first ? it : it - items0;
    const int64_t r = i / per_row;
    const int64_t c0 = (i - r * per_row) * seg + lane;
    const T* s = static_cast<const T*>(j.src) + r * j.ld_src;
    T* d = static_cast<T*>(j.dst) + r * j.ld_dst;
    T v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c = c0 + 32 * u;
      v[u] = c < j.cols ? s[c] : T(0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c = c0 + 32 * u;
      if (c < j.cols) d[c] = v[u];
    }
  }
}

// Both jobs of a relayout: fp32 matrices copied, each transposed or not
// (job.transpose), in 64 x 64 tiles through shared memory: a tile is read
// along its source rows and written along its destination rows, so both
// sides stay coalesced, and each thread has its 16 loads in flight before
// the barrier. Element (r, c) of a transposed job's source lands at (c, r) of
// its destination. The tile's rows are padded to 65 floats, so the column
// reads of the transposed store hit 32 different banks. A job with dst_lo
// also writes lo(x) there, at the same place as x in dst (dst may be null).
constexpr int kRt = 64;

// lo(x) = x - hi(x), hi(x) = x with its 13 low fraction bits cleared, as the
// tensor cores read an fp32 operand of a kind::tf32 MMA. The subtraction is
// exact: hi(x) and x share sign and exponent, so the difference is x's 13
// low fraction bits, a value an fp32 holds exactly (also for subnormal x).
// lo(inf) is NaN (inf - inf): as on the converter kernel, a product term with
// an infinite input comes out NaN.
__device__ __forceinline__ float tf32_lo(float x) {
  return x - __uint_as_float(__float_as_uint(x) & 0xffffe000u);
}

__global__ void __launch_bounds__(256) relayout_kernel(const RepitchJob j0, const RepitchJob j1) {
  __shared__ float tile[kRt][kRt + 1];
  grid_dependency_wait();
  grid_launch_dependents();
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8 threads
  const int64_t tc0 = (j0.cols + kRt - 1) / kRt, tc1 = (j1.cols + kRt - 1) / kRt;
  const int64_t tiles0 = ((j0.rows + kRt - 1) / kRt) * tc0;
  const int64_t tiles = tiles0 + ((j1.rows + kRt - 1) / kRt) * tc1;
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const bool first = t < tiles0;
    const RepitchJob& j = first ? j0 : j1;
    const int64_t tcols = first ? tc0 : tc1;
    const int64_t i = first ? t : t - tiles0;
    const int64_t r0 = (i / tcols) * kRt, c0 = (i % tcols) * kRt;
    const float* src = static_cast<const float*>(j.src);
    float* dst = static_cast<float*>(j.dst);
    float* dst_lo = static_cast<float*>(j.dst_lo);
    float v[kRt / 8][2];
#pragma unroll
    for (int k = 0; k < kRt / 8; ++k)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t r = r0 + ty + 8 * k, c = c0 + tx + 32 * h;
        v[k][h] = r < j.rows && c < j.cols ? src[r * j.ld_src + c] : 0.0f;
      }
#pragma unroll
    for (int k = 0; k < kRt / 8; ++k)
#pragma unroll
      for (int h = 0; h < 2; ++h) tile[ty + 8 * k][tx + 32 * h] = v[k][h];
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kRt / 8; ++k)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (j.transpose) {
          // destination row c0 + ty + 8k, column r0 + tx + 32h
          const int64_t c = c0 + ty + 8 * k, r = r0 + tx + 32 * h;
          if (c < j.cols && r < j.rows) {
            const float x = tile[tx + 32 * h][ty + 8 * k];
            if (dst) dst[c * j.ld_dst + r] = x;
            if (dst_lo) dst_lo[c * j.ld_dst + r] = tf32_lo(x);
          }
        } else {
          const int64_t r = r0 + ty + 8 * k, c = c0 + tx + 32 * h;
          if (r < j.rows && c < j.cols) {
            const float x = tile[ty + 8 * k][tx + 32 * h];
            if (dst) dst[r * j.ld_dst + c] = x;
            if (dst_lo) dst_lo[r * j.ld_dst + c] = tf32_lo(x);
          }
        }
      }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_relayout(const RepitchJob& j0, const RepitchJob& j1, int sm_count,
                            cudaStream_t stream) {
  const int64_t tiles = ((j0.rows + kRt - 1) / kRt) * ((j0.cols + kRt - 1) / kRt) +
                        ((j1.rows + kRt - 1) / kRt) * ((j1.cols + kRt - 1) / kRt);
  if (tiles <= 0) return cudaSuccess;
  const int64_t cap = static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * 8;
  const dim3 grid(static_cast<unsigned>(tiles < cap ? tiles : cap));
  return launch_kernel(relayout_kernel, grid, dim3(256), 0, stream, j0, j1);
}

cudaError_t launch_repitch(const RepitchJob& j0, const RepitchJob& j1, int elem_bytes,
                           int sm_count, cudaStream_t stream) {
  // one segment per warp while there are fewer than 8 blocks an SM's worth
  const int64_t seg = 32 * kUnroll;
  const int64_t segments = (j0.cols > 0 ? j0.rows * ((j0.cols + seg - 1) / seg) : 0) +
                           (j1.cols > 0 ? j1.rows * ((j1.cols + seg - 1) / seg) : 0);
  if (segments <= 0) return cudaSuccess;
  const int64_t blocks = (segments + 7) / 8;  // 8 warps a block
  const int64_t cap = static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * 8;
  const dim3 grid(static_cast<unsigned>(blocks < cap ? blocks : cap));
  if (elem_bytes == 4)
    return launch_kernel(repitch_kernel<uint32_t>, grid, dim3(256), 0, stream, j0, j1);
  return launch_kernel(repitch_kernel<uint16_t>, grid, dim3(256), 0, stream, j0, j1);
}

}  // namespace gemm14
