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
// sides stay coalesced. A thread moves 4 x 4 consecutive elements of a row
// (one 16-byte load or store each where the job's base and pitch allow it,
// else 4-byte ones), all 4 loads in flight before the barrier. Element (r, c)
// of a transposed job's source lands at (c, r) of its destination. The
// tile's rows are padded to 65 floats (the column reads of the transposed
// store see at most 2-way bank conflicts). A job with dst_lo also writes
// lo(x) there, at the same place as x in dst (dst may be null). One CTA a
// tile, up to 256 an SM: the block scheduler balances the last tiles.
// Measured against 4-byte accesses and 8 CTAs an SM looping over tiles: TF32
// 3072^3 with B transposed first 80.8 -> 77.8 us, 8192^3 1366 -> 1328 us,
// fp32 3072^3 with A transposed first 905.1 -> 902.7 us.
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

// Up to 4 consecutive elements of a destination row (n of them inside it),
// and their lo parts: one 16-byte store each when `vec` and all 4 are inside.
__device__ __forceinline__ void put4(float* dst, float* dst_lo, int64_t off, float4 w, int64_t n,
                                     bool vec) {
  if (vec && n >= 4) {
    if (dst) *reinterpret_cast<float4*>(dst + off) = w;
    if (dst_lo)
      *reinterpret_cast<float4*>(dst_lo + off) =
          make_float4(tf32_lo(w.x), tf32_lo(w.y), tf32_lo(w.z), tf32_lo(w.w));
    return;
  }
  const float e[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int u = 0; u < 4; ++u)
    if (u < n) {
      if (dst) dst[off + u] = e[u];
      if (dst_lo) dst_lo[off + u] = tf32_lo(e[u]);
    }
}

__device__ __forceinline__ bool al16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15) == 0;
}

__global__ void __launch_bounds__(256) relayout_kernel(const RepitchJob j0, const RepitchJob j1) {
  __shared__ float tile[kRt][kRt + 1];
  grid_dependency_wait();
  grid_launch_dependents();
  const int q = threadIdx.x & 15, g = threadIdx.x >> 4;  // float4 column q, row group g
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
    // 16-byte accesses where the job's base and pitch allow them
    const bool vload = al16(src) && (j.ld_src & 3) == 0;
    const bool vstore = (!dst || al16(dst)) && (!dst_lo || al16(dst_lo)) && (j.ld_dst & 3) == 0;
    // tile rows g + 16k, columns 4q .. 4q+3: a half-warp reads 256 contiguous bytes
    float4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t r = r0 + g + 16 * k, c = c0 + 4 * q;
      if (r < j.rows && vload && c + 3 < j.cols) {
        v[k] = *reinterpret_cast<const float4*>(src + r * j.ld_src + c);
      } else {
        const bool in = r < j.rows;
        const float* s = src + r * j.ld_src;
        v[k].x = in && c < j.cols ? s[c] : 0.0f;
        v[k].y = in && c + 1 < j.cols ? s[c + 1] : 0.0f;
        v[k].z = in && c + 2 < j.cols ? s[c + 2] : 0.0f;
        v[k].w = in && c + 3 < j.cols ? s[c + 3] : 0.0f;
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float* row = tile[g + 16 * k] + 4 * q;
      row[0] = v[k].x;
      row[1] = v[k].y;
      row[2] = v[k].z;
      row[3] = v[k].w;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (j.transpose) {
        // destination row c0 + g + 16k (a source column), columns r0 + 4q .. +3
        const int64_t c = c0 + g + 16 * k, r = r0 + 4 * q;
        if (c < j.cols && r < j.rows) {
          const int tcn = g + 16 * k;
          const float4 w = make_float4(tile[4 * q][tcn], tile[4 * q + 1][tcn],
                                       tile[4 * q + 2][tcn], tile[4 * q + 3][tcn]);
          put4(dst, dst_lo, c * j.ld_dst + r, w, j.rows - r, vstore);
        }
      } else {
        const int64_t r = r0 + g + 16 * k, c = c0 + 4 * q;
        if (r < j.rows && c < j.cols) {
          const float* row = tile[g + 16 * k] + 4 * q;
          put4(dst, dst_lo, r * j.ld_dst + c, make_float4(row[0], row[1], row[2], row[3]),
               j.cols - c, vstore);
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
  const int64_t cap = static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * 256;
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
