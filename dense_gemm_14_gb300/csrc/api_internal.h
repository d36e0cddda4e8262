// api_internal.h -- what the host-buffer runtime (host_path.cu) uses of the
// C-ABI layer (api.cu). Nothing here crosses the library boundary.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace gemm14 {

// gemm14_gemm_ex on `stream` with device pointers (its own checks included).
int product_on_stream(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K,
                      float alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
                      float beta, float* C, int64_t ldc, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream);

// The argument checks of gemm14_gemm_ex; the pointers may be host pointers.
int validate_product(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K,
                     const void* A, int64_t lda, const void* B, int64_t ldb, const void* C,
                     int64_t ldc);

// Workspace bytes with which such a call on these device operands would use
// the stream-K schedule on the current device (0: it would not split); for
// TF32 and 3xTF32 also the room for their K-major copies and lo parts.
size_t product_workspace_bytes(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K,
                               const void* A, int64_t lda, const void* B, int64_t ldb,
                               const void* C, int64_t ldc);

// Bytes per element of A and B for a gemm14_dtype (4 or 2).
int operand_bytes(int dtype);

// Share of the worker slots kept busy by such a call on the current device,
// with dense device operands (pitches rounded to 16 bytes) and a workspace:
// 1 when it runs the stream-K schedule, else tiles / (waves x workers).
double schedule_efficiency(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K);

// The current device's index, checked as by every entry point (a gemm14_status).
int current_device_index(int* device);

// Reads and clears the current device's error word once its kernels are
// known to be done: GEMM14_OK, GEMM14_ERR_TIMEOUT or GEMM14_ERR_CUDA.
int take_device_error();

// Records a CUDA failure as this thread's last error text.
void note_cuda_error(const char* what, cudaError_t e);

}  // namespace gemm14
