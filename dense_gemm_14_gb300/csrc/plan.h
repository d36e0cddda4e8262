// plan.h -- the library's launch policy (plan.cu): which kernel, tile shape
// and loader a product takes, when its tiles are split over SMs (stream-K),
// and which of its operands are first copied into the caller's workspace.
// Host-only; nothing here crosses the library boundary.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>

#include "../../include/gemm14.h"

namespace gemm14 {

// Whether 16-bit products may use the CTA-pair kernel (gemm14_set_pair_kernel).
extern std::atomic<int> g_pair_enabled;

bool aligned(const void* p, uintptr_t a);
bool is_tf32_mode(int dtype);
int elem_bytes_of(int dtype);  // bytes of an element of A and B
int hgemm_bn_for(int64_t N);   // one-SM tensor-core tile width for N columns

// The plan (kernel, loader, tile, ring, grid) of a product on operands with
// these addresses and pitches on a GPU with sm_count SMs (no launch when M, N
// or K is 0). The pointers only enter through their alignment. split_ok: the
// call has a workspace for a stream-K split (an fp32 product of over 2^30
// FLOP then stays on the large kernel's tiles, which split over every SM,
// rather than taking the small-product kernel).
void plan_for(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K, const void* A,
              int64_t lda, const void* B, int64_t ldb, const void* C, int64_t ldc, int sm_count,
              gemm14_plan* p, bool split_ok = false);
void plan_for(int dtype, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
              const void* B, int64_t ldb, const void* C, int64_t ldc, int sm_count,
              gemm14_plan* p, bool split_ok = false);

// Stream-K policy: the workers a plan's tiles are split over (0: unsplit),
// the tile slots each worker keeps, and the workspace bytes that takes.
int slots_per_worker(const gemm14_plan& plan);
int pair_split_workers(int64_t tiles, int64_t L, int clusters);
int one_sm_split_workers(int kernel, int64_t tiles, int64_t L, int G);
// k_terms: 3 for the pair kernel's split-precision 3xTF32 run (3 L k-blocks).
size_t workspace_need(const gemm14_plan& plan, int sm_count, int64_t K, int k_terms = 1);

// Re-pitching into the caller's workspace. An operand whose base or row
// pitch is not a multiple of 16 bytes cannot be read by TMA; with a large
// enough workspace the call copies it there with a 16-byte pitch (a memory-
// bound pass of one read and one write per element) and runs the TMA loaders
// on the copy. Workspace layout: the stream-K region first (its flag words at
// the start, where they always are), then the copy of A, then that of B, then
// (3xTF32 split ahead of the call) lo(A) and lo(B).
struct Repitch {
  bool a = false, b = false;     // which operands are copied
  bool a_t = false, b_t = false; // ... transposed (tf32: into K-major storage)
  int transa = 0, transb = 0;    // the call's storage of op(A), op(B) after the copies
  int64_t lda = 0, ldb = 0;      // their pitches in the workspace
  size_t sk_bytes = 0;           // the stream-K region (flags + slots)
  size_t a_off = 0, b_off = 0;   // byte offsets of the copies
  // 3xTF32 on the pair kernel: lo(A) (M x K) and lo(B) (N x K), K-major with
  // pitch ld_lo, at a_lo_off and b_lo_off; A and B (copied or as stored) are
  // then K-major too and the product runs 3 terms (GemmArgs::k_terms)
  bool split = false;
  int64_t ld_lo = 0;
  size_t a_lo_off = 0, b_lo_off = 0;
  size_t total = 0;              // workspace bytes the call needs for all of it
};

size_t round256(size_t x);

// Fills *r for a call on `sms` SMs: which operands are copied (re-pitched or
// transposed) into the workspace, where, and the bytes that needs in all.
void plan_repitch(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K,
                  const void* A, int64_t lda, const void* B, int64_t ldb, const void* C,
                  int64_t ldc, int sms, Repitch* r);

}  // namespace gemm14
