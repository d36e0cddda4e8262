/*
 * gemm14.h -- C ABI of the GB300 (sm_103a) dense GEMM library libgemm14.so.
 *
 * Operation (all entry points): C = A * B with
 *     C[i][j] = sum_{k < K} A[i][k] * B[k][j],   0 <= i < M, 0 <= j < N,
 * the matrix product of gpu-hpc-book ch.06 "高级 cuda 特性 —— 从矩阵乘法(gemm)说起"
 * (Advanced CUDA features, starting from GEMM; opening section and
 * "缓存缺失与带宽约束分析" item (4)) and of "Kernel 优化指南" (cuda-kernel-academy
 * module 02), "GEMM 优化路径", Level 1, whose kernels take (M, N, K) and
 * row-major pointers; this interface adds leading dimensions and a stream.
 *
 * Layout: A, B and C are row-major. Element (i, k) of A is A[i * lda + k];
 * (k, j) of B is B[k * ldb + j]; (i, j) of C is C[i * ldc + j]. Leading
 * dimensions are counted in elements: lda >= K, ldb >= N, ldc >= N (each at
 * least 1). C is overwritten (alpha, beta and stored transposes: see
 * gemm14_gemm_ex); A and B are only read. C must not overlap A or B.
 * Reads of A and B stay inside each one's storage span, from its first
 * element to the last element of its last row; the 16-bit software loader
 * (operands TMA cannot address) may read padding elements between rows inside
 * that span, whose values it does not use.
 *
 * Pointers are DEVICE pointers in the current CUDA device's address space
 * (e.g. torch CUDA tensors' data_ptr()). `stream` is a cudaStream_t (NULL =
 * legacy default stream). Calls are asynchronous: the work is enqueued on
 * `stream` and the function returns without synchronising. The caller owns
 * every buffer; the library allocates and frees no device memory and keeps no
 * pointer after it returns.
 *
 * Degenerate sizes: M == 0 or N == 0 returns GEMM14_OK and launches nothing;
 * K == 0 sets the M x N block of C to zero (the empty sum).
 *
 * Errors: every entry point returns a gemm14_status and never aborts, prints
 * or exits. Invalid arguments are detected on the host before any CUDA call.
 * A device-side failure (a bounded wait inside a kernel that expired) is
 * recorded in a device error word and reported by gemm14_check_device_error.
 *
 * Only compute capability 10.3 (GB300) is supported; any other device gives
 * GEMM14_ERR_UNSUPPORTED_DEVICE. Sizes up to 2^31 - 1 per dimension.
 * Thread safety: all entry points are reentrant.
 */
#ifndef GEMM14_H
#define GEMM14_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gemm14_status {
  GEMM14_OK = 0,
  GEMM14_ERR_INVALID_ARG = 1,        /* negative or too large size, ld too small, NULL
                                        pointer with a non-empty extent, misaligned
                                        element pointer, bad dtype */
  GEMM14_ERR_UNSUPPORTED_DEVICE = 2, /* no CUDA device, or it is not compute capability 10.3 */
  GEMM14_ERR_CUDA = 3,               /* a CUDA runtime/driver call failed; see
                                        gemm14_last_error_string() */
  GEMM14_ERR_TIMEOUT = 4,            /* a kernel's bounded wait expired (device-side) */
  GEMM14_ERR_DEVICE_CHECK = 5        /* a device-side bounds check failed and its access was
                                        skipped (only a library built with
                                        GEMM14_DEVICE_CHECKS runs these checks) */
} gemm14_status;

/*
 * Element types and arithmetic, for gemm14_gemm_ex and the planning queries:
 *   F32        fp32 inputs, fp32 FMAs on the CUDA cores (gemm_f32);
 *   BF16, F16  16-bit inputs, fp32 accumulation on the tensor cores;
 *   TF32       fp32 inputs rounded to tf32 on the tensor cores (gemm_tf32_f32acc);
 *   F32_3XTF32 fp32 inputs, split tf32 arithmetic on the tensor cores that
 *              meets the fp32 bound (gemm_f32_3xtf32).
 */
enum {
  GEMM14_DTYPE_F32 = 0,
  GEMM14_DTYPE_BF16 = 1,
  GEMM14_DTYPE_F16 = 2,
  GEMM14_DTYPE_TF32 = 3,
  GEMM14_DTYPE_F32_3XTF32 = 4
};

/*
 * fp32 inputs, fp32 FFMA accumulation on the CUDA cores, fp32 output.
 * A, B, C: 4-byte aligned. The fast loader (TMA) is used when A and B are
 * 16-byte aligned and lda, ldb are multiples of 4; otherwise an equivalent
 * cp.async loader is used (same results). 16-byte stores are used for C when
 * C is 16-byte aligned and ldc is a multiple of 4.
 * A product whose 128 x 256 output tiles would fill at most half the SMs runs
 * on 64 x 64 tiles instead, the k range of each tile split over a cluster of
 * up to 8 CTAs and added up in a fixed order on chip (no workspace): its last
 * bits may differ from the large tiles' (another summation order), within the
 * same bound, and are the same with or without a workspace.
 * Follows the register-tiled, shared-memory-tiled kernels of gpu-hpc-book
 * ch.06, "矩阵乘法中的分块与数据复用" (Shared Memory Tiling, Register Tiling).
 */
int gemm_f32(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B,
             int64_t ldb, float* C, int64_t ldc, void* stream);

/*
 * bf16 inputs (raw bfloat16 bit patterns), fp32 accumulation on the tensor
 * cores (tcgen05), fp32 output. Inputs are rounded to bf16 by the caller.
 * A, B: 2-byte aligned; C: 4-byte aligned. The fast loader (TMA) reads each
 * operand that is 16-byte aligned with a leading dimension that is a multiple
 * of 8; a software loader fills the same shared-memory tiles for the other
 * operand(s) (same results, slower).
 * The tensor-core path of "Kernel 优化指南", "Level 4: Tensor Cores (WMMA)"
 * (half-precision inputs, float accumulator), and of gpu-hpc-book ch.06,
 * "Tensor Cores".
 */
int gemm_bf16_f32acc(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                     const void* B, int64_t ldb, float* C, int64_t ldc, void* stream);

/* As gemm_bf16_f32acc with IEEE binary16 (fp16) inputs. */
int gemm_f16_f32acc(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                    int64_t ldb, float* C, int64_t ldc, void* stream);

/*
 * fp32 inputs on the tensor cores (tcgen05 kind::tf32, fp32 accumulation in
 * tensor memory), fp32 output. TF32 is the pages' tensor-core format for fp32
 * data (gpu-hpc-book ch.06, "Tensor Cores": fp32's 8 exponent bits, 10
 * fraction bits).
 *   gemm_tf32_f32acc: every input is read as tf32 the way the tensor cores
 *     read an fp32 operand, tf32(x) = x with its 13 low fraction bits
 *     cleared (truncation toward zero), and the products of those values are
 *     summed in fp32: against the truncated inputs, the fp32 bound; against
 *     the fp32 inputs |C - A B| <= 4e-3 (|A||B|) element-wise.
 *   gemm_f32_3xtf32: each input x is split into hi = tf32(x) and lo = x - hi
 *     (exact), and C = hi(A) hi(B) + hi(A) lo(B) + lo(A) hi(B) summed in fp32
 *     (the split-precision scheme known as 3xTF32): within the fp32 bound,
 *     |C - A B| <= 1e-5 (|A||B|), at tensor-core speed. Through
 *     gemm14_gemm_ex with a workspace of gemm14_workspace_bytes_ex bytes, lo(A)
 *     and lo(B) are first written into the workspace (with K-major copies of
 *     operands stored otherwise) and the product runs as three k sums, lo(A)
 *     hi(B), hi(A) lo(B), hi(A) hi(B), on CTA pairs: the same bound, other
 *     bits (another order of the same terms).
 * Arguments, layout and rules as gemm_f32. A and B 16-byte aligned with lda,
 * ldb multiples of 4 run on CTA pairs of tensor-core SMs (256 x 256 tiles);
 * other operands run on gemm_f32's kernel, whose exact fp32 products meet both
 * bounds. Infinite inputs give NaN where a product would be infinite (lo =
 * inf - inf), and a NaN whose payload lies only in the 13 low fraction bits
 * is read as an infinity; finite inputs whose products overflow behave as in
 * gemm_f32.
 */
int gemm_tf32_f32acc(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                     const float* B, int64_t ldb, float* C, int64_t ldc, void* stream);
int gemm_f32_3xtf32(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                    const float* B, int64_t ldb, float* C, int64_t ldc, void* stream);

/*
 * Stream-K variants. Same operation and arguments as gemm_f32 /
 * gemm_bf16_f32acc / gemm_f16_f32acc, plus a caller-owned DEVICE workspace.
 * With a workspace of at least gemm14_workspace_bytes(...) bytes, the one-SM
 * kernels split the k-blocks of the last wave and a half of output tiles
 * evenly over all SMs instead of leaving SMs idle in a partial last wave, or,
 * for products of fewer tiles than half the SMs, spread all their k-blocks
 * over the SMs (16-bit tiles over at most 4 SMs each, with 16 or more
 * k-blocks apiece) (the "stream-K" schedule): a tile shared by several SMs is finished by the
 * SM holding its first k-blocks, which adds the others' partial sums from the
 * workspace in a fixed order, so results are deterministic run to run (they
 * may differ in the last bits from the data-parallel schedule, which sums a
 * tile's k-blocks in one run). With workspace == NULL, a smaller workspace, a
 * product whose tiles fill whole waves, or one with between half and all of
 * a wave of tiles (where splitting measured slower), the call is exactly the
 * plain entry point. The CTA-pair kernel (wide 16-bit products) splits in the
 * same way with a cluster of two SMs as the worker.
 * workspace: 16-byte aligned (else GEMM14_ERR_INVALID_ARG), zero-filled
 * before its first use. Its first bytes (one 4-byte word per SM, rounded up
 * to 256 bytes) hold publication flags that only ever contain zero or the
 * number of a finished call, so a workspace may be reused by any later call,
 * of any shape, without clearing; it must not be used by two calls that may
 * run at the same time. Each flag is cleared by the one tile owner that waits
 * for it, so a call captured in a CUDA graph (its number fixed at capture) may
 * be replayed any number of times.
 * Re-pitching: an operand TMA cannot read (base or row pitch not a multiple
 * of 16 bytes) is first copied into the workspace with a 16-byte pitch when
 * the workspace has gemm14_workspace_bytes_ex(...) bytes for this call's
 * operands; the product then runs on the TMA loaders (the same kernels, and
 * the same bits, as for aligned operands). The copies lie after the stream-K
 * region, never over the flag words. With less room the call reads such an
 * operand as it is, with the element-wise loaders.
 */
int gemm_f32_ws(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B,
                int64_t ldb, float* C, int64_t ldc, void* workspace, size_t workspace_bytes,
                void* stream);
int gemm_bf16_f32acc_ws(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                        const void* B, int64_t ldb, float* C, int64_t ldc, void* workspace,
                        size_t workspace_bytes, void* stream);
int gemm_f16_f32acc_ws(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                       const void* B, int64_t ldb, float* C, int64_t ldc, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * gemm_bf16_f32acc without any device allocation by the caller or the
 * library. The pages have no counterpart to this entry point; it exists for
 * callers that may not allocate device memory: code inside a framework whose
 * memory pool has reserved the GPU and owns every allocation, plug-ins that
 * must not touch the allocator, and latency-critical paths that cannot take
 * the implicit device synchronisation of cudaMalloc / cudaFree. The caller
 * passes A, B and C exactly as for gemm_bf16_f32acc; the stream-K scratch
 * that gemm_bf16_f32acc_ws would take from the caller comes instead from a
 * 20 MiB array built into the library, which every GPU that loads the library
 * holds until the process exits. Operands that TMA cannot read are re-pitched
 * into the same array when they fit beside the split's region, as the
 * workspace entry points do with theirs. It calls no cudaMalloc, cudaFree or
 * other allocating routine.
 * Limit: a product whose split needs more than the 20 MiB returns
 * GEMM14_ERR_INVALID_ARG, and gemm14_last_error_string() says how many bytes
 * were needed (gemm_bf16_f32acc then computes it unsplit, with no scratch).
 * The largest split is one 128 x 256 fp32 slot per SM plus a flag word each,
 * so this happens only on GPUs with more than 159 SMs; on 152 SMs every
 * product runs, split exactly as gemm_bf16_f32acc_ws would split it.
 * Products that need no scratch run as gemm_bf16_f32acc.
 * Set-up: the first call on each device looks up the array's device address
 * and clears its flag words on the caller's stream; make that first call
 * before any stream capture. Every call shares the one array, which keeps the
 * last call's contents (only its flag words must start at zero, and calls
 * leave them holding finished calls' numbers): calls that may overlap on the
 * GPU race with each other and must not be issued.
 */
int gemm_bf16_f32acc_noalloc(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                             const void* B, int64_t ldb, float* C, int64_t ldc, void* stream);

/*
 * The extended product, for every element type and arithmetic (dtype =
 * GEMM14_DTYPE_*):
 *     C = alpha * op(A) * op(B) + beta * C,
 * op(A) an M x K matrix and op(B) a K x N matrix. It generalises the
 * accumulate form of the pages' asynchronous tensor-core MMA (gpu-hpc-book
 * ch.06 "高级 cuda 特性 —— 从矩阵乘法(gemm)说起", "Tensor Cores" / "wgmma":
 * D = A * B + D with either operand optionally transposed and D scaled by
 * 0 or 1) to any fp32 alpha and beta.
 * Storage (row-major throughout):
 *   transa = 0: A is stored M x K, op(A)[i][k] = A[i * lda + k], lda >= K;
 *   transa = 1: A is stored K x M, op(A)[i][k] = A[k * lda + i], lda >= M;
 *   transb = 0: B is stored K x N, op(B)[k][j] = B[k * ldb + j], ldb >= N;
 *   transb = 1: B is stored N x K, op(B)[k][j] = B[j * ldb + k], ldb >= K;
 *   C is M x N, C[i * ldc + j], ldc >= N. Any other transa / transb value is
 *   GEMM14_ERR_INVALID_ARG.
 * Arithmetic: the sum over k is formed exactly as by gemm_f32 /
 * gemm_bf16_f32acc / gemm_f16_f32acc (bit-identical for alpha = 1,
 * beta = 0, with the same workspace; 3xTF32 with a workspace sums its terms
 * in another order, see gemm_f32_3xtf32); then each element is written as
 * alpha * sum (beta == 0) or as fmaf(alpha, sum, beta * C) in fp32.
 * beta == 0: C is not read (NaN or infinity in C does not propagate).
 * K == 0 or alpha == 0: A and B are not read; C becomes beta * C (beta == 1
 * launches nothing, beta == 0 zeroes C).
 * Loaders: operands take TMA under the same alignment rules as the plain
 * entry points (16-byte aligned, pitches multiples of 16 bytes) in either
 * storage, and the equivalent software loader otherwise.
 * workspace / workspace_bytes: as for the *_ws calls (NULL, 0 allowed),
 * re-pitching included; gemm14_workspace_bytes_ex gives the bytes for these
 * operands (for TMA-addressable ones it equals gemm14_workspace_bytes(dtype,
 * M, N, K, ...), which does not depend on transa / transb).
 * Other rules (device pointers, stream, errors, degenerate sizes) as above.
 */
int gemm14_gemm_ex(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K,
                   float alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
                   float beta, float* C, int64_t ldc, void* workspace, size_t workspace_bytes,
                   void* stream);

/*
 * Workspace bytes that let the *_ws call of this dtype and shape use the
 * stream-K schedule on a GPU with sm_count SMs (sm_count <= 0: the current
 * device's). 0 means the call would not split tiles (whole waves, or
 * between half and one wave of tiles) or the arguments are invalid. Assumes operands
 * TMA can address (16-byte aligned, pitches multiple of 16 bytes).
 */
size_t gemm14_workspace_bytes(int dtype, int64_t M, int64_t N, int64_t K, int sm_count);

/*
 * Workspace bytes for a gemm14_gemm_ex (or *_ws) call on exactly these
 * operands: the stream-K region as above, plus, for an operand TMA cannot
 * read, room for its copy with a 16-byte pitch (so that the call re-pitches
 * it); for TF32 and 3xTF32, room for K-major copies of operands stored
 * otherwise, and for 3xTF32 room for lo(A) and lo(B). Pointers are only inspected for their alignment, never dereferenced;
 * no CUDA call is made when sm_count > 0. 0: the call needs no workspace, or
 * the arguments are invalid.
 */
size_t gemm14_workspace_bytes_ex(int dtype, int transa, int transb, int64_t M, int64_t N,
                                 int64_t K, const void* A, int64_t lda, const void* B,
                                 int64_t ldb, const void* C, int64_t ldc, int sm_count);

/* Static text for a status code (never NULL). */
const char* gemm14_status_string(int status);

/* Text of the last CUDA failure seen by this thread ("" if none). */
const char* gemm14_last_error_string(void);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word. Returns GEMM14_ERR_DEVICE_CHECK if a kernel of a checked build
 * skipped an access its bounds checks rejected since the last check, else
 * GEMM14_ERR_TIMEOUT if a kernel recorded an expired wait,
 * GEMM14_ERR_CUDA if the synchronisation failed, else OK.
 */
int gemm14_check_device_error(void* stream);

/*
 * Host-buffer product: C = alpha * op(A) op(B) + beta * C, as gemm14_gemm_ex,
 * with A, B and C in HOST memory, computed on the current device. The library
 * copies the operands in, runs the product and copies C back, on three
 * streams of its own (copies in, kernels, copies out), with device buffers
 * from a memory pool of its own. This call is the exception to the rules
 * above on pointers, ownership and allocation.
 *
 * Pipelining: op(A) is sent in `panels` row panels (0: the library's choice;
 * stored K x M A, transa = 1: one panel), after all of B; panel p is computed
 * once it is in and copied out once computed, while panel p + 1 goes in.
 * Consecutive calls pipeline in the same way: a call's operands go in while
 * earlier calls compute and copy out.
 *
 * Asynchrony: the call enqueues the work and returns; *ticket (not NULL)
 * names it for gemm14_host_wait. Until that wait returns, the caller must not
 * change A, B or C, nor read C. Pinned host memory (cudaHostAlloc, or pinned
 * torch tensors) gives asynchronous copies at the link's rate; pageable
 * memory works but CUDA stages its copies through pinned buffers.
 *
 * Ordering: a call whose A, B (or C when beta != 0) overlaps the C of a call
 * still in flight waits, on the device, for that call's C to be back in host
 * memory. Calls are otherwise ordered only by their streams: products run in
 * call order, and copies out finish in call order.
 *
 * Errors: invalid arguments (as gemm14_gemm_ex, with NULL host pointers where
 * they are read) are reported before anything is enqueued, with *ticket
 * untouched. Transfer or launch failures give GEMM14_ERR_CUDA. Degenerate
 * sizes enqueue nothing (M == 0 or N == 0; beta == 1 with K == 0 or
 * alpha == 0) and still return a ticket.
 * Memory: the pool keeps its buffers for reuse for the life of the process.
 */
int gemm14_gemm_host(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K,
                     float alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
                     float beta, float* C, int64_t ldc, int panels, uint64_t* ticket);

/*
 * Blocks until the call named by `ticket` has its C in host memory. Returns
 * GEMM14_OK, GEMM14_ERR_TIMEOUT if a kernel of the device recorded an expired
 * wait (the device error word, read and cleared as by
 * gemm14_check_device_error), GEMM14_ERR_CUDA if the work failed, or
 * GEMM14_ERR_INVALID_ARG for a ticket never issued. A ticket already waited
 * for returns GEMM14_OK at once.
 */
int gemm14_host_wait(uint64_t ticket);

/* Waits for every host-buffer call in flight (on every device), as gemm14_host_wait. */
int gemm14_host_synchronize(void);

/* Launch plan chosen for a call (host-side only; no CUDA call is made). */
typedef struct gemm14_plan {
  int kernel;     /* 1 = fp32 SIMT (FFMA), 2 = tcgen05 on one SM per tile,
                     3 = tcgen05 on CTA pairs (two SMs per 256 x 256 tile),
                     4 = tcgen05 kind::tf32 on CTA pairs (TF32 / 3xTF32),
                     5 = kernel 3 with kind::tf32 MMAs (TF32, A stored M x K and B
                         stored N x K: both read as stored),
                     6 = fp32 FFMA on 64 x 64 tiles, the k range of each tile split
                         over a cluster of grid / tiles CTAs (products whose
                         128 x 256 tiles would fill at most half the SMs; with a
                         workspace, only those of at most 2^30 FLOP),
                     0 = no launch */
  int loader;     /* 1 = TMA (kernel 6: 16-byte cp.async), 2 = software loader
                     (cp.async for fp32; kernel 6: 4-byte cp.async); kernel 2
                     only: 3 = software loader for A and TMA for B, 4 = TMA for
                     A and software loader for B; 0 = none */
  int bm, bn, bk; /* output tile rows x columns, k-block depth */
  int stages;     /* shared-memory ring depth (kernel 4: operand stages the converter
                     warps fill, 4 for TF32 and 2 for 3xTF32) */
  int threads;    /* threads per CTA */
  int smem_bytes; /* dynamic shared memory per CTA */
  int vec_store;  /* 1 if C takes 16-byte stores */
  int64_t tiles;  /* output tiles */
  int grid;       /* CTAs launched (persistent: min(tiles, sm_count); for kernel 3,
                     2 x min(tiles, sm_count / 2); for kernel 6, tiles x the
                     cluster size) */
} gemm14_plan;

/*
 * Fills *plan with what the matching gemm_* call would launch on a GPU with
 * `sm_count` SMs. Validates arguments exactly like the entry points (pointers
 * are only inspected for NULL and alignment, never dereferenced). Returns a
 * gemm14_status; makes no CUDA call.
 */
int gemm14_plan_gemm(int dtype, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                     const void* B, int64_t ldb, const void* C, int64_t ldc, int sm_count,
                     gemm14_plan* plan);

/* As gemm14_plan_gemm for a gemm14_gemm_ex call with these transposes. */
int gemm14_plan_gemm_ex(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K,
                        const void* A, int64_t lda, const void* B, int64_t ldb, const void* C,
                        int64_t ldc, int sm_count, gemm14_plan* plan);

/*
 * The 16-bit entry points compute 256 x 256 output tiles on pairs of SMs
 * (a cluster of two CTAs sharing each tile's B operand) when the operands are
 * TMA-addressable and M, N > 128; otherwise tiles on one SM, of 128 rows, or
 * of 64 rows when the 128-row tiles would be fewer than the SMs. The kernels
 * accumulate in the same order and give bit-identical results.
 * gemm14_set_pair_kernel(0) restricts all later calls in the process to the
 * one-SM kernel, (1) allows pairs again (the default); returns the previous
 * setting. If pairs cannot be launched on the device the library falls back
 * to the one-SM kernel by itself.
 */
int gemm14_set_pair_kernel(int enable);

/*
 * Failure-detection hook for tests. The NEXT gemm_* call made by this thread
 * runs with the given fault mode and per-wait time limit, then both reset:
 *   fault 0 = none; 1 = the kernel's producer never loads its first shared-
 *   memory stage, so every wait for that stage expires after wait_limit_ns,
 *   the kernel records GEMM14_ERR_TIMEOUT in the device error word, drains
 *   its in-flight copies and exits; C is left incomplete.
 *   wait_limit_ns = 0 keeps the default limit (2 s).
 * No fault makes the GPU fault, trap or hang: waits are bounded, the context
 * stays usable, and gemm14_check_device_error reports the timeout.
 * The fp32 small-product kernel (plan kernel 6) synchronises only through
 * block and cluster barriers, with no mbarrier wait to expire: a call that
 * runs on it consumes the request and computes C as usual.
 * Returns GEMM14_ERR_INVALID_ARG for an unknown mode.
 */
int gemm14_debug_inject(int fault, uint64_t wait_limit_ns);

/* Library version, major * 10000 + minor * 100 + patch. */
int gemm14_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMM14_H */
