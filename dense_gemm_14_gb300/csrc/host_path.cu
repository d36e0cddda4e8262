// host_path.cu -- the host-buffer runtime behind gemm14_gemm_host: operands
// in host memory, copied in, multiplied and copied back on three streams of
// the library's own (copies in, kernels, copies out), so that the transfers
// over the host link overlap the kernels, within a product (row panels) and
// from one product to the next. Device buffers come from a stream-ordered
// memory pool of the library's own, which caches them for reuse.
// The contract is documented in include/gemm14.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <memory>
#include <mutex>
#include <vector>

#include "../../include/gemm14.h"
#include "api_internal.h"

namespace gemm14 {
namespace {

constexpr int kMaxHostDevices = 64;

// An event destroyed with its last owner: a call's completion event may be
// waited for by several threads while the issuing thread retires it.
struct EventHolder {
  cudaEvent_t ev = nullptr;
  ~EventHolder() {
    if (ev) cudaEventDestroy(ev);
  }
};

// A call in flight: its ticket, device, completion (recorded on the copy-out
// stream after its last copy) and the bytes of host memory its C covers.
struct Pending {
  uint64_t ticket;
  int device;
  std::shared_ptr<EventHolder> done;
  uintptr_t c_lo, c_hi;
};

// Per device: the three streams, the memory pool, and the stream-K workspace
// (used by the kernel stream only, in its order).
struct Runtime {
  bool ready = false;
  cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
  cudaMemPool_t pool = nullptr;
  void* ws = nullptr;
  size_t ws_bytes = 0;
};

std::mutex g_mutex;  // guards everything below
Runtime g_rt[kMaxHostDevices];
std::vector<Pending> g_pending;
uint64_t g_next_ticket = 1;

int cuda_ok(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return GEMM14_OK;
  note_cuda_error(what, e);
  return GEMM14_ERR_CUDA;
}

// Creates the device's streams and pool on first use (g_mutex held). The pool
// keeps freed memory (no release threshold) and never makes an allocation
// wait for a free on another stream: it grows instead, so that the copy-in
// stream never waits behind the copy-out stream.
int runtime_for(int dev, Runtime** out) {
  Runtime& rt = g_rt[dev];
  if (!rt.ready) {
    int st;
    if ((st = cuda_ok(cudaStreamCreateWithFlags(&rt.in, cudaStreamNonBlocking), "stream")) ||
        (st = cuda_ok(cudaStreamCreateWithFlags(&rt.comp, cudaStreamNonBlocking), "stream")) ||
        (st = cuda_ok(cudaStreamCreateWithFlags(&rt.out, cudaStreamNonBlocking), "stream")))
      return st;
    cudaMemPoolProps props{};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    if ((st = cuda_ok(cudaMemPoolCreate(&rt.pool, &props), "cudaMemPoolCreate"))) return st;
    uint64_t keep = UINT64_MAX;
    int no = 0;
    if ((st = cuda_ok(cudaMemPoolSetAttribute(rt.pool, cudaMemPoolAttrReleaseThreshold, &keep),
                      "cudaMemPoolSetAttribute")) ||
        (st = cuda_ok(cudaMemPoolSetAttribute(rt.pool, cudaMemPoolReuseAllowInternalDependencies,
                                              &no),
                      "cudaMemPoolSetAttribute")))
      return st;
    rt.ready = true;
  }
  *out = &rt;
  return GEMM14_OK;
}

// Row panels of a host-buffer product: one for small products (transfers too
// short to pipeline); else up to one per 1024 rows of C, at most 8, taking the
// most panels whose own schedule keeps at least 85 % of the worker slots busy
// (a panel of a partial wave would leave SMs idle for its whole run). E.g. fp32
// 3072^3: 3 panels are 96 tiles on 152 SMs each (63 %), 2 panels 144 (95 %).
// Measured on GB300 with consecutive fp32 3072^3 and bf16 8192^3 products:
// 2.50 ms per pair with 3 fp32 panels, 2.13-2.15 ms with 1 or 2.
int64_t default_panels(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K) {
  if (transa || M * N * K < (int64_t(1) << 31) || M < 2048) return 1;
  for (int64_t P = std::min<int64_t>(8, M / 1024); P > 1; --P)
    if (schedule_efficiency(dtype, transa, transb, (M + P - 1) / P, N, K) >= 0.85) return P;
  return 1;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Host bytes [lo, hi) of a rows x cols matrix with row pitch ld elements.
void span(const void* p, int64_t rows, int64_t cols, int64_t ld, int eb, uintptr_t* lo,
          uintptr_t* hi) {
  *lo = reinterpret_cast<uintptr_t>(p);
  *hi = rows > 0 && cols > 0 ? *lo + static_cast<uintptr_t>(((rows - 1) * ld + cols) * eb) : *lo;
}

}  // namespace
}  // namespace gemm14

using namespace gemm14;

namespace gemm14 {
namespace {

// Makes `in` wait for every call in flight whose C overlaps [lo, hi) (g_mutex held).
int wait_for_writers(cudaStream_t in, uintptr_t lo, uintptr_t hi) {
  if (lo == hi) return GEMM14_OK;
  for (const Pending& p : g_pending) {
    if (lo < p.c_hi && p.c_lo < hi) {
      const int st = cuda_ok(cudaStreamWaitEvent(in, p.done->ev, 0), "cudaStreamWaitEvent");
      if (st) return st;
    }
  }
  return GEMM14_OK;
}

// One stream waits for the work enqueued so far on another.
int order(cudaStream_t before, cudaStream_t after) {
  cudaEvent_t e = nullptr;
  int st = cuda_ok(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "cudaEventCreate");
  if (st) return st;
  if (!(st = cuda_ok(cudaEventRecord(e, before), "cudaEventRecord")))
    st = cuda_ok(cudaStreamWaitEvent(after, e, 0), "cudaStreamWaitEvent");
  cudaEventDestroy(e);  // released once recorded work completes
  return st;
}

// Grows the kernel stream's stream-K workspace to `need` bytes, in that
// stream's order (the old one is freed after the kernels that use it).
int ensure_workspace(Runtime& rt, size_t need) {
  if (need <= rt.ws_bytes) return GEMM14_OK;
  int st;
  if (rt.ws && (st = cuda_ok(cudaFreeAsync(rt.ws, rt.comp), "cudaFreeAsync"))) return st;
  rt.ws = nullptr;
  rt.ws_bytes = 0;
  if ((st = cuda_ok(cudaMallocFromPoolAsync(&rt.ws, need, rt.pool, rt.comp), "workspace")) ||
      (st = cuda_ok(cudaMemsetAsync(rt.ws, 0, need, rt.comp), "cudaMemsetAsync")))
    return st;
  rt.ws_bytes = need;
  return GEMM14_OK;
}

struct HostCall {
  int dtype, transa, transb;
  int64_t M, N, K;
  float alpha, beta;
  const void* A;
  int64_t lda;
  const void* B;
  int64_t ldb;
  float* C;
  int64_t ldc;
  int64_t panels;
};

// Enqueues one product (g_mutex held). On success *done is its completion.
int enqueue(Runtime& rt, const HostCall& c, std::shared_ptr<EventHolder>* done) {
  const int eb = operand_bytes(c.dtype);
  const bool reads_ab = c.K > 0 && c.alpha != 0.0f;
  const bool reads_c = c.beta != 0.0f;
  const int64_t rows_a = c.transa ? c.K : c.M, cols_a = c.transa ? c.M : c.K;
  const int64_t rows_b = c.transb ? c.N : c.K, cols_b = c.transb ? c.K : c.N;
  // Device pitches rounded up to 16 bytes, so that every operand is one the
  // kernels' TMA loaders take.
  const int64_t lda_d = round_up(std::max<int64_t>(cols_a, 1), 16 / eb);
  const int64_t ldb_d = round_up(std::max<int64_t>(cols_b, 1), 16 / eb);
  const int64_t ldc_d = round_up(c.N, 4);
  uintptr_t lo, hi;
  int st;
  if (reads_ab) {
    span(c.A, rows_a, cols_a, c.lda, eb, &lo, &hi);
    if ((st = wait_for_writers(rt.in, lo, hi))) return st;
    span(c.B, rows_b, cols_b, c.ldb, eb, &lo, &hi);
    if ((st = wait_for_writers(rt.in, lo, hi))) return st;
  }
  if (reads_c) {
    span(c.C, c.M, c.N, c.ldc, 4, &lo, &hi);
    if ((st = wait_for_writers(rt.in, lo, hi))) return st;
  }
  char *a_d = nullptr, *b_d = nullptr, *c_d = nullptr;
  if (reads_ab &&
      ((st = cuda_ok(cudaMallocFromPoolAsync(reinterpret_cast<void**>(&a_d),
                                             rows_a * lda_d * eb, rt.pool, rt.in), "A buffer")) ||
       (st = cuda_ok(cudaMallocFromPoolAsync(reinterpret_cast<void**>(&b_d),
                                             rows_b * ldb_d * eb, rt.pool, rt.in), "B buffer"))))
    return st;
  if ((st = cuda_ok(cudaMallocFromPoolAsync(reinterpret_cast<void**>(&c_d),
                                            c.M * ldc_d * 4, rt.pool, rt.in), "C buffer")))
    return st;
  if (reads_ab) {
    if ((st = cuda_ok(cudaMemcpy2DAsync(b_d, ldb_d * eb, c.B, c.ldb * eb, cols_b * eb, rows_b,
                                        cudaMemcpyHostToDevice, rt.in), "copy of B")))
      return st;
    if (c.transa &&
        (st = cuda_ok(cudaMemcpy2DAsync(a_d, lda_d * eb, c.A, c.lda * eb, cols_a * eb, rows_a,
                                        cudaMemcpyHostToDevice, rt.in), "copy of A")))
      return st;
  }
  // Operands the kernels do not read still need valid pointers.
  const void* a_ptr = reads_ab ? static_cast<const void*>(a_d) : c_d;
  const void* b_ptr = reads_ab ? static_cast<const void*>(b_d) : c_d;
  const int64_t P = std::max<int64_t>(1, std::min<int64_t>(c.transa ? 1 : c.panels, c.M));
  for (int64_t p = 0; p < P; ++p) {
    const int64_t r0 = c.M * p / P, r1 = c.M * (p + 1) / P;
    if (r1 == r0) continue;
    if (reads_ab && !c.transa &&
        (st = cuda_ok(cudaMemcpy2DAsync(a_d + r0 * lda_d * eb, lda_d * eb,
                                        static_cast<const char*>(c.A) + r0 * c.lda * eb,
                                        c.lda * eb, cols_a * eb, r1 - r0,
                                        cudaMemcpyHostToDevice, rt.in), "copy of A")))
      return st;
    if (reads_c &&
        (st = cuda_ok(cudaMemcpy2DAsync(c_d + r0 * ldc_d * 4, ldc_d * 4, c.C + r0 * c.ldc,
                                        c.ldc * 4, c.N * 4, r1 - r0, cudaMemcpyHostToDevice,
                                        rt.in), "copy of C")))
      return st;
    if ((st = order(rt.in, rt.comp))) return st;
    const char* a_panel = reads_ab && !c.transa ? static_cast<const char*>(a_ptr) + r0 * lda_d * eb
                                                : static_cast<const char*>(a_ptr);
    float* c_panel = reinterpret_cast<float*>(c_d) + r0 * ldc_d;
    const size_t need = product_workspace_bytes(c.dtype, c.transa, c.transb, r1 - r0, c.N, c.K,
                                                a_panel, lda_d, b_ptr, ldb_d, c_panel, ldc_d);
    if ((st = ensure_workspace(rt, need))) return st;
    if ((st = product_on_stream(c.dtype, c.transa, c.transb, r1 - r0, c.N, c.K, c.alpha, a_panel,
                                lda_d, b_ptr, ldb_d, c.beta, c_panel, ldc_d, rt.ws, rt.ws_bytes,
                                rt.comp)))
      return st;
    if ((st = order(rt.comp, rt.out))) return st;
    if ((st = cuda_ok(cudaMemcpy2DAsync(c.C + r0 * c.ldc, c.ldc * 4, c_panel, ldc_d * 4, c.N * 4,
                                        r1 - r0, cudaMemcpyDeviceToHost, rt.out), "copy of C")))
      return st;
  }
  auto holder = std::make_shared<EventHolder>();
  if ((st = cuda_ok(cudaEventCreateWithFlags(&holder->ev, cudaEventDisableTiming),
                    "cudaEventCreate")) ||
      (st = cuda_ok(cudaEventRecord(holder->ev, rt.out), "cudaEventRecord")))
    return st;
  // Every use of the buffers precedes this point of the copy-out stream.
  for (char* b : {a_d, b_d, c_d})
    if (b && (st = cuda_ok(cudaFreeAsync(b, rt.out), "cudaFreeAsync"))) return st;
  *done = std::move(holder);
  return GEMM14_OK;
}

}  // namespace
}  // namespace gemm14

extern "C" {

int gemm14_gemm_host(int dtype, int transa, int transb, int64_t M, int64_t N, int64_t K,
                     float alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
                     float beta, float* C, int64_t ldc, int panels, uint64_t* ticket) {
  if (!ticket || panels < 0) return GEMM14_ERR_INVALID_ARG;
  int st = validate_product(dtype, transa, transb, M, N, K, A, lda, B, ldb, C, ldc);
  if (st != GEMM14_OK) return st;
  int dev = -1;
  if ((st = current_device_index(&dev)) != GEMM14_OK) return st;
  if (dev < 0 || dev >= kMaxHostDevices) return GEMM14_ERR_UNSUPPORTED_DEVICE;
  const bool reads_ab = K > 0 && alpha != 0.0f;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (M == 0 || N == 0 || (!reads_ab && beta == 1.0f)) {
    *ticket = g_next_ticket++;  // nothing to do: complete as issued
    return GEMM14_OK;
  }
  Runtime* rt = nullptr;
  if ((st = runtime_for(dev, &rt)) != GEMM14_OK) return st;
  const HostCall call{dtype, transa, transb, M, N, K, alpha, beta, A, lda, B, ldb, C, ldc,
                      panels ? panels : default_panels(dtype, transa, transb, M, N, K)};
  std::shared_ptr<EventHolder> done;
  if ((st = enqueue(*rt, call, &done)) != GEMM14_OK) return st;
  uintptr_t lo, hi;
  span(C, M, N, ldc, 4, &lo, &hi);
  const uint64_t t = g_next_ticket++;
  g_pending.push_back(Pending{t, dev, std::move(done), lo, hi});
  *ticket = t;
  return GEMM14_OK;
}

int gemm14_host_wait(uint64_t ticket) {
  std::shared_ptr<EventHolder> done;
  int dev = -1;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (ticket == 0 || ticket >= g_next_ticket) return GEMM14_ERR_INVALID_ARG;
    for (const Pending& p : g_pending)
      if (p.ticket == ticket) {
        done = p.done;
        dev = p.device;
      }
  }
  if (!done) return GEMM14_OK;  // nothing was enqueued, or already waited for
  int prev = -1;
  int st = cuda_ok(cudaGetDevice(&prev), "cudaGetDevice");
  if (st) return st;
  if (prev != dev && (st = cuda_ok(cudaSetDevice(dev), "cudaSetDevice"))) return st;
  st = cuda_ok(cudaEventSynchronize(done->ev), "cudaEventSynchronize");
  if (st == GEMM14_OK) st = take_device_error();
  if (prev != dev) cudaSetDevice(prev);
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    g_pending.erase(std::remove_if(g_pending.begin(), g_pending.end(),
                                   [ticket](const Pending& p) { return p.ticket == ticket; }),
                    g_pending.end());
  }
  return st;
}

int gemm14_host_synchronize(void) {
  std::vector<uint64_t> tickets;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    for (const Pending& p : g_pending) tickets.push_back(p.ticket);
  }
  int first = GEMM14_OK;
  for (uint64_t t : tickets) {
    const int st = gemm14_host_wait(t);
    if (first == GEMM14_OK) first = st;
  }
  return first;
}

}  // extern "C"
