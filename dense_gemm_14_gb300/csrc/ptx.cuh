// ptx.cuh -- inline-PTX wrappers for the sm_103a building blocks the kernels
// use: mbarriers (with bounded waits), TMA tile loads, cp.async with zero fill,
// and the tcgen05 tensor-core family (TMEM alloc, MMA, commit, TMEM loads).
//
// Every wait here is bounded: a wait that does not finish within its limit
// (kWaitTimeoutNs unless the call set another) or that sees the CTA's abort
// flag returns false instead of spinning forever, so a protocol bug ends the
// kernel with an error status instead of hanging the GPU.
#pragma once

#include <cstdint>
#include <cuda.h>  // CUtensorMap (type only; the driver is reached at run time)

#include "checks.h"

namespace gemm14 {

// Bits OR-ed into the library's device error word (and kDevErrBounds, the
// device-side bounds checks' bit, in checks.h).
enum : unsigned { kDevErrTimeout = 1u, kDevErrBadConfig = 2u };

constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // default limit of one wait: 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------- programmatic dependent launch
// The kernels are launched with programmatic stream serialisation, so a grid
// may start while the grid before it on the stream is still running. Every
// thread calls grid_dependency_wait() before its first access to global
// memory: it returns once the earlier grid has completed and its writes are
// visible (at once when there is no such grid). After it, the grid lets the
// next one start its own launch and prologue (grid_launch_dependents); that
// grid in turn waits in grid_dependency_wait() for this one to complete.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA / tcgen05) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// How a kernel waits: where to report an expired wait, the CTA's abort flag,
// and the time limit of one wait.
struct WaitCtx {
  unsigned* err;
  volatile int* abort_flag;
  unsigned long long limit_ns;
  uint32_t peer_abort;  // cluster address of the peer CTA's abort flag (0: no peer)
};

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity);

// Slow path of mbar_wait: spins with a time limit. On expiry it records
// kDevErrTimeout in *err and raises the CTA-wide abort flag (and the peer
// CTA's, for a CTA pair) so the other roles stop waiting too.
template <bool kClusterScope>
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity,
                                                   const WaitCtx& w) {
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity))
      return true;
    if ((i & 31u) == 0) {
      if (*w.abort_flag) return false;
      if (globaltimer_ns() - t0 > w.limit_ns) {
        atomicOr(w.err, kDevErrTimeout);
        *w.abort_flag = 1;
        if (w.peer_abort)
          asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(w.peer_abort), "r"(1u) : "memory");
        return false;
      }
    }
  }
}

// Wait with only a time limit (no abort flag): used to drain copies still in
// flight after an abort. Returns false if the limit expired.
static __device__ __noinline__ bool mbar_wait_timed(uint64_t* bar, uint32_t parity,
                                             unsigned long long limit_ns) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}

// Waits until the barrier phase with the given parity has completed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow<false>(bar, parity, w);
}

// As mbar_wait, for a barrier that receives arrivals from the peer CTA.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  const WaitCtx& w) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  return mbar_wait_slow<true>(bar, parity, w);
}

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// All threads of both CTAs: release this CTA's prior writes, acquire the peer's.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// One arrival on an mbarrier in another CTA of the cluster (release, cluster scope).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ void st_shared_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// try_wait with cluster-scope acquire (for barriers that receive remote arrivals).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// ---------------------------------------------------------------- global flags
// Publishes `value` at `flag` after every write this thread (and, through a
// preceding CTA barrier, its CTA) made before it (release, GPU scope).
__device__ __forceinline__ void flag_publish(unsigned* flag, unsigned value) {
  __threadfence();
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(flag), "r"(value) : "memory");
}

// Clears a flag that its one waiter has seen (GPU scope). The next call on
// the stream starts after this grid completes and finds it 0, so a launch
// replayed with the same epoch (a captured CUDA graph) never takes a previous
// replay's publication for its own.
__device__ __forceinline__ void flag_clear(unsigned* flag) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(flag), "r"(0u) : "memory");
}

// Waits until *flag == value (acquire, GPU scope), bounded like mbar_wait.
// flag_wait_inline is the loop itself, for a caller that holds many live
// registers across the wait (a call would have to save them); flag_wait is
// the same loop as a call.
__device__ __forceinline__ bool flag_wait_inline(const unsigned* flag, unsigned value,
                                                 const WaitCtx& w) {
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v == value) return true;
    if ((i & 15u) == 15u) {
      if (*w.abort_flag) return false;
      if (globaltimer_ns() - t0 > w.limit_ns) {
        atomicOr(w.err, kDevErrTimeout);
        *w.abort_flag = 1;
        if (w.peer_abort)
          asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(w.peer_abort), "r"(1u) : "memory");
        return false;
      }
    }
    __nanosleep(64);
  }
}
static __device__ __noinline__ bool flag_wait(const unsigned* flag, unsigned value,
                                              const WaitCtx& w) {
  return flag_wait_inline(flag, value, w);
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled TMA load of one box at (x = inner coordinate, y = outer coordinate)
// into shared memory; completion is signalled on `bar` as transaction bytes.
// Out-of-range elements of the box are zero-filled by the hardware.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// The same load for a CTA pair: the box lands in this CTA's shared memory,
// completion is signalled on `bar_cluster_addr`, an mbarrier that may live in
// the peer CTA (the pair's leader).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, int32_t x,
                                                 int32_t y, uint32_t bar_cluster_addr) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster_addr)
      : "memory");
}

// 2-D tiled TMA store of one box from shared memory to (x, y); out-of-range
// parts of the box are not written. Bulk-group completion: commit, then wait
// until at most N of this thread's groups still read shared memory (the
// buffer may be rewritten) or, with wait_all, until every group is done.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* smem_src,
                                             int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(smem_u32(smem_src))
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------- cp.async
// 4-byte asynchronous global->shared copy; src_bytes = 0 writes zeros and reads
// nothing (used for out-of-range tile elements).
__device__ __forceinline__ void cp_async_4(uint32_t smem_dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}

// The barrier receives one arrival when all of this thread's earlier cp.async
// copies have landed (the barrier's expected count must include it).
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// ---------------------------------------------------------------- shared loads
__device__ __forceinline__ float4 lds128(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_result)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// CTA-pair (cta_group::2) forms: one warp of EACH CTA of the pair executes
// alloc / relinquish / dealloc; the pair gets the same TMEM columns.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_result)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Pair MMA, issued by one thread of the leader CTA: A rows split between the
// two CTAs, B columns split between them, D in each CTA's TMEM (its rows).
__device__ __forceinline__ void tc_mma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}
// The same pair MMA with tf32 operands (fp32 bit patterns in shared memory,
// K = 8 per instruction), fp32 accumulation.
__device__ __forceinline__ void tc_mma_tf32_pair(uint32_t d_tmem, uint64_t a_desc,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}
// Arrives once on the barrier at this shared offset in every CTA of cta_mask
// when the pair MMAs issued so far by this thread have completed.
__device__ __forceinline__ void tc_commit_pair_multicast(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], one instruction of shape given by
// the instruction descriptor; accumulate selects D += (true) or D = (false).
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// The barrier receives one arrival once every tcgen05 operation this thread
// issued before the commit has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Loads 32 consecutive fp32 columns of this thread's TMEM lane (lane = warp's
// 32-lane quarter + lane id) into registers; call tc_wait_ld before use.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma (64 bits): start address,
// leading- and stride-dimension byte offsets (all >> 4), descriptor version 1,
// base offset 0 and the 128-byte swizzle mode. Tiles are 1024-byte aligned.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // version
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor for kind::f16 with fp32 accumulation: A and B both
// fp16 (is_bf16 = false) or both bf16; A K-major, B MN-major; shape M x N.
// a_mn / b_mn: the operand is MN-major in shared memory (M or N contiguous)
// rather than K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32acc(bool is_bf16, int M, int N, bool a_mn,
                                                        bool b_mn) {
  return (1u << 4)                                  // D format: f32
         | ((is_bf16 ? 1u : 0u) << 7)               // A format
         | ((is_bf16 ? 1u : 0u) << 10)              // B format
         | ((a_mn ? 1u : 0u) << 15)                 // A major-ness
         | ((b_mn ? 1u : 0u) << 16)                 // B major-ness
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// Instruction descriptor for kind::tf32 with fp32 accumulation, both
// operands K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_tf32_f32acc(int M, int N) {
  return (1u << 4)                                  // D format: f32
         | (2u << 7)                                // A format: tf32
         | (2u << 10)                               // B format: tf32
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// Shared-memory layout of one 64-deep k-block of a 16-bit operand with the
// 128-byte swizzle, as the kernels' loaders write it:
//  K-major:  128-byte rows of 64 k, 8-row groups 1024 B apart (stride
//            offset); a K = 16 slice starts 32 B further along the rows.
//  MN-major: boxes of 64 (m or n) x 64 k rows, 8 KB each, boxes 8 KB apart
//            (leading offset), 8-k groups 1024 B apart; a K = 16 slice starts
//            16 rows (2048 B) further.
struct OperandDesc {
  uint32_t step;  // bytes from one K = 16 slice to the next
  uint32_t lbo;   // leading byte offset of the descriptor
};
__device__ __forceinline__ OperandDesc operand_desc(bool k_major) {
  return k_major ? OperandDesc{32u, 16u} : OperandDesc{2048u, 8192u};
}

}  // namespace gemm14
