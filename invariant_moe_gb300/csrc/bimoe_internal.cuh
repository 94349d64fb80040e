// bimoe_internal.cuh -- shared device helpers of the CUDA library (sm_103a).
//
// Inline-PTX wrappers for mbarriers, TMA tensor copies and the tcgen05
// tensor-core / tensor-memory instructions, plus the bounded-wait discipline:
// every spin on an mbarrier gives up after a wall-clock limit, records
// BI_DEVERR_WAIT_TIMEOUT in the device error word and lets the kernel unwind
// (drain its own copies, free its tensor memory, return) instead of hanging.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/bimoe.h"

namespace bimoe {

// Wall-clock limit of one mbarrier wait.  Every legitimate wait in these
// kernels lasts microseconds; one second means something is broken.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// ------------------------------------------------------------- host side --
// Device error word of the current device (defined in api.cu).
int *device_error_word();
int num_sms();
// Unique id of the CUDA context current on this host thread (cuCtxGetId: ids
// are never reused within a process), or 0 when no context is current.
// Facts that belong to a context -- device addresses of __device__ symbols,
// per-function attributes such as the dynamic shared-memory limit -- are
// cached under this id and redone when it changes (a cudaDeviceReset, or a
// caller running in a context other than the device's primary one).
unsigned long long current_context_id();
// Per-device record of the context in which a one-time set-up was done.
struct ContextSetup {
  unsigned long long ctx[64] = {};
  // true when `dev`'s set-up has not been done in the current context
  bool pending(int dev) const { return dev >= 0 && dev < 64 && (ctx[dev] == 0 || ctx[dev] != current_context_id()); }
  void done(int dev) {
    if (dev >= 0 && dev < 64) ctx[dev] = current_context_id();
  }
};
// Encode a 2-D bf16 TMA map over a row-major [rows, cols] tensor with a
// [box_rows, 64]-element box and 128-byte swizzle.  Returns false on failure.
bool make_tma_2d_bf16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                      uint32_t box_rows);
// Same for a row-major fp32 tensor with a [box_rows, 32]-element box.
// The gate/up weights W13 [E, 2I, K] bf16 viewed as {K, 16, 2, E*2I/16}:
// a box {64, 16, 2, 4} at group g lands 16 gate rows, the 16 up rows of the
// same features (I rows further), and so on for four groups: 64 features'
// interleaved rows in one copy, 128-byte swizzled like the 2-D map's.
bool make_tma_inter_bf16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t I, uint64_t K);
bool make_tma_2d_f32(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows);
void set_error(const char *fmt, ...);

// Launches `kernel` as a programmatic dependent of the previous work on the
// stream (programmatic stream serialization) and, for cluster_x > 1, in
// clusters of cluster_x CTAs.  Every kernel of this library begins with
// griddep_wait(), so its launch overlaps the end of its predecessor while
// every memory access still follows it.  Only the short kernels with small
// grids (griddep_wait_small_release) trigger their dependents early; for the
// rest the trigger is each CTA's exit: CTAs of a dependent grid parked on the
// SMs while a large grid runs were measured to slow it.
template <typename... KArgs, typename... Args>
bi_status launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t stream, int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  if (e != cudaSuccess) {
    set_error("kernel launch: %s", cudaGetErrorString(e));
    return BI_ERR_CUDA;
  }
  return BI_OK;
}

#define BI_CHECK_LAUNCH()                                                  \
  do {                                                                     \
    cudaError_t e_ = cudaGetLastError();                                   \
    if (e_ != cudaSuccess) {                                               \
      ::bimoe::set_error("launch failed: %s", cudaGetErrorString(e_));     \
      return BI_ERR_CUDA;                                                  \
    }                                                                      \
  } while (0)

// ----------------------------------------------------------- device side --
__device__ __forceinline__ void report_error(int *err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Programmatic dependent launch.  launch_dependents lets a grid launched
// after this one with the programmatic-serialization attribute start its
// prologue early; griddep_wait, in that dependent grid, returns once every
// grid it depends on has completed and its memory is visible (a no-op
// without such a dependency).  Neither spins in software.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// For the short kernels of the path: wait for the predecessor and, when this
// grid is small (a decode-sized batch: at most 64 CTAs, most SMs idle), let
// the successor grid launch at once; its CTAs park at their own
// griddep_wait until this grid has finished, and a GEMM successor sets up its
// barriers and tensor memory meanwhile.  Larger grids leave the trigger to
// CTA exit (parked successor CTAs were measured to slow them).
__device__ __forceinline__ void griddep_wait_small_release() {
  griddep_wait();
  if (gridDim.x * gridDim.y * gridDim.z <= 64u) griddep_launch_dependents();
}

// ---- L2
// Drops the 128-byte line at p (128-byte aligned) from L2 without writing it
// back: its contents become indeterminate.  Only for data nothing reads again.
__device__ __forceinline__ void discard_l2_line(const void *p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// One lane of a fully active warp is elected (the same lane for every lane's
// answer).  Issuing tcgen05 / TMA instructions under this predicate from
// warp-uniform code keeps their operands (descriptors, coordinates) in
// uniform registers; issuing them from inside a `lane == 0` branch does not.
__device__ __forceinline__ bool elect_one() {
  uint32_t p;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(p));
  return p != 0;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase with the given parity (acquire on success);
// `cluster` selects cluster scope for barriers signalled by the other CTA of
// a pair.
template <bool CLUSTER>
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if (CLUSTER)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns
// false (after flagging) when the limit passes or another warp of the CTA has
// already aborted (*abort != 0; abort may be null for waits that must not be
// cut short, such as draining copies before exit).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          int *err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (abort && *abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        if (abort) *abort = 1;
        report_error(err, BI_DEVERR_WAIT_TIMEOUT);
        return false;
      }
    }
  }
}

// Same, for a barrier that receives arrivals from the other CTA of a pair
// (remote arrivals, multicast commits, the peer's TMA completions): the
// acquire is at cluster scope.
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, volatile int *abort,
                                             int *err) {
  if (mbar_try_wait_cl(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (abort && *abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        if (abort) *abort = 1;
        report_error(err, BI_DEVERR_WAIT_TIMEOUT);
        return false;
      }
    }
  }
}

// ---- grid-wide arrival count (one launch whose CTAs are all resident)
// Release-add / acquire-load of a global counter at GPU scope, and the proxy
// fence that orders generic-proxy global accesses with the thread's later
// TMA (async-proxy) accesses.
__device__ __forceinline__ void red_release_gpu_add(unsigned *p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Atomic add with acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int *p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Bounded wait for *p >= target (acquire).  Returns false (after flagging, as
// mbar_wait) when the limit passes or *abort is set.
__device__ __forceinline__ bool wait_count_geq(const unsigned *p, unsigned target, volatile int *abort,
                                               int *err) {
  if (ld_acquire_gpu(p) >= target) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    __nanosleep(64);
    if (ld_acquire_gpu(p) >= target) return true;
    if (abort && *abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      if (abort) *abort = 1;
      report_error(err, BI_DEVERR_WAIT_TIMEOUT);
      return false;
    }
  }
}

// ---- thread-block clusters (CTA pairs)
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
__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier given by its cluster address (own or peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// Relaxed arrivals: no release of the thread's earlier memory writes.  For
// signals that order only tensor-memory reads (already complete after
// tcgen05.wait::ld and fenced by tcgen05.fence::before_thread_sync), so the
// arriving thread does not wait for its global stores to drain.
__device__ __forceinline__ void mbar_arrive_relaxed(uint32_t bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// Every thread of every CTA of the cluster; used only at kernel entry and
// exit, which all threads reach on every path.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 2-D tiled load of box (c0 = inner/column coordinate, c1 = row coordinate).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// 2-D tiled load into this CTA's shared memory whose completion is counted
// on an mbarrier of either CTA of the pair (cluster address of the barrier).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map,
                                                 uint32_t bar_cluster, int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}

// 4-D tiled load (the interleaved gate/up weight map: coordinates {k, row
// in group, gate/up half, 16-row group}).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int32_t c0,
                                            int32_t c1, int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar_cluster,
                                                 int32_t c0, int32_t c1, int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// Four rows r0..r3 of a 2-D tensor map whose box is one row of 64 bf16
// (tile::gather4): 4 x 128 bytes land at dst as consecutive rows, in the
// map's swizzle, completion counted in bytes on the mbarrier.  c0 is the
// column, a multiple of 64.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap *map, uint32_t bar, int32_t c0,
                                            int32_t r0, int32_t r1, int32_t r2, int32_t r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
      : "memory");
}
// The same, completing on an mbarrier of either CTA of a pair.
__device__ __forceinline__ void tma_gather4_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar_cluster,
                                                 int32_t c0, int32_t r0, int32_t r1, int32_t r2, int32_t r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
      : "memory");
}

// ---- tcgen05 (5th-generation tensor cores, tensor memory)
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
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
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on an mbarrier when every previously issued tcgen05.mma of this
// thread has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// CTA-pair forms (cta_group::2).  Allocation, permit release and
// deallocation are executed by one warp in each CTA of the pair; the MMA and
// its commits are issued by one thread of the even CTA only.  A kernel uses
// either these or the cta_group::1 forms above, never both.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
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
// D (+)= A * B^T over the pair: A rows 0..127 from the even CTA's shared
// memory and rows 128..255 from the odd CTA's (same address), B columns
// 0..N/2-1 from the even CTA and N/2..N-1 from the odd CTA; D rows 0..127
// land in the even CTA's tensor memory, rows 128..255 in the odd CTA's.
__device__ __forceinline__ void umma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the mbarrier at this shared address in every CTA of
// cta_mask when all previously issued pair MMAs of this thread completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}
// 32 lanes x 32 consecutive fp32 columns; thread i of the warp receives lane
// (taddr.lane + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzle: rows of 64 bf16 (128 B), 8-row swizzle atoms of
// 1024 B stacked along M/N (stride byte offset 1024), descriptor version 1,
// layout type 2 (SWIZZLE_128B).  The tile base must be 1024-byte aligned;
// stepping K by 16 elements inside the atom adds 32 B to the start address.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;            // leading byte offset (unused here) = 16 B
  d |= static_cast<uint64_t>(1024 >> 4) << 32;    // stride byte offset = 1024 B
  d |= static_cast<uint64_t>(1) << 46;            // descriptor version
  d |= static_cast<uint64_t>(2) << 61;            // 128-byte swizzle
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator, bf16 A
// and B, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace bimoe
