// common.cuh -- device helpers shared by the decode kernels (sm_103a).
//
// PTX wrappers for mbarriers, TMA (cp.async.bulk.tensor) and L2 bulk prefetch, the
// bounded-wait helper every kernel uses, and bf16 unpacking. Nothing here computes a
// result of the method; the kernels do.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssd {

// Tile geometry shared by the split-K engine and its host-side planner.
constexpr int TILE_N = 128;     // W rows per tile (tcgen05 MMA M)
constexpr int TILE_K = 64;      // k per block: one 128-byte swizzle row of bf16
constexpr int WBOX_ROWS = 64;   // rows per W TMA box (two boxes per tile)
constexpr int XBOX_ROWS = 16;   // activation rows per TMA box (MMA N granularity)
constexpr int MAX_B = 64;        // decode batch of every operation
constexpr int MAX_B_WIDE = 256;  // rows of one tensor-core projection launch
constexpr int MAX_ROWS = 512;    // rows of a projection call (launches of <= 256 rows each)
constexpr int MAX_E = 512;
constexpr int MAX_TOPK = 16;
// shared memory of the routing tail: ids [B*topk], token masks [E], offsets [E]
constexpr int ROUTE_SCRATCH_BYTES = 4 * MAX_B * MAX_TOPK + 8 * MAX_E + 4 * MAX_E;

// Device status bits (dec_sync_status maps them to dec_status).
constexpr unsigned ST_TIMEOUT = 1u;
constexpr unsigned ST_BAD_ROUTING = 2u;  // an expert index out of range or repeated

// Mode of the split-K engine's epilogue.
enum EngineMode : int {
  MODE_LINEAR = 0,   // Y = bf16(acc (+R))
  MODE_FRONT = 1,    // router + latent product: partial tiles only, added by a dependent kernel
  MODE_GATEUP = 2,   // A = bf16(silu(gate) * up)
  MODE_DOWN = 3      // Yp = acc (fp32)
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------- thread-block clusters ----
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// Every thread of every CTA of the cluster arrives (release) and waits (acquire): the
// distributed-shared-memory stores made before it are visible after it. Executed by
// whole warps at the same point.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The same split in two: a relaxed arrival (orders nothing) early on, and the matching
// wait where the other CTAs must be known to be running (before the first store into
// their shared memory). Either may be executed by diverged threads.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier ----

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with the given parity, for at most limit_ns. On time-out
// set ST_TIMEOUT in *status and the CTA-wide abort flag, and return false. Any waiter
// that sees the abort flag returns false as well, so one time-out ends every loop of
// the CTA without a second full wait.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  unsigned *status, volatile int *abort_flag,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicOr(status, ST_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}

// Used only after a time-out: wait up to limit_ns for a phase (an in-flight copy of
// this CTA landing) without touching the status word. Returns whether it completed.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity,
                                                uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}

// --------------------------------------------------------------------- TMA ----

// 2-D tiled TMA load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// Same, with an L2 cache policy from createpolicy (evict-first for weights read once).
__device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *map,
                                                        uint64_t *bar, int c0, int c1,
                                                        uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

// Same, into this CTA's shared memory, with the completion counted on an mbarrier of the
// CTA pair (bar_cluster: a shared::cluster address, in this CTA or its pair partner).
__device__ __forceinline__ void tma_load_2d_pair_hint(void *dst, const CUtensorMap *map,
                                                      uint32_t bar_cluster, int c0, int c1,
                                                      uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes.L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *map,
                                                 uint32_t bar_cluster, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}

// 2-D tiled TMA store shared -> global of one box (coordinates c0 inner, c1 outer; parts
// of the box outside the tensor are not written), tracked by this thread's bulk group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int c0,
                                             int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until every bulk group this thread committed has completed (its writes done).
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Orders this thread's generic-proxy shared-memory writes before later async-proxy
// (TMA) reads of them; executed by the writers before the barrier that precedes the copy.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Bulk prefetch of [addr, addr+bytes) into L2 (addr 16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void prefetch_l2_bulk(const void *addr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                   reinterpret_cast<uint64_t>(addr)),
               "r"(bytes)
               : "memory");
}

// 1-D bulk copy global -> shared memory of `bytes` (a multiple of 16, both addresses
// 16-byte aligned), completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load_1d(void *dst, const void *src, uint32_t bytes,
                                             uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes),
      "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------- atomics ----
// GPU-scope acquire-release add. Issued by one thread after a CTA barrier, it publishes
// every write the CTA made before the barrier (release is cumulative) and, for the
// thread that sees the final count, makes every other CTA's published writes visible
// (acquire); a following CTA barrier extends that to the whole CTA.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int *p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

// GPU-scope release add without a return value: issued by one thread after a CTA
// barrier, it publishes every write the CTA made before the barrier.
__device__ __forceinline__ void red_add_release_gpu(int *p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Orders this thread's generic-proxy accesses to global memory with its async-proxy
// ones (TMA): data written by ordinary stores and then read by cp.async.bulk.tensor.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Wait until *cnt >= target (GPU-scope acquire), for at most limit_ns; on time-out the
// same as mbar_wait_bounded.
__device__ __forceinline__ bool wait_count_bounded(const int *cnt, int target, unsigned *status,
                                                   volatile int *abort_flag,
                                                   uint64_t limit_ns) {
  if (ld_acquire_gpu(cnt) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 8; ++i) {
      __nanosleep(64);
      if (ld_acquire_gpu(cnt) >= target) return true;
    }
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicOr(status, ST_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}

// ------------------------------------------------ programmatic dependent launch ----
// griddep_wait: block until the previous kernel of the stream has completed and its
// writes are visible (a no-op when the launch was not programmatic). Everything that
// reads an activation, a route map or the workspace, or writes any output, comes after
// it; only static weights may be loaded before it. The "memory" clobber keeps the
// compiler from hoisting ordinary loads above the wait.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Let the next kernel of the stream be scheduled as SMs free up.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ named barriers ----

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------- loads ----

// Streaming 128-bit load of static weights: read-only path, no L1 allocation.
// Only ever used on weights, never on activations a previous kernel writes.
__device__ __forceinline__ uint4 ld_weight_stream(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ------------------------------------------------------------------- bf16 ----

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t *>(&b);
}

// Order-preserving map of a float onto uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t f32_order_key(float f) {
  uint32_t u = __float_as_uint(f + 0.0f);  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace ssd
