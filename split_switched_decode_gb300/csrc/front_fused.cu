// front_fused.cu -- the MoE front end in one kernel: router + latent product on tensor
// cores, split-K reduction on chip, top-k routing, renormalisation and the routing
// inverse map.
//
// "Hyper Optimizing Kimi K3 in vLLM", Part 1 / 3 "Improve MoE scheduling and overlap":
// the router scores and the latent input projection are computed as one matrix product
// over the concatenated weight W_cat = [router rows ; latent rows], which removes
// repeated weight reads and kernel launches ahead of the expert computation. Here the
// routing that follows the product runs in the same launch.
//
// Work split. W_cat is cut into T tiles of 128 rows; tile t is handled by one
// thread-block cluster of S CTAs (S a power of two, 16 for the Kimi shape), CTA c of the
// cluster multiplying k-blocks [c*KB/S, (c+1)*KB/S) of the tile with every token:
//
//   warp 0     TMA producer (lane 0): before the dependency wait it issues the weight
//              boxes of the first `nst` k-blocks into the stage ring and an L2 prefetch
//              of the rest of its weights, then lets the next kernel of the stream be
//              scheduled; after the wait, the activation boxes and the remaining weights
//   warp 1     tensor-memory owner and MMA issuer (lane 0): tcgen05.mma M128 x N16*NXB
//              x K16, fp32 accumulator in tensor memory
//   warps 4-7  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM lanes
//              32*(w%4)..+31 = tile rows) and st.async of each token's partial rows
//              straight from registers into the receive area of the CTA of the cluster
//              that owns the token (token b -> CTA b % S), completion counted in bytes on
//              that CTA's mbarrier
//
// Every CTA that owns tokens then adds the S partials of each of its tokens in CTA
// order (fixed order: the bits do not depend on timing), tells each sender that its
// rows have landed (remote mbarrier arrive: a CTA leaves only when all its receivers
// have), and writes the latent rows as bf16 and the router logits as fp32. Acquire-
// release arrival counters then elect the router CTA(s) that route -- a warp per token:
// a lower bound from the lanes' largest logits, the candidates above it, their exact
// ranks -- renormalise the chosen weights, write topk_idx / topk_w and the optional full
// softmax, and the CTA that builds the route map with all its threads. No CTA ever waits
// for a CTA outside its cluster; inside a cluster the hardware co-schedules all CTAs.
#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "routing.cuh"
#include "tcgen05.cuh"

namespace ssd {

namespace {

constexpr int FF_THREADS = 256;

__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}

// Bring a 64 x 128 box of a tensor map into L2 (no shared-memory destination).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap *map, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1)
               : "memory");
}

// Remote mbarrier arrival on a barrier of a CTA of the cluster (relaxed: it only tells
// that CTA that the data it sent has landed; nothing is published with it).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t mbar_cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                   mbar_cluster_addr)
               : "memory");
}

// Stores into shared memory of a CTA of the cluster whose completion is counted in bytes
// on that CTA's mbarrier (addresses mapped with mapa).
__device__ __forceinline__ void st_async_f32(uint32_t addr, float a, uint32_t mbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(
                   addr),
               "r"(__float_as_uint(a)), "r"(mbar)
               : "memory");
}
__device__ __forceinline__ void st_async_v2(uint32_t addr, float a, float b, uint32_t mbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(
          addr),
      "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(mbar)
      : "memory");
}
__device__ __forceinline__ void st_async_v4(uint32_t addr, float a, float b, float c, float d,
                                            uint32_t mbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, "
      "[%5];" ::"r"(addr),
      "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(__float_as_uint(c)),
      "r"(__float_as_uint(d)), "r"(mbar)
      : "memory");
}

template <int NXB>
__global__ void __launch_bounds__(FF_THREADS, 2)
    front_fused_kernel(const __grid_constant__ CUtensorMap wmap,
                       const __grid_constant__ CUtensorMap xmap, const FrontFusedParams p) {
  constexpr int NC = 16 * NXB;  // MMA N = accumulator columns = token columns
  constexpr uint32_t STAGE = 16384u + NXB * 2048u;
  // two accumulators (even and odd k-blocks, one MMA-issuing warp each)
  constexpr uint32_t TMEM_COLS = 2 * NC < 32 ? 32u : static_cast<uint32_t>(2 * NC);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int S = p.S, nsl = p.nsl, nst = p.nst;
  uint8_t *ring = smem;                                           // nst stages
  float *recv = reinterpret_cast<float *>(smem + nst * STAGE);      // [S][128][nsl]
  uint64_t *full = reinterpret_cast<uint64_t *>(recv + S * nsl * 128);  // [nst]
  uint64_t *empty = full + nst;                                   // [nst]
  uint64_t *acc_full = empty + nst;   // both accumulators final (two commits)
  uint64_t *recv_bar = acc_full + 1;  // this CTA's tokens: every sender's rows landed
  uint64_t *sent_bar = recv_bar + 1;  // every destination has received this CTA's rows
  uint64_t *drain = sent_bar + 1;     // [2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 2);
  volatile int *flags = reinterpret_cast<volatile int *>(tmem_slot + 1);  // [0] abort [1] last

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = static_cast<int>(cluster_ctarank());
  const int t = blockIdx.x >> p.log2S;
  const int kb0 = (c * p.KB) >> p.log2S, kb1 = ((c + 1) * p.KB) >> p.log2S;
  const int nkb = kb1 - kb0;  // >= 1: S <= KB
  // tokens owned by this CTA: b = c, c + S, c + 2S, ... < B
  const int nslc = (c < p.B) ? ((p.B - 1 - c) >> p.log2S) + 1 : 0;
  const int ndst = p.B < S ? p.B : S;  // CTAs of the cluster that own tokens
  // a receive area holds nsl slots per (sender, row); with 16-CTA clusters one vector
  // store per destination fills all of them, otherwise only the receiver's own tokens
  const int recv_slots = (S == 16) ? nsl : nslc;
  const int nissue = (nst & 1) ? 1 : 2;  // MMA-issuing warps (each owns every other stage)

  if (tid == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 2);
    mbar_init(recv_bar, 1);
    mbar_init(sent_bar, static_cast<uint32_t>(ndst));
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
    if (nslc > 0)
      mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>(S * 128 * recv_slots * 4));
    else
      mbar_arrive(recv_bar);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Every thread arrives (release: the barrier initialisations above) and waits before
  // its first access to another CTA of the cluster, so nothing reaches a CTA whose
  // barriers are not initialised yet.
  cluster_arrive_release();

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&wmap);
      prefetch_tensormap(&xmap);
      const uint64_t pol = policy_evict_first();
      const int pre = nkb < nst ? nkb : nst;
      for (int q = 0; q < pre; ++q) {  // weights only: they do not depend on earlier kernels
        mbar_arrive_expect_tx(&full[q], STAGE);
        tma_load_2d_hint(ring + q * STAGE, &wmap, &full[q], (kb0 + q) * TILE_K,
                                t * TILE_N, pol);
      }
      for (int kb = kb0 + pre; kb < kb1; ++kb) tma_prefetch_l2_2d(&wmap, kb * TILE_K, t * TILE_N);
      // the next kernel may start loading (router CTAs with trig_late: once routed)
      if (!(p.trig_late && t < p.TR)) griddep_launch_dependents();
      griddep_wait();
      bool ok = true;
      int q = 0;
      for (; q < nkb; ++q) {
        const int st = q % nst;
        uint8_t *dst = ring + st * STAGE;
        if (q >= pre) {
          if (!mbar_wait_bounded(&empty[st], ((q / nst) & 1) ^ 1, p.status, flags,
                                 p.wait_limit_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[st], STAGE);
          tma_load_2d_hint(dst, &wmap, &full[st], (kb0 + q) * TILE_K, t * TILE_N, pol);
        }
        tma_load_2d(dst + 16384, &xmap, &full[st], (kb0 + q) * TILE_K, 0);
      }
      if (!ok) {  // after a time-out: let this CTA's copies in flight land before exit
        const int q0 = q > nst ? q - nst : 0;
        for (int qq = q0; qq < q; ++qq)
          (void)mbar_wait_drain(&full[qq % nst], (qq / nst) & 1, 10000000ull);
      }
    }
    if (lane != 0) griddep_wait();
    cluster_wait();
  } else if (warp == 1 || warp == 2) {
    // --------------------------------------------------------------- MMA issuers
    // Warp 1 takes the even k-blocks into accumulator 0, warp 2 the odd ones into
    // accumulator 1: one thread issues a tcgen05.mma about every 100 cycles, two
    // threads overlap their issue. The ring depth is even, so every stage belongs to
    // one issuer, which waits on each of its fills in turn (a parity wait never runs
    // ahead of a fill it has not seen). Every warp sleeps in the dependency wait before it
    // polls an mbarrier: the next kernel of the stream is resident on the same SMs
    // early, and polling warps there would take issue slots from this one's tail.
    griddep_wait();
    if (lane == 0) {
      const int me = warp - 1;
      const uint32_t idesc = idesc_bf16(NC);
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(me * NC);
      bool ok = true;
      // an odd ring depth (not planned) falls back to one issuer
      for (int q = me; q < nkb && (me < nissue); q += nissue) {
        const int st = q % nst;
        if (!mbar_wait_bounded(&full[st], (q / nst) & 1, p.status, flags, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(ring + st * STAGE);
        const uint64_t adesc = sw128_desc(a_addr);
        const uint64_t bdesc = sw128_desc(a_addr + 16384u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // K = 16 per MMA: +32 bytes along the swizzled row
          tc_mma(d_tmem, adesc + 2u * kk, bdesc + 2u * kk, idesc, (q > me || kk > 0) ? 1u : 0u);
        tc_commit(&empty[st]);  // the stage is free once these MMAs have read it
      }
      if (ok) {
        tc_commit(acc_full);  // this accumulator is final (also when it got no k-block)
      } else {
        tc_commit(&drain[me]);  // let the MMAs issued so far finish before memory is freed
        (void)mbar_wait_drain(&drain[me], 0u, 10000000ull);
      }
    }
    cluster_wait();
  } else if (warp >= 4) {
    // ----------------------------------------------------------------- epilogue
    // Thread r holds row r of the partial tile for every token column. Token b's value
    // goes to CTA b % S of the cluster, into its receive area [src][row][slot] at slot
    // b / S: with 16-CTA clusters one vector store per destination carries every slot.
    const int r = 32 * (warp & 3) + lane;  // tile row == tensor-memory lane
    griddep_wait();
    (void)mbar_wait_bounded(acc_full, 0u, p.status, flags, p.wait_limit_ns);
    named_bar_sync(2, 128);
    const bool go = !flags[0];  // uniform across the 128 epilogue threads after the barrier
    float v[NC];
    if (go) {
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
      float v1[NC];
#pragma unroll
      for (int cc = 0; cc < NC / 16; ++cc) {
        tmem_ld16(taddr + 16u * cc, v + 16 * cc);
        tmem_ld16(taddr + static_cast<uint32_t>(NC) + 16u * cc, v1 + 16 * cc);
      }
      tmem_wait_ld();
      const bool two = nissue == 2 && nkb > 1;  // accumulator 1: odd k-blocks (or unwritten)
#pragma unroll
      for (int j = 0; j < NC; ++j) v[j] = two ? v[j] + v1[j] : v[j];
    }
    tc_fence_before();
    cluster_wait();
    if (go) {
      const uint32_t row_off = static_cast<uint32_t>((c * 128 + r) * nsl * 4);
      if (S == 16) {
#pragma unroll
        for (int d = 0; d < 16; ++d) {
          if (d < ndst) {
            const uint32_t dst = cluster_map(recv, static_cast<uint32_t>(d)) + row_off;
            const uint32_t mb = cluster_map(recv_bar, static_cast<uint32_t>(d));
            if (NXB == 1) st_async_f32(dst, v[d], mb);
            if (NXB == 2) st_async_v2(dst, v[d], v[(d + 16) % NC], mb);
            if (NXB == 4)
              st_async_v4(dst, v[d], v[(d + 16) % NC], v[(d + 32) % NC], v[(d + 48) % NC], mb);
          }
        }
      } else {
#pragma unroll
        for (int b = 0; b < NC; ++b) {
          if (b < p.B) {
            const uint32_t d = static_cast<uint32_t>(b & (S - 1));
            st_async_f32(cluster_map(recv, d) + row_off + 4u * static_cast<uint32_t>(b >> p.log2S),
                         v[b], cluster_map(recv_bar, d));
          }
        }
      }
    }
  } else {
    griddep_wait();
    cluster_wait();  // warp 3: nothing to do until the tokens arrive
  }

  // ------------------------------------------ this CTA's tokens: reduce, publish
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
  const bool router = t < p.TR;
  if (nslc > 0) {
    (void)mbar_wait_bounded(recv_bar, 0u, p.status, flags, p.wait_limit_ns);
    for (int q = tid; q < nslc * 128; q += FF_THREADS) {
      const int rr = q / nslc, j = q - rr * nslc;
      float z = 0.f;
      for (int src = 0; src < S; ++src) z += recv[(src * 128 + rr) * nsl + j];  // CTA order
      const int b = c + (j << p.log2S), n = t * TILE_N + rr;
      if (n < p.E)
        p.logits[static_cast<size_t>(b) * p.E + n] = z;
      else if (n < p.E + p.L)
        p.latent[static_cast<size_t>(b) * p.L + (n - p.E)] = f32_to_bf16_rn(z);
    }
    // tell every sender its rows have landed (it may exit once all its receivers did)
    if (tid < S) mbar_arrive_remote(cluster_map(sent_bar, static_cast<uint32_t>(tid)));
  }
  __syncthreads();
  // ------------------------------------------------- routing: last router CTA(s)
  // Up to p.single_b tokens one arrival counter elects the last router CTA, which routes
  // every token (a warp per token) and builds the route map. Beyond, the three (TR)
  // router CTAs owning a token group (the same cluster rank) elect their last one, which
  // routes that group; a second counter over the groups elects the CTA that builds the
  // route map from the published top-k ids.
  // With trig_late the router CTAs let the next kernel start only here (a CTA that exits
  // counts as triggered; a routing warp triggers once its logits are loaded): the next
  // kernel's burst of weight loads would otherwise queue in front of these L2 reads.
  const bool single = p.B <= p.single_b;
  int *cnt_all = p.counter;           // [0]: every router CTA (single) / every group
  int *cnt_grp = p.counter + 1 + c;   // [1 + c]: the TR router CTAs of group c
  if (router && nslc > 0 && tid == 0)
    flags[1] = single ? (atom_add_acq_rel_gpu(cnt_all, 1) == p.TR * ndst - 1)
                      : (atom_add_acq_rel_gpu(cnt_grp, 1) == p.TR - 1);
  __syncthreads();
  if (!flags[1]) {
    if (tid == 0) (void)mbar_wait_bounded(sent_bar, 0u, p.status, flags, p.wait_limit_ns);
    return;
  }
  // routing and route-map scratch in the idle stage ring
  int32_t *sidx = reinterpret_cast<int32_t *>(ring);                      // [B*topk]
  unsigned long long *smask =
      reinterpret_cast<unsigned long long *>(sidx + MAX_B * MAX_TOPK);   // [E]
  int *soff = reinterpret_cast<int *>(smask + MAX_E);                     // [E]
  int *swarp = soff + MAX_E;                                              // [16]
  uint64_t *rscr = reinterpret_cast<uint64_t *>(swarp + 16) +
                   warp * (RT_CMAX + MAX_TOPK);                           // [8][RT_CMAX+16]
  const int topk = p.topk;
  // this CTA's tokens: every token (single), else the group's b = c + j*S
  const int ntok = single ? p.B : nslc;
  for (int j = warp; j < ntok; j += FF_THREADS / 32) {
    const int b = single ? j : c + (j << p.log2S);
    const float *lg = p.logits + static_cast<size_t>(b) * p.E;
    int32_t *si = single ? sidx + b * topk : nullptr;
    if (p.probs != nullptr) {  // the full softmax as well
      if (p.trig_late && lane == 0) griddep_launch_dependents();
      route_token_sorted(lg, p.E, topk, p.topk_idx + b * topk, p.topk_w + b * topk,
                         p.probs + static_cast<size_t>(b) * p.E, si);
    } else {
      if (p.E <= 12 * 32)
        route_token_filtered<12>(lg, p.E, topk, p.topk_idx + b * topk, p.topk_w + b * topk,
                                 si, rscr, p.trig_late != 0);
      else
        route_token_filtered<16>(lg, p.E, topk, p.topk_idx + b * topk, p.topk_w + b * topk,
                                 si, rscr, p.trig_late != 0);
    }
  }
  if (single) {
    if (tid == 0) *cnt_all = 0;  // every arrival of this call is in: ready for the next
    __syncthreads();
    if (p.route_map != nullptr)
      build_route_map_cta(sidx, p.B, topk, p.E, p.route_map, smask, soff, swarp);
  } else {
    if (tid == 0) *cnt_grp = 0;
    __syncthreads();
    if (tid == 0) flags[1] = (atom_add_acq_rel_gpu(cnt_all, 1) == ndst - 1);
    __syncthreads();
    if (flags[1]) {
      if (tid == 0) *cnt_all = 0;
      const int P = p.B * topk;
      for (int q = tid; q < P; q += FF_THREADS) sidx[q] = __ldcg(p.topk_idx + q);
      __syncthreads();
      if (p.route_map != nullptr)
        build_route_map_cta(sidx, p.B, topk, p.E, p.route_map, smask, soff, swarp);
    }
  }
  // every receiver has taken this CTA's rows (and nothing else targets it) before exit
  if (tid == 0) (void)mbar_wait_bounded(sent_bar, 0u, p.status, flags, p.wait_limit_ns);
}

template <int NXB>
cudaError_t launch_nxb(const CUtensorMap &wmap, const CUtensorMap &xmap,
                       const FrontFusedParams &p, size_t smem, cudaStream_t s) {
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(front_fused_kernel<NXB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             FRONT_FUSED_SMEM_MAX);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(front_fused_kernel<NXB>,
                               cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  return launch_pdl_cluster(front_fused_kernel<NXB>, dim3(p.T * p.S), dim3(FF_THREADS), smem, s,
                            p.S, wmap, xmap, p);
}

template <int NXB>
int max_clusters_nxb(int S, size_t smem) {
  if (cudaFuncSetAttribute(front_fused_kernel<NXB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           FRONT_FUSED_SMEM_MAX) != cudaSuccess ||
      cudaFuncSetAttribute(front_fused_kernel<NXB>,
                           cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S);
  cfg.blockDim = dim3(FF_THREADS);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(S);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, front_fused_kernel<NXB>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace

size_t front_fused_smem(int S, int nxb, int nst, int nsl) {
  const size_t stage = 16384 + static_cast<size_t>(nxb) * 2048;
  return 1024 + nst * stage + static_cast<size_t>(S) * nsl * 512 + (2 * nst + 5) * 8 + 64;
}

int front_fused_max_clusters(int S, int nxb, size_t smem) {
  switch (nxb) {
    case 1: return max_clusters_nxb<1>(S, smem);
    case 2: return max_clusters_nxb<2>(S, smem);
    case 4: return max_clusters_nxb<4>(S, smem);
    default: return 0;
  }
}

cudaError_t launch_front_fused(const CUtensorMap &wmap, const CUtensorMap &xmap,
                               const FrontFusedParams &p, int nxb, size_t smem, cudaStream_t s) {
  switch (nxb) {
    case 1: return launch_nxb<1>(wmap, xmap, p, smem, s);
    case 2: return launch_nxb<2>(wmap, xmap, p, smem, s);
    case 4: return launch_nxb<4>(wmap, xmap, p, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ssd
