// engine_pair.cu -- wide projections (65-512 rows per call) on CTA-pair tensor-core
// tiles.
//
// Speculative-decode verification multiplies one weight matrix by many activation rows
// (sequences x (draft length + 1) tokens). With one CTA per 128-row weight tile, every
// tile re-reads all M activation rows from L2 (M x 128 bytes per 16 KB of weights per
// k-block), and from M = 128 on those bytes, not the weights, bound each SM. Here two CTAs
// share one MMA (tcgen05 .cta_group::2, M = 256 weight rows): each CTA stages its own 128
// weight rows and half of the activation rows of every k-block, so each SM receives half
// the activation bytes per weight byte, and a 512-row call is one launch that reads W
// once.
//
// One cluster of 4 CTAs per 256-row slice of W (weight tiles 2c and 2c+1):
//   rank 0: tile 2c,   k-half 0  -- issues the pair MMA of ranks 0 and 1
//   rank 1: tile 2c+1, k-half 0
//   rank 2: tile 2c,   k-half 1  -- issues the pair MMA of ranks 2 and 3
//   rank 3: tile 2c+1, k-half 1
// A launch covers NCOL = 128..512 batch columns (a multiple of 64) as NMMA MMAs of N = NPER
// per K step (one of NCOL up to 256, else two of NCOL / 2). Per k-block each CTA loads its 16 KB weight box
// and NMMA activation boxes of NPER / 2 rows (rows NPER m + (NPER / 2) h .. for MMA m,
// h = rank & 1), so MMA m covers batch columns NPER m .. NPER m + NPER - 1 (rows beyond
// the batch read as zeros). Batch column j accumulates in tensor-memory column j.
//
// Ring: the even CTA's full barrier of a stage counts both CTAs' bytes (the odd CTA's
// copies signal it through the CTA-pair form of the TMA load); the MMA thread arms each
// stage's next fill when it consumes the current one, so every copy either CTA issues
// lands on an armed phase; the commit that frees a stage arrives on the empty barriers of
// both CTAs (multicast), and after the last k-block a multicast commit tells both CTAs
// that their accumulators are final.
//
// Tail: the two k-halves of a weight tile are ranks r and r ^ 2. k-half 0 finishes batch
// columns [0, NCOL / 2), k-half 1 the rest. Once every CTA of the cluster is past its
// MMAs (cluster barrier 1: every ring is idle), each CTA writes the partner's columns of
// its accumulator into the partner's ring; after cluster barrier 2 each adds its own half
// to the received one (+ R, loaded as one TMA tile meanwhile), rounds once to bf16 into a
// tile in its ring, releases tensor memory and writes the tile to Y with one TMA store
// (rows of Y not 16-byte aligned: per-thread stores). No partial tile goes through
// global memory and no counter is used.
#include <atomic>

#include "engine.cuh"
#include "tcgen05.cuh"

namespace ssd {

namespace {

constexpr int PAIR_THREADS = 192;  // warp 0 TMA, warp 1 MMA + tensor memory, warps 2-5 tail
constexpr int PAIR_SMEM_LIMIT = 232448;

// NCOL batch columns per launch (a multiple of 64 from 128 to 512): NMMA MMAs of N = NPER
// per K step, each CTA of a pair staging XROWS = NPER / 2 activation rows per MMA. Every
// box and stage starts on a 1024-byte boundary (XBYTES is a multiple of 1024), as the
// 128-byte swizzle of the TMA copies and of the MMA descriptors requires.
template <int NCOL>
struct PairConfig {
  static constexpr int NMMA = NCOL > 256 ? 2 : 1;
  static constexpr int NPER = NCOL / NMMA;
  static constexpr int XROWS = NPER / 2;
  static constexpr int XBYTES = XROWS * 128;
  static constexpr int STAGE_BYTES = 16384 + NMMA * XBYTES;
  static constexpr int TAIL = 256;
  static constexpr int FIT = (PAIR_SMEM_LIMIT - 1024 - TAIL) / STAGE_BYTES;
  static constexpr int STAGES = FIT > 8 ? 8 : FIT;
  static constexpr int HALF = NCOL / 2;              // batch columns one k-half finishes
  static constexpr uint32_t TMEM_COLS = NCOL <= 128 ? 128u : (NCOL <= 256 ? 256u : 512u);
  static constexpr int RECV_BYTES = HALF * 128 * 4;  // the partner's partial of them
  static constexpr int TILE_BYTES = HALF * 128 * 2;  // R in, Y out: bf16 [HALF][128]
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + TAIL;
  static_assert(STAGES >= 4, "pipeline too shallow");
  static_assert(HALF % 32 == 0, "the tail moves whole groups of 32 columns");
  static_assert(NPER % 32 == 0 && NPER <= 256, "CTA-pair MMA: N a multiple of 32, <= 256");
  static_assert(RECV_BYTES + TILE_BYTES <= STAGES * STAGE_BYTES, "tail does not fit the ring");
  static_assert(XBYTES % 1024 == 0, "activation boxes on 1024-byte boundaries");
};

// The weight box of tile t, k-block kb (row-major W, or the tile-packed 16 KB block).
__device__ __forceinline__ void pair_load_w(const EngineParams &p, const CUtensorMap *wmap,
                                            uint8_t *dst, uint32_t bar, int t, int kb,
                                            uint64_t pol) {
  if (p.packed)
    tma_load_2d_pair_hint(dst, wmap, bar, 0, (t * p.KB + kb) * TILE_N, pol);
  else
    tma_load_2d_pair_hint(dst, wmap, bar, kb * TILE_K, t * TILE_N, pol);
}

template <int NCOL>
__global__ void __launch_bounds__(PAIR_THREADS, 1)
    engine_pair_kernel(const __grid_constant__ CUtensorMap wmap,
                       const __grid_constant__ CUtensorMap xmap,
                       const __grid_constant__ CUtensorMap ymap,
                       const __grid_constant__ CUtensorMap rmap, const EngineParams p) {
  using C = PairConfig<NCOL>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *ring = smem;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t *empty = full + C::STAGES;
  uint64_t *acc_full = empty + C::STAGES;
  uint64_t *drain = acc_full + 1;
  uint64_t *rbar = drain + 1;  // the residual tile has landed
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(rbar + 1);
  volatile int *flags = reinterpret_cast<volatile int *>(tmem_slot + 1);  // [0] abort

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t h = rank & 1u;      // weight tile of the slice
  const uint32_t kh = rank >> 1;     // k-half
  const uint32_t lead = rank & ~1u;  // the pair's MMA-issuing CTA
  const bool leader = h == 0;
  const int t = 2 * static_cast<int>(blockIdx.x >> 2) + static_cast<int>(h);
  const int kb0 = (static_cast<int>(kh) * p.KB) >> 1;
  const int nkb = (((static_cast<int>(kh) + 1) * p.KB) >> 1) - kb0;  // >= 1: KB >= 2

  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    mbar_init(rbar, 1);
    flags[0] = 0;
    // the even CTA arms the first fill of every stage for both CTAs' bytes
    if (leader)
      for (int s = 0; s < C::STAGES && s < nkb; ++s)
        mbar_arrive_expect_tx(&full[s], 2u * C::STAGE_BYTES);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // every CTA of the cluster has initialised and armed its barriers before a copy or a
  // commit of another CTA can signal one
  cluster_sync_all();

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tensormap(&wmap);
      prefetch_tensormap(&xmap);
      const uint64_t pol = policy_evict_first();  // weights are read once per launch
      const uint32_t bar0 = cluster_map(full, lead);  // the pair's full barriers
      const int pre = nkb < C::STAGES ? nkb : C::STAGES;
      for (int q = 0; q < pre; ++q)  // weights only: they do not depend on earlier kernels
        pair_load_w(p, &wmap, ring + q * C::STAGE_BYTES, bar0 + 8u * q, t, kb0 + q, pol);
      griddep_wait();
      for (int q = 0; q < nkb; ++q) {
        const int st = q % C::STAGES;
        uint8_t *dst = ring + st * C::STAGE_BYTES;
        const uint32_t bar = bar0 + 8u * static_cast<uint32_t>(st);
        if (q >= pre) {
          if (!mbar_wait_bounded(&empty[st], ((q / C::STAGES) & 1) ^ 1, p.status, flags,
                                 p.wait_limit_ns))
            break;
          pair_load_w(p, &wmap, dst, bar, t, kb0 + q, pol);
        }
#pragma unroll
        for (int m = 0; m < C::NMMA; ++m)
          tma_load_2d_pair(dst + 16384 + m * C::XBYTES, &xmap, bar, (kb0 + q) * TILE_K,
                           C::NPER * m + C::XROWS * static_cast<int>(h));
      }
      // every load of this CTA is issued: the next kernel may be scheduled as SMs free up
      griddep_launch_dependents();
    } else {
      griddep_wait();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    griddep_wait();
    if (leader && lane == 0) {
      const uint32_t idesc = idesc_bf16_pair(C::NPER);
      const uint16_t mask = static_cast<uint16_t>(3u << lead);
      bool ok = true;
      int q = 0;
      for (; q < nkb; ++q) {
        const int st = q % C::STAGES;
        if (!mbar_wait_bounded(&full[st], (q / C::STAGES) & 1, p.status, flags,
                               p.wait_limit_ns)) {
          ok = false;
          break;
        }
        // arm the stage's next fill (both CTAs issue it only after this stage is freed)
        if (q + C::STAGES < nkb) mbar_arrive_expect_tx(&full[st], 2u * C::STAGE_BYTES);
        tc_fence_after();
        const uint32_t a_addr = smem_u32(ring + st * C::STAGE_BYTES);
        const uint64_t adesc = sw128_desc(a_addr);
#pragma unroll
        for (int m = 0; m < C::NMMA; ++m) {
          const uint64_t bdesc = sw128_desc(a_addr + 16384u + static_cast<uint32_t>(m * C::XBYTES));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // K = 16 per MMA: +32 bytes along the swizzled row
            tc_mma_pair(tmem_base + static_cast<uint32_t>(C::NPER * m), adesc + 2u * kk,
                        bdesc + 2u * kk, idesc,
                        (q > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit_pair_mc(&empty[st], mask);  // both CTAs' stage is free once read
      }
      if (ok) {
        tc_commit_pair_mc(acc_full, mask);  // both accumulators final
      } else {
        // after a time-out: let the MMAs issued so far finish, then the copies of both
        // CTAs into the stages armed but not consumed, before any memory is released
        tc_commit_pair(drain);
        (void)mbar_wait_drain(drain, 0u, 10000000ull);
        const int qe = q + C::STAGES < nkb ? q + C::STAGES : nkb;
        for (int qq = q; qq < qe; ++qq)
          (void)mbar_wait_drain(&full[qq % C::STAGES], (qq / C::STAGES) & 1u, 10000000ull);
      }
    }
  } else {
    griddep_wait();
    (void)mbar_wait_bounded(acc_full, 0u, p.status, flags, p.wait_limit_ns);
  }

  // ---------------------------------------------------------------------- tail
  tc_fence_before();
  __syncthreads();
  const bool go = !flags[0];  // uniform across the CTA after the barrier
  // 1: every CTA of the cluster is past its MMAs (or gave up): every ring is idle
  cluster_sync_all();
  tc_fence_after();
  float *recv = reinterpret_cast<float *>(ring);                        // [HALF][128] fp32
  uint16_t *tile = reinterpret_cast<uint16_t *>(ring + C::RECV_BYTES);  // [HALF][128] bf16
  const int own0 = static_cast<int>(kh) * C::HALF;  // first batch column this CTA finishes
  const int oth0 = C::HALF - own0;                  // the partner's
  const int r = 32 * (warp & 3) + lane;             // tile row == tensor-memory lane
  const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
  // Y (and R) as whole tiles by TMA when their rows are 16-byte aligned: per-thread
  // stores from every SM at once are limited by the stores each SM keeps in flight
  const bool tma_out = p.vec_y != 0;
  if (go && tma_out && p.R != nullptr && tid == 64) {
    mbar_arrive_expect_tx(rbar, static_cast<uint32_t>(C::HALF * 128 * 2));
    tma_load_2d(tile, &rmap, rbar, t * TILE_N, own0);
  }
  if (go && warp >= 2) {
    const uint32_t dst = cluster_map(recv, rank ^ 2u) + 4u * static_cast<uint32_t>(r);
    // CG columns per tensor-memory wait: the loads' latency is paid once per group
    constexpr int CG = C::HALF % 64 == 0 ? 64 : 32;
    for (int c = 0; c < C::HALF && oth0 + c < p.B; c += CG) {
      float v[CG];
#pragma unroll
      for (int q = 0; q < CG / 16; ++q)
        tmem_ld16(taddr + static_cast<uint32_t>(oth0 + c + 16 * q), v + 16 * q);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < CG; ++j) st_cluster_f32(dst + 512u * static_cast<uint32_t>(c + j), v[j]);
    }
  }
  tc_fence_before();
  // 2: the partner's columns have landed in this CTA's ring
  cluster_sync_all();
  tc_fence_after();
  if (go && warp >= 2) {
    // this CTA's columns: its own k-half plus the received one (+ R), rounded once
    const bool res = tma_out && p.R != nullptr;
    if (res && !mbar_wait_bounded(rbar, 0u, p.status, flags, p.wait_limit_ns))
      (void)mbar_wait_drain(rbar, 0u, 10000000ull);  // the copy lands before the CTA exits
    // 32 columns at a time, every shared-memory read of the group before its writes (the
    // compiler cannot tell the areas apart, so interleaved they would run one by one)
    for (int c = 0; c < C::HALF && own0 + c < p.B; c += 32) {
      float v[32], o[32];
      tmem_ld16(taddr + static_cast<uint32_t>(own0 + c), v);
      tmem_ld16(taddr + static_cast<uint32_t>(own0 + c + 16), v + 16);
#pragma unroll
      for (int j = 0; j < 32; ++j) o[j] = recv[(c + j) * 128 + r];
      if (res) {
        uint16_t rb[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) rb[j] = tile[(c + j) * 128 + r];
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j)
          tile[(c + j) * 128 + r] = f32_to_bf16_rn((v[j] + o[j]) + bf16_to_f32(rb[j]));
      } else {
        tmem_wait_ld();
        if (tma_out) {
#pragma unroll
          for (int j = 0; j < 32; ++j) tile[(c + j) * 128 + r] = f32_to_bf16_rn(v[j] + o[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) recv[(c + j) * 128 + r] = v[j] + o[j];
        }
      }
    }
    if (tma_out) fence_proxy_async_smem();  // the tile is read by the TMA store next
  }
  // the accumulator is read: release tensor memory before the stores
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  if (go && tma_out && !flags[0]) {
    if (tid == 64) {
      tma_store_2d(&ymap, tile, t * TILE_N, own0);  // rows >= B, columns >= N clipped
      bulk_commit_group();
      bulk_wait_all();
    }
  } else if (go && warp >= 2) {
    const int ncol = min(C::HALF, p.B - own0);  // columns of the batch this CTA stores
    for (int c = r; c < ncol * 16; c += 128) {
      const int j = c >> 4, row8 = (c & 15) * 8;
      const int col = own0 + j, n0 = t * TILE_N + row8;
      if (n0 >= p.N) continue;
      const float *src = recv + j * 128 + row8;
      for (int e = 0; e < 8 && n0 + e < p.N; ++e) {
        float y = src[e];
        const size_t off = static_cast<size_t>(col) * p.N + n0 + e;
        if (p.R != nullptr) y += bf16_to_f32(p.R[off]);
        p.Y[off] = f32_to_bf16_rn(y);
      }
    }
  }
}

template <int NCOL>
cudaError_t set_pair_attrs() {
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(engine_pair_kernel<NCOL>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, PairConfig<NCOL>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  return cudaSuccess;
}

template <int NCOL>
cudaError_t launch_pair_t(const CUtensorMap &wmap, const CUtensorMap &xmap,
                          const CUtensorMap &ymap, const CUtensorMap &rmap, const EngineParams &p,
                          cudaStream_t s) {
  cudaError_t e = set_pair_attrs<NCOL>();
  if (e != cudaSuccess) return e;
  const int slices = (p.T + 1) / 2;
  return launch_pdl_cluster(engine_pair_kernel<NCOL>, dim3(4 * slices), dim3(PAIR_THREADS),
                            PairConfig<NCOL>::SMEM, s, 4, wmap, xmap, ymap, rmap, p);
}

template <int NCOL>
cudaError_t max_clusters_t(int *n) {
  cudaError_t e = set_pair_attrs<NCOL>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(4 * 64);
  cfg.blockDim = dim3(PAIR_THREADS);
  cfg.dynamicSmemBytes = PairConfig<NCOL>::SMEM;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeClusterDimension;
  a[0].val.clusterDim.x = 4;
  a[0].val.clusterDim.y = 1;
  a[0].val.clusterDim.z = 1;
  cfg.attrs = a;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(n, engine_pair_kernel<NCOL>, &cfg);
}

}  // namespace

int pair_cols(int B) { return B <= 128 ? 128 : (B + 63) / 64 * 64; }

cudaError_t engine_pair_max_clusters(int ncol, int *n) {
  switch (ncol) {
    case 128: return max_clusters_t<128>(n);
    case 192: return max_clusters_t<192>(n);
    case 256: return max_clusters_t<256>(n);
    case 320: return max_clusters_t<320>(n);
    case 384: return max_clusters_t<384>(n);
    case 448: return max_clusters_t<448>(n);
    default: return max_clusters_t<512>(n);
  }
}

cudaError_t launch_engine_pair(int ncol, const CUtensorMap &wmap, const CUtensorMap &xmap,
                               const CUtensorMap &ymap, const CUtensorMap &rmap,
                               const EngineParams &p, cudaStream_t s) {
  if (p.mode != MODE_LINEAR || p.grouped || p.KB < 2 || p.T < 1 || p.B < 1 || p.B > ncol ||
      ncol < 128 || ncol > 512 || ncol % 64 != 0)
    return cudaErrorNotSupported;
  switch (ncol) {
    case 128: return launch_pair_t<128>(wmap, xmap, ymap, rmap, p, s);
    case 192: return launch_pair_t<192>(wmap, xmap, ymap, rmap, p, s);
    case 256: return launch_pair_t<256>(wmap, xmap, ymap, rmap, p, s);
    case 320: return launch_pair_t<320>(wmap, xmap, ymap, rmap, p, s);
    case 384: return launch_pair_t<384>(wmap, xmap, ymap, rmap, p, s);
    case 448: return launch_pair_t<448>(wmap, xmap, ymap, rmap, p, s);
    default: return launch_pair_t<512>(wmap, xmap, ymap, rmap, p, s);
  }
}

}  // namespace ssd
