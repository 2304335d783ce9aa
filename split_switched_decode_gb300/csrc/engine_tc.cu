// engine_tc.cu -- split-K engine with tcgen05 tensor-core tiles ("swap-AB").
//
// Same schedule, TMA staging, reduction and epilogues as engine_cc.cu (engine.cuh);
// only the multiply differs. The weight tile is the MMA A operand (M = 128 rows) and
// the activation rows are the B operand (N = 16 x boxes = 16..64 columns), both
// K-major with the 128-byte swizzle exactly as TMA wrote them, so no data is
// rearranged in shared memory. One CTA per SM, warp-specialised:
//
//   warp 0     TMA producer (lane 0): weight + activation boxes into an 8-deep ring
//   warp 1     tensor-memory owner and MMA issuer (lane 0): 4 x tcgen05.mma
//              (M128 x N x K16) per 64-wide k-block into an fp32 accumulator in
//              tensor memory; tcgen05.commit frees the stage when those MMAs finish
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (warp w reads lanes
//              32*(w%4)..+31 = tile rows), then the split-K reduction and epilogue
//
// The accumulator is double-buffered (2 x 64 columns) so the epilogue of one segment
// overlaps the MMAs of the next. The tensor cores keep the multiply off the CUDA
// cores, which would bound the CUDA-core tiles from about 8 batch columns upward.
//
// Wide projections (speculative-decode verification: B x (draft length + 1) rows, up
// to 256): NG groups of 64 batch columns share every weight tile -- one MMA with
// N = 16 x boxes <= 256 per K step into 2 x 64*NG accumulator columns (all 512 at
// NG = 4) -- and the epilogue reduces and stores the column groups one after another,
// each with its own partial slots and arrival counter.
//
// Whole-tile schedule (p.dyn, grouped launches): each CTA streams a static share of whole
// tiles and claims the rest one at a time from a counter. engine_tc_moe_kernel (below)
// runs the routed experts' gate/up and down, and by default the shared expert's, as one
// launch of claimed whole tiles.
//
// Pair schedule (p.pair): every tile is split into exactly two k-halves and the two
// workers of a tile run as a 2-CTA cluster. Instead of partial tiles in global memory
// and an arrival counter, each CTA hands the partner the accumulator columns the
// partner finishes through distributed shared memory (the epilogue scratch, or for
// wide tiles the idle stage buffers once both CTAs are past their MMAs) and, after a
// cluster barrier, adds first half + second half for its own columns -- the same order
// as the global reduction -- and stores Y.
#include <atomic>

#include "engine.cuh"
#include "tcgen05.cuh"

namespace ssd {

namespace {

constexpr int TC_THREADS = 192;  // 6 warps
constexpr int TC_SMEM_LIMIT = 232448;
template <int MAXC, int NG>
struct TCConfig {
  static constexpr uint32_t TMEM_COLS = 128u * NG;  // two accumulators of 64*NG columns
  static constexpr int NC = MAXC < 16 ? 16 : MAXC;  // accumulator columns read back
  static constexpr int NXB = NC / 16 * NG;          // 16-row activation boxes per stage
  static constexpr int STAGE_BYTES = 16384 + NXB * 2048;
  static constexpr int SCRATCH_BYTES = 64 * MAXC * 4;  // gate/up pairing
  static constexpr int TAIL = 512;
  static constexpr int BUDGET = TC_SMEM_LIMIT - 1024 - TAIL;
  static constexpr int FIT = (BUDGET - SCRATCH_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = FIT > 8 ? 8 : FIT;
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + SCRATCH_BYTES + TAIL;
  static_assert(STAGES >= 4, "pipeline too shallow");
};

// MMA issuer (one thread): one segment's k-blocks into accumulator buffer seg % 2,
// 4 x tcgen05.mma (M128 x N x K16) per k-block; each stage is released by a commit once
// its MMAs have read it, and the accumulator by a commit after the last. False after a
// time-out.
template <int STAGES, int STAGE_BYTES, int NG>
__device__ __forceinline__ bool mma_segment(const SegInfo &s, uint32_t seg, uint32_t &q,
                                            uint32_t tmem_base, uint8_t *stage_mem,
                                            uint64_t *full, uint64_t *empty, uint64_t *acc_full,
                                            uint64_t *acc_empty, const EngineParams &p,
                                            volatile int *flags) {
  const uint32_t idesc = idesc_bf16(16 * seg_xboxes(s));
  const uint32_t buf = seg & 1u;
  if (!mbar_wait_bounded(&acc_empty[buf], ((seg >> 1) & 1u) ^ 1u, p.status, flags,
                         p.wait_limit_ns))
    return false;
  tc_fence_after();
  const uint32_t d_tmem = tmem_base + buf * 64u * NG;
  for (int kb = s.kb0; kb < s.kb1; ++kb, ++q) {
    const int st = static_cast<int>(q % STAGES);
    if (!mbar_wait_bounded(&full[st], (q / STAGES) & 1u, p.status, flags, p.wait_limit_ns))
      return false;
    tc_fence_after();
    const uint32_t a_addr = smem_u32(stage_mem + st * STAGE_BYTES);
    const uint64_t adesc = sw128_desc(a_addr);
    const uint64_t bdesc = sw128_desc(a_addr + 16384u);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)  // K = 16 per MMA: +32 bytes along the swizzled row
      tc_mma(d_tmem, adesc + 2u * kk, bdesc + 2u * kk, idesc, (kb > s.kb0 || kk > 0) ? 1u : 0u);
    tc_commit(&empty[st]);  // the stage is free once these MMAs have read it
  }
  tc_commit(&acc_full[buf]);  // accumulator ready for the epilogue
  return true;
}

template <int MAXC, int NG>
__global__ void __launch_bounds__(TC_THREADS, 1)
    engine_tc_kernel(const __grid_constant__ CUtensorMap wmap,
                     const __grid_constant__ CUtensorMap xmap, const EngineParams p) {
  using C = TCConfig<MAXC, NG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *stage_mem = smem;
  float *scratch = reinterpret_cast<float *>(smem + C::STAGES * C::STAGE_BYTES);
  uint8_t *tail = smem + C::STAGES * C::STAGE_BYTES + C::SCRATCH_BYTES;
  uint64_t *full = reinterpret_cast<uint64_t *>(tail);
  uint64_t *empty = full + C::STAGES;
  uint64_t *acc_full = empty + C::STAGES;   // [2]
  uint64_t *acc_empty = acc_full + 2;       // [2]
  uint64_t *drain = acc_empty + 2;          // [1]
  uint64_t *tready = drain + 1;             // [4] whole-tile schedule: slot written
  uint64_t *tfree = tready + 4;             // [4] whole-tile schedule: slot read
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tfree + 4);
  volatile int *flags = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *tslot = flags + 3;          // [4] tile of segment seg in slot seg % 4
  volatile int *etile = tslot + 4;          // [2] the epilogue's copy, by segment parity

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int w = blockIdx.x;
  // pair mode: this CTA's own half of the columns of its (single) segment
  constexpr int PH = MAXC >= 2 ? MAXC / 2 : 1;
  float keep[PH];
  int pair_t = 0, pair_ncols = 0;
  // a grouped launch reads the route map right away: wait for the previous kernel
  // unless the map was complete before that kernel started (rm_ready)
  if (p.grouped && !p.rm_ready) griddep_wait();
  const int ngroups = p.grouped ? rm_num_used(p) : 1;
  const int64_t total = static_cast<int64_t>(ngroups) * p.T * p.KB;
  const int64_t begin = sk_start(total, p.G, w);
  const int64_t end = sk_start(total, p.G, w + 1);

  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&tready[i], 1);
      mbar_init(&tfree[i], 2);  // the MMA issuer and epilogue thread 0
    }
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // pair mode: every thread arrives here and waits before this CTA's first store into
  // the partner's shared memory (epilogue warps: before their loop; producer and MMA
  // warps: after theirs), so no store reaches a CTA that has not started
  if (p.pair) cluster_arrive_relaxed();

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (!p.grouped) prefetch_weights_l2(p, begin, end, C::STAGES, lane);
    if (lane == 0 && p.dyn)
      engine_produce_dyn<C::STAGES, C::STAGE_BYTES>(p, &wmap, &xmap, stage_mem, full, empty,
                                                    tslot, tready, tfree, flags,
                                                    ngroups * p.T);
    else if (lane == 0)
      engine_produce<C::STAGES, C::STAGE_BYTES>(p, &wmap, &xmap, stage_mem, full, empty, flags,
                                                begin, end);
    else
      griddep_wait();
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    griddep_wait();
    if (lane == 0) {
      uint32_t q = 0;
      bool ok = true;
      if (p.dyn) {
        for (uint32_t seg = 0; ok; ++seg) {
          const int sl = static_cast<int>(seg & 3u);
          if (!mbar_wait_bounded(&tready[sl], (seg >> 2) & 1u, p.status, flags, p.wait_limit_ns))
            break;
          const int tile = tslot[sl];
          mbar_arrive(&tfree[sl]);
          if (tile < 0) break;
          SegInfo s;
          const int64_t it = static_cast<int64_t>(tile) * p.KB;
          seg_info(p, it, it + p.KB, s);
          ok = mma_segment<C::STAGES, C::STAGE_BYTES, NG>(s, seg, q, tmem_base, stage_mem, full,
                                                       empty, acc_full, acc_empty, p, flags);
        }
      } else {
        uint32_t seg = 0;
        for (int64_t it = begin; it < end && ok; ++seg) {
          SegInfo s;
          seg_info(p, it, end, s);
          ok = mma_segment<C::STAGES, C::STAGE_BYTES, NG>(s, seg, q, tmem_base, stage_mem, full,
                                                       empty, acc_full, acc_empty, p, flags);
          it += s.kb1 - s.kb0;
        }
      }
      if (flags[0]) {  // let every MMA issued so far finish before the memory is freed
        tc_commit(drain);
        (void)mbar_wait_drain(drain, 0u, 10000000ull);
      }
    }
  } else {
    // --------------------------------------------------------------- epilogue
    griddep_wait();
    if (p.pair) cluster_wait();
    const int r = 32 * (warp & 3) + lane;  // tile row == tensor-memory lane
    uint32_t seg = 0;
    // whole-tile schedule (grouped launches: one column group, no pair): thread 0 takes
    // each segment's tile from the producer's slot, waits for its accumulator and hands
    // the tile to the other 127 threads through etile across the barrier (so all take
    // the same branches); every segment is a whole tile, so there is no reduction
    for (; p.dyn; ++seg) {
      const int sl = static_cast<int>(seg & 3u);
      const uint32_t buf = seg & 1u;
      if (r == 0) {
        const bool got =
            mbar_wait_bounded(&tready[sl], (seg >> 2) & 1u, p.status, flags, p.wait_limit_ns);
        int t = (got && !flags[0]) ? tslot[sl] : -1;
        mbar_arrive(&tfree[sl]);
        if (t >= 0 && (!mbar_wait_bounded(&acc_full[buf], (seg >> 1) & 1u, p.status, flags,
                                          p.wait_limit_ns) ||
                       flags[0]))
          t = -1;
        etile[seg & 1u] = t;
      }
      named_bar_sync(2, 128);
      const int tile = etile[seg & 1u];
      if (tile < 0) break;
      SegInfo s;
      const int64_t it = static_cast<int64_t>(tile) * p.KB;
      seg_info(p, it, it + p.KB, s);
      tc_fence_after();
      float v[C::NC];
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + buf * 64u * NG;
#pragma unroll
      for (int c = 0; c < C::NC / 16; ++c) tmem_ld16(taddr + 16u * c, v + 16 * c);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
      float acc[MAXC];
#pragma unroll
      for (int j = 0; j < MAXC; ++j) acc[j] = v[j];
      epilogue_rows<MAXC>(p, s, r, acc, scratch, 2, flags);
    }
    for (int64_t it = begin; !p.dyn && it < end; ++seg) {
      SegInfo s;
      seg_info(p, it, end, s);
      const uint32_t buf = seg & 1u;
      (void)mbar_wait_bounded(&acc_full[buf], (seg >> 1) & 1u, p.status, flags, p.wait_limit_ns);
      named_bar_sync(2, 128);
      if (flags[0]) break;  // uniform across the 128 epilogue threads after the barrier
      tc_fence_after();
      if (NG > 1 && p.pair) {  // the accumulator stays in tensor memory for the pair tail
        pair_t = s.t;
        pair_ncols = s.ncols;
        it += s.kb1 - s.kb0;
        continue;
      }
      const int ng = NG == 1 ? 1 : (s.ncols + 63) >> 6;  // column groups of this segment
#pragma unroll 1
      for (int g = 0; g < ng; ++g) {
        float v[C::NC];
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * (warp & 3)) << 16) +
                               buf * 64u * NG + 64u * g;
#pragma unroll
        for (int c = 0; c < C::NC / 16; ++c) tmem_ld16(taddr + 16u * c, v + 16 * c);
        tmem_wait_ld();
        if (g == ng - 1) {  // every column group read: the buffer is free for the MMAs
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
        float acc[MAXC];
#pragma unroll
        for (int j = 0; j < MAXC; ++j) acc[j] = v[j];
        if (NG == 1 && p.pair) {
          // the two k-halves of the tile are this CTA and its cluster partner: send the
          // partner the columns it finishes, keep the ones this CTA finishes
          const uint32_t me = cluster_ctarank();
          const uint32_t dst = cluster_map(scratch, me ^ 1u) + 4u * r;
          if (me == 0) {  // keeps columns 0..PH-1, sends PH..2PH-1 (indices fixed per branch)
#pragma unroll
            for (int jj = 0; jj < PH; ++jj) {
              if (PH + jj < s.ncols) st_cluster_f32(dst + 512u * jj, acc[PH + jj]);
              keep[jj] = acc[jj];
            }
          } else {        // keeps PH..2PH-1, sends 0..PH-1
#pragma unroll
            for (int jj = 0; jj < PH; ++jj) {
              if (jj < s.ncols) st_cluster_f32(dst + 512u * jj, acc[jj]);
              keep[jj] = acc[PH + jj];
            }
          }
          pair_t = s.t;
          pair_ncols = s.ncols;
          continue;
        }
        SegInfo sg = s;
        if (NG > 1) {
          sg.cgrp = g;
          sg.xrow0 = 64 * g;
          sg.ncols = min(64, s.ncols - 64 * g);
        }
        if (reduce_tile<MAXC>(p, sg, total, w, begin, r, acc, 2, flags))
          epilogue_rows<MAXC>(p, sg, r, acc, scratch, 2, flags);
      }
      it += s.kb1 - s.kb0;
    }
  }
  if (p.pair && warp < 2) cluster_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (NG > 1 && p.pair) {
    // Wide pair tail. Column group g is finished by the CTA of rank g % 2 (rank 0: groups
    // 0 and 2, rank 1: groups 1 and 3). Once both CTAs are past their MMAs (barrier 1:
    // every stage buffer on both sides is idle), each reads its accumulator from tensor
    // memory group by group and puts it in its own stage memory (its groups) or in the
    // partner's (the partner's groups); after barrier 2 each adds first k-half + second
    // k-half for its groups, adds R, rounds once and stores.
    float *own = reinterpret_cast<float *>(stage_mem);           // [2][64][128]
    float *recv = reinterpret_cast<float *>(stage_mem + 65536);  // [2][64][128]
    const uint32_t me = cluster_ctarank();
    const int ng = (pair_ncols + 63) >> 6;
    cluster_sync_all();
    if (warp >= 2) {
      const int r = 32 * (warp & 3) + lane;
      const uint32_t recv_remote = cluster_map(recv, me ^ 1u) + 4u * r;
      for (int g = 0; g < ng; ++g) {
        float v[64];
        const uint32_t taddr =
            tmem_base + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + 64u * g;
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld16(taddr + 16u * c, v + 16 * c);
        tmem_wait_ld();
        const int gi = g >> 1;  // index among the owner's groups
        if ((g & 1) == static_cast<int>(me)) {
#pragma unroll
          for (int j = 0; j < 64; ++j) own[(gi * 64 + j) * 128 + r] = v[j];
        } else {
#pragma unroll
          for (int j = 0; j < 64; ++j)
            st_cluster_f32(recv_remote + 512u * static_cast<uint32_t>(gi * 64 + j), v[j]);
        }
      }
    }
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    if (warp >= 2) {
      const int r = 32 * (warp & 3) + lane;
      for (int g = static_cast<int>(me); g < ng; g += 2) {
        const int gi = g >> 1;
#pragma unroll 8
        for (int j = 0; j < 64; ++j) {
          const int at = (gi * 64 + j) * 128 + r;
          own[at] = me == 0 ? own[at] + recv[at] : recv[at] + own[at];
        }
      }
      named_bar_sync(2, 128);
      for (int g = static_cast<int>(me); g < ng; g += 2) {
        const int gi = g >> 1;
        for (int c = r; c < 64 * 16; c += 128) {
          const int j = c >> 4, row8 = (c & 15) * 8;
          const int col = 64 * g + j, n0 = pair_t * 128 + row8;
          if (col >= pair_ncols || n0 >= p.N) continue;
          const float *src = own + (gi * 64 + j) * 128 + row8;
          if (p.vec_y) {
            store_y8(p, col, n0, *reinterpret_cast<const float4 *>(src),
                     *reinterpret_cast<const float4 *>(src + 4));
          } else {
            for (int e = 0; e < 8 && n0 + e < p.N; ++e) {
              float y = src[e];
              const size_t off = static_cast<size_t>(col) * p.N + n0 + e;
              if (p.R != nullptr) y += bf16_to_f32(p.R[off]);
              p.Y[off] = f32_to_bf16_rn(y);
            }
          }
        }
      }
    }
  }
  if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
  if (NG == 1 && p.pair) {
    // Both CTAs of the pair reach this point on every path (also after a time-out), so
    // the cluster barrier always completes. Then each adds its half of the columns in
    // worker order (first k-half + second k-half), adds R, rounds once and stores.
    cluster_sync_all();
    if (warp >= 2) {
      const int r = 32 * (warp & 3) + lane;
      const int me = static_cast<int>(cluster_ctarank());
#pragma unroll
      for (int jj = 0; jj < PH; ++jj) {
        const float o = scratch[jj * 128 + r];
        scratch[jj * 128 + r] = me == 0 ? keep[jj] + o : o + keep[jj];
      }
      named_bar_sync(2, 128);
      if (p.vec_y) {
        for (int c = r; c < PH * 16; c += 128) {
          const int jj = c >> 4, row8 = (c & 15) * 8;
          const int j = me * PH + jj, n0 = pair_t * 128 + row8;
          if (j >= pair_ncols || n0 >= p.N) continue;
          const float4 a = *reinterpret_cast<const float4 *>(scratch + jj * 128 + row8);
          const float4 b = *reinterpret_cast<const float4 *>(scratch + jj * 128 + row8 + 4);
          store_y8(p, j, n0, a, b);
        }
      } else {
        const int n = pair_t * 128 + r;
        for (int jj = 0; jj < PH; ++jj) {
          const int j = me * PH + jj;
          if (j >= pair_ncols || n >= p.N) continue;
          float y = scratch[jj * 128 + r];
          const size_t off = static_cast<size_t>(j) * p.N + n;
          if (p.R != nullptr) y += bf16_to_f32(p.R[off]);
          p.Y[off] = f32_to_bf16_rn(y);
        }
      }
    }
  }
}

template <int MAXC, int NG = 1>
cudaError_t launch_t(const CUtensorMap &wmap, const CUtensorMap &xmap, const EngineParams &p,
                     cudaStream_t s) {
  using C = TCConfig<MAXC, NG>;
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(engine_tc_kernel<MAXC, NG>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  if (p.pair)
    return launch_pdl_cluster(engine_tc_kernel<MAXC, NG>, dim3(p.G), dim3(TC_THREADS), C::SMEM,
                              s, 2, wmap, xmap, p);
  return launch_pdl(engine_tc_kernel<MAXC, NG>, dim3(p.G), dim3(TC_THREADS), C::SMEM, s, wmap,
                    xmap, p);
}

// ---------------------------------------------------------------------------
// Weight and activation loads of one whole tile (local index t of its phase) into the
// stage ring; claims the next tile STAGES k-blocks before the end. False after a time-out.
template <int STAGES, int STAGE_BYTES>
__device__ __forceinline__ bool moe_tile_loads(const EngineParams &p, const CUtensorMap *wmap,
                                               const CUtensorMap *xmap, int t, int shared_g,
                                               uint8_t *stage_mem, uint64_t *full,
                                               uint64_t *empty, volatile int *flags, uint32_t &q,
                                               int &ahead, int *ctr, uint64_t pol) {
  SegInfo s;
  const int64_t it = static_cast<int64_t>(t) * p.KB;
  seg_info(p, it, it + p.KB, s, shared_g);
  const int nxb = (16 * seg_xboxes(s) + p.xbox_rows - 1) / p.xbox_rows;
  const uint32_t bytes = stage_tx_bytes(p, s);
  const int claim_kb = p.KB > STAGES ? p.KB - STAGES : 0;
  for (int kb = 0; kb < p.KB; ++kb, ++q) {
    if (kb == claim_kb) ahead = atomicAdd(ctr, 1);
    const int st = static_cast<int>(q % STAGES);
    uint8_t *dst = stage_mem + st * STAGE_BYTES;
    const uint32_t par = ((q / STAGES) & 1u) ^ 1u;
    if (!mbar_wait_bounded(&empty[st], par, p.status, flags, p.wait_limit_ns)) return false;
    mbar_arrive_expect_tx(&full[st], bytes);
    load_weights(p, s, wmap, dst, &full[st], kb, pol);
    for (int i = 0; i < nxb; ++i)
      tma_load_2d(dst + 16384 + i * p.xbox_rows * 128, xmap, &full[st], kb * TILE_K,
                  s.xrow0 + p.xbox_rows * i);
  }
  return true;
}

// Routed experts in one launch. Tiles are numbered gate/up first (used expert g, tile
// t: g*T1 + t), then down (n1 + g*T2 + t), and every CTA claims them one at a time from
// one counter, each a whole tile over all of its k-blocks (no partial tiles, no
// reduction). A down tile reads its expert's A, which the expert's T1 gate/up tiles
// write: each gate/up tile, once its rows of A are stored, adds one to the expert's
// ready count (release), and the producer loads a down tile's A only after an acquire
// read sees all T1 (then a proxy fence, since TMA reads what ordinary stores wrote); once
// it sees every gate/up tile of the launch done (a second count), one fence covers all of
// its later down tiles. No down tile is claimed before the last gate/up tile, and every
// claimed tile is held by a running CTA, so a wait only ever depends on CTAs that are
// running. While it waits, the producer has the down tile's first weight blocks pulled
// into L2.
template <int STAGES, int STAGE_BYTES>
__device__ __forceinline__ void moe_produce(const EngineParams &p1, const EngineParams &p2,
                                            const CUtensorMap *wmap1, const CUtensorMap *xmap1,
                                            const CUtensorMap *wmap2, const CUtensorMap *xmap2,
                                            const CUtensorMap *wmap1s, const CUtensorMap *wmap2s,
                                            uint8_t *stage_mem, uint64_t *full, uint64_t *empty,
                                            volatile int *tslot, uint64_t *tready,
                                            uint64_t *tfree, volatile int *flags, int n1,
                                            int ntot, int shared_g) {
  prefetch_tensormap(wmap1);
  prefetch_tensormap(xmap1);
  prefetch_tensormap(wmap2);
  prefetch_tensormap(xmap2);
  if (shared_g >= 0) {
    prefetch_tensormap(wmap1s);
    prefetch_tensormap(wmap2s);
  }
  const uint64_t pol = policy_evict_first();
  // Before the dependency wait: the first claims go to about the first G gate/up tiles,
  // so pull the first weight blocks of tile blockIdx.x into L2 (writes nothing; packed
  // banks: one bulk prefetch per 16 KB block).
  if (p1.rm_ready && p1.packed && p1.w_base != nullptr &&
      static_cast<int>(blockIdx.x) / p1.T != shared_g && static_cast<int>(blockIdx.x) < n1) {
    SegInfo s;
    const int64_t it = static_cast<int64_t>(blockIdx.x) * p1.KB;
    seg_info(p1, it, it + p1.KB, s);
    for (int kb = 0; kb < STAGES && kb < p1.KB; ++kb)
      prefetch_l2_bulk(p1.w_base + static_cast<long long>(s.pblk + kb) * 16384, 16384u);
  }
  griddep_wait();
  const int *gu_done = p1.dyn_ctr + 1;  // gate/up tiles whose rows of A are stored
  uint32_t q = 0;
  bool ok = true;
  bool all_ready = false;  // every expert's A seen complete (and fenced) by this thread
  int ahead = -1;  // the next tile, claimed STAGES k-blocks before the current one ends
  for (uint32_t seg = 0;; ++seg) {
    int t = ahead;
    if (t < 0) t = ok ? atomicAdd(p1.dyn_ctr, 1) : ntot;
    ahead = -1;
    int tile = (ok && t < ntot) ? t : -1;
    const int sl = static_cast<int>(seg & 3u);
    if (tile >= n1 && !all_ready) {  // a down tile: its expert's A must be complete
      const int g = (tile - n1) / p2.T;
      if (ld_acquire_gpu(gu_done) >= n1)
        all_ready = true;  // then one proxy fence covers every later down tile
      else if (ld_acquire_gpu(p1.ready + g) < p1.T) {
        if (p2.packed && p2.w_base != nullptr && g != shared_g) {
          SegInfo s;
          const int64_t it = static_cast<int64_t>(tile - n1) * p2.KB;
          seg_info(p2, it, it + p2.KB, s);
          for (int kb = 0; kb < STAGES && kb < p2.KB; ++kb)
            prefetch_l2_bulk(p2.w_base + static_cast<long long>(s.pblk + kb) * 16384, 16384u);
        }
        if (!wait_count_bounded(p1.ready + g, p1.T, p1.status, flags, p1.wait_limit_ns)) {
          ok = false;
          tile = -1;
        }
      }
      fence_proxy_async_global();
    }
    if (ok && !mbar_wait_bounded(&tfree[sl], ((seg >> 2) & 1u) ^ 1u, p1.status, flags,
                                 p1.wait_limit_ns)) {
      ok = false;
      tile = -1;
    }
    tslot[sl] = tile;
    mbar_arrive(&tready[sl]);
    if (tile < 0) break;
    // the phases' parameters and tensor maps stay compile-time operands in each branch
    if (tile >= n1)
      ok = moe_tile_loads<STAGES, STAGE_BYTES>(p2, (tile - n1) / p2.T == shared_g ? wmap2s : wmap2,
                                               xmap2, tile - n1, shared_g, stage_mem, full, empty,
                                               flags, q, ahead, p1.dyn_ctr, pol);
    else
      ok = moe_tile_loads<STAGES, STAGE_BYTES>(p1, tile / p1.T == shared_g ? wmap1s : wmap1, xmap1,
                                               tile, shared_g, stage_mem, full, empty, flags, q,
                                               ahead, p1.dyn_ctr, pol);
  }
  griddep_launch_dependents();
  if (flags[0]) {
    // after a time-out: let this CTA's copies still in flight land before it exits
    const uint32_t q0 = q > STAGES ? q - STAGES : 0u;
    for (uint32_t qq = q0; qq < q; ++qq)
      (void)mbar_wait_drain(&full[qq % STAGES], (qq / STAGES) & 1u, 10000000ull);
  }
}

template <int MAXC>
__global__ void __launch_bounds__(TC_THREADS, 1)
    engine_tc_moe_kernel(const __grid_constant__ CUtensorMap wmap1,
                         const __grid_constant__ CUtensorMap xmap1,
                         const __grid_constant__ CUtensorMap wmap2,
                         const __grid_constant__ CUtensorMap xmap2,
                         const __grid_constant__ CUtensorMap wmap1s,
                         const __grid_constant__ CUtensorMap wmap2s, const EngineParams p1,
                         const EngineParams p2) {
  using C = TCConfig<MAXC, 1>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *stage_mem = smem;
  float *scratch = reinterpret_cast<float *>(smem + C::STAGES * C::STAGE_BYTES);
  uint8_t *tail = smem + C::STAGES * C::STAGE_BYTES + C::SCRATCH_BYTES;
  uint64_t *full = reinterpret_cast<uint64_t *>(tail);
  uint64_t *empty = full + C::STAGES;
  uint64_t *acc_full = empty + C::STAGES;   // [2]
  uint64_t *acc_empty = acc_full + 2;       // [2]
  uint64_t *drain = acc_empty + 2;          // [1]
  uint64_t *tready = drain + 1;             // [4]
  uint64_t *tfree = tready + 4;             // [4]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tfree + 4);
  volatile int *flags = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *tslot = flags + 3;          // [4]
  volatile int *etile = tslot + 4;          // [2]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the route map picks the experts: read it now only if it was complete before the
  // previous kernel of the stream started
  if (!p1.rm_ready) griddep_wait();
  const int U = rm_num_used(p1);
  // groups: the used experts, then (with_shared) the shared expert
  const int shared_g = p1.with_shared ? U : -1;
  const int ng = U + (p1.with_shared ? 1 : 0);
  const int n1 = ng * p1.T;
  const int ntot = n1 + ng * p2.T;

  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&tready[i], 1);
      mbar_init(&tfree[i], 2);  // the MMA issuer and epilogue thread 0
    }
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0)
      moe_produce<C::STAGES, C::STAGE_BYTES>(p1, p2, &wmap1, &xmap1, &wmap2, &xmap2, &wmap1s,
                                             &wmap2s, stage_mem, full, empty, tslot, tready,
                                             tfree, flags, n1, ntot, shared_g);
    else
      griddep_wait();
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    griddep_wait();
    if (lane == 0) {
      uint32_t q = 0;
      bool ok = true;
      for (uint32_t seg = 0; ok; ++seg) {
        const int sl = static_cast<int>(seg & 3u);
        if (!mbar_wait_bounded(&tready[sl], (seg >> 2) & 1u, p1.status, flags, p1.wait_limit_ns))
          break;
        const int tile = tslot[sl];
        mbar_arrive(&tfree[sl]);
        if (tile < 0) break;
        SegInfo s;
        if (tile >= n1) {
          const int64_t it = static_cast<int64_t>(tile - n1) * p2.KB;
          seg_info(p2, it, it + p2.KB, s, shared_g);
        } else {
          const int64_t it = static_cast<int64_t>(tile) * p1.KB;
          seg_info(p1, it, it + p1.KB, s, shared_g);
        }
        ok = mma_segment<C::STAGES, C::STAGE_BYTES, 1>(s, seg, q, tmem_base, stage_mem, full,
                                                      empty, acc_full, acc_empty, p1, flags);
      }
      if (flags[0]) {  // let every MMA issued so far finish before the memory is freed
        tc_commit(drain);
        (void)mbar_wait_drain(drain, 0u, 10000000ull);
      }
    }
  } else {
    // --------------------------------------------------------------- epilogue
    griddep_wait();
    const int r = 32 * (warp & 3) + lane;  // tile row == tensor-memory lane
    for (uint32_t seg = 0;; ++seg) {
      const int sl = static_cast<int>(seg & 3u);
      const uint32_t buf = seg & 1u;
      // thread 0 takes the segment's tile from the producer's slot and waits for its
      // accumulator; the other 127 threads learn both through etile across the barrier,
      // so every thread takes the same branches around the named barriers below
      if (r == 0) {
        const bool got =
            mbar_wait_bounded(&tready[sl], (seg >> 2) & 1u, p1.status, flags, p1.wait_limit_ns);
        int t = (got && !flags[0]) ? tslot[sl] : -1;
        mbar_arrive(&tfree[sl]);
        if (t >= 0 && (!mbar_wait_bounded(&acc_full[buf], (seg >> 1) & 1u, p1.status, flags,
                                          p1.wait_limit_ns) ||
                       flags[0]))
          t = -1;
        etile[seg & 1u] = t;
      }
      named_bar_sync(2, 128);
      const int tile = etile[seg & 1u];
      if (tile < 0) break;
      const bool down = tile >= n1;
      SegInfo s;
      if (down) {
        const int64_t it = static_cast<int64_t>(tile - n1) * p2.KB;
        seg_info(p2, it, it + p2.KB, s, shared_g);
      } else {
        const int64_t it = static_cast<int64_t>(tile) * p1.KB;
        seg_info(p1, it, it + p1.KB, s, shared_g);
      }
      tc_fence_after();
      float v[C::NC];
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + buf * 64u;
#pragma unroll
      for (int c = 0; c < C::NC / 16; ++c) tmem_ld16(taddr + 16u * c, v + 16 * c);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
      float acc[MAXC];
#pragma unroll
      for (int j = 0; j < MAXC; ++j) acc[j] = v[j];
      if (down) {
        epilogue_rows<MAXC>(p2, s, r, acc, scratch, 2, flags);
      } else {
        epilogue_rows<MAXC>(p1, s, r, acc, scratch, 2, flags);
        // this tile's rows of A are stored: count them for the expert's down tiles
        fence_proxy_async_global();
        named_bar_sync(2, 128);
        if (r == 0) {
          red_add_release_gpu(p1.ready + s.gt / p1.T, 1);
          red_add_release_gpu(p1.dyn_ctr + 1, 1);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

template <int MAXC>
cudaError_t launch_moe_t(const CUtensorMap &wmap1, const CUtensorMap &xmap1,
                         const CUtensorMap &wmap2, const CUtensorMap &xmap2,
                         const CUtensorMap &wmap1s, const CUtensorMap &wmap2s,
                         const EngineParams &p1, const EngineParams &p2, cudaStream_t s) {
  using C = TCConfig<MAXC, 1>;
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(engine_tc_moe_kernel<MAXC>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  return launch_pdl(engine_tc_moe_kernel<MAXC>, dim3(p1.G), dim3(TC_THREADS), C::SMEM, s, wmap1,
                    xmap1, wmap2, xmap2, wmap1s, wmap2s, p1, p2);
}

}  // namespace

cudaError_t launch_engine_tc(int maxc, const CUtensorMap &wmap, const CUtensorMap &xmap,
                             const EngineParams &p, cudaStream_t s) {
  if (p.dyn && (p.dyn < 0 || p.dyn > 256 || !p.grouped || p.ngrp != 1 || p.defer || p.pair ||
                p.dyn_ctr == nullptr))
    return cudaErrorInvalidValue;
  if (p.pair && ((p.ngrp > 1 && maxc != 64) || p.grouped || p.defer || p.mode != MODE_LINEAR ||
                 p.G != 2 * p.T || p.KB % 2 != 0))
    return cudaErrorInvalidValue;
  if (p.ngrp > 1) {  // wide projection: 64-column groups, 2 or up to 4 of them
    if (maxc != 64 || p.ngrp > 4 || p.mode != MODE_LINEAR || p.grouped)
      return cudaErrorInvalidValue;
    return p.ngrp == 2 ? launch_t<64, 2>(wmap, xmap, p, s) : launch_t<64, 4>(wmap, xmap, p, s);
  }
  switch (maxc) {
    case 2: return launch_t<2>(wmap, xmap, p, s);
    case 4: return launch_t<4>(wmap, xmap, p, s);
    case 8: return launch_t<8>(wmap, xmap, p, s);
    case 16: return launch_t<16>(wmap, xmap, p, s);
    case 32: return launch_t<32>(wmap, xmap, p, s);
    case 64: return launch_t<64>(wmap, xmap, p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ssd

namespace ssd {

cudaError_t launch_engine_tc_moe(int maxc, const CUtensorMap &wmap1, const CUtensorMap &xmap1,
                                 const CUtensorMap &wmap2, const CUtensorMap &xmap2,
                                 const CUtensorMap &wmap1s, const CUtensorMap &wmap2s,
                                 const EngineParams &p1, const EngineParams &p2,
                                 cudaStream_t s) {
  if (!p1.grouped || !p2.grouped || p1.mode != MODE_GATEUP || p2.mode != MODE_DOWN ||
      p1.dyn_ctr == nullptr || p1.ready == nullptr || p1.ngrp != 1 || p2.ngrp != 1 ||
      p1.defer || p2.defer || p1.pair || p2.pair || p1.slot_cols != p2.slot_cols ||
      p1.route_map != p2.route_map || p1.G < 1 || p1.with_shared != p2.with_shared)
    return cudaErrorInvalidValue;
  switch (maxc) {
    case 2: return launch_moe_t<2>(wmap1, xmap1, wmap2, xmap2, wmap1s, wmap2s, p1, p2, s);
    case 4: return launch_moe_t<4>(wmap1, xmap1, wmap2, xmap2, wmap1s, wmap2s, p1, p2, s);
    case 8: return launch_moe_t<8>(wmap1, xmap1, wmap2, xmap2, wmap1s, wmap2s, p1, p2, s);
    case 16: return launch_moe_t<16>(wmap1, xmap1, wmap2, xmap2, wmap1s, wmap2s, p1, p2, s);
    case 32: return launch_moe_t<32>(wmap1, xmap1, wmap2, xmap2, wmap1s, wmap2s, p1, p2, s);
    case 64: return launch_moe_t<64>(wmap1, xmap1, wmap2, xmap2, wmap1s, wmap2s, p1, p2, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ssd
