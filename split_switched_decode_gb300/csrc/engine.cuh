// engine.cuh -- schedule, deterministic split-K reduction and epilogues shared by the
// CUDA-core (engine_cc.cu) and tensor-core (engine_tc.cu) split-K kernels.
//
// "Hyper Optimizing Kimi K3 in vLLM", Part 1 / 1 "Tune shapes for the workload": at
// larger batches the projections use split-K kernels that divide the matrix
// multiplication across more GPU workers.
//
// Work decomposition. A launch covers `groups` independent products that share N and
// K (one for a projection, one per used expert for the grouped expert GEMV). Each
// product is cut into T output tiles of 128 weight rows and KB k-blocks of 64. The
// flattened sequence of (group, tile, k-block) iterations is divided into G contiguous
// ranges of equal length (+-1), one per CTA ("worker"): every SM streams the same
// number of weight bytes, whatever N, K and the number of groups are. A worker walks
// its range in "segments", one per tile it touches. A segment covering a whole tile
// ends in the epilogue directly; otherwise the worker stores its partial tile in its
// workspace slot and bumps the tile's arrival counter, and the worker that arrives
// last adds the partials of all contributors in worker order (fixed order, so the
// result is bit-identical run to run for a fixed G), runs the epilogue and resets the
// counter to zero for the next launch; no CTA waits on another. The one exception is
// the tensor-core "pair" schedule (engine_tc.cu): when every tile is split into two
// k-halves, the two workers of a tile are launched as a 2-CTA cluster, which the
// hardware co-schedules, and add their halves on chip after a cluster barrier.
#pragma once

#include "common.cuh"
#include "internal.h"
#include "routing.cuh"

namespace ssd {

__device__ __forceinline__ int64_t sk_start(int64_t total, int G, int w) {
  return static_cast<int64_t>(w) * total / G;
}

// Worker whose range holds iteration i (requires G <= total: no empty ranges).
__device__ __forceinline__ int sk_worker_of(int64_t total, int G, int64_t i) {
  return static_cast<int>(((i + 1) * static_cast<int64_t>(G) - 1) / total);
}

__device__ __forceinline__ int rm_num_used(const EngineParams &p) {
  return min(max(p.route_map[2 * p.E + 1 + 2 * p.P], 0), p.E);
}

struct SegInfo {
  int gt;      // global tile id (group * T + tile)
  int t;       // tile within its group
  int kb0;     // first k-block of the segment
  int kb1;     // one past the last k-block
  int ncols;   // activation rows (batch columns) of the group
  int xrow0;   // first activation row of the group (of the column group: wide projections)
  int cgrp;    // column group of 64 batch columns (wide projections; else 0)
  int wrow0;   // W row of tile rows 0..63
  int wrow1;   // W row of tile rows 64..127
  bool full;   // the segment covers the whole tile
  int pblk;    // tile-packed W: block of this tile's k-block 0 ((expert * T + t) * KB)
};

// shared_g: the group index of the shared expert inside a grouped launch (after the used
// experts), or -1: its weights come from their own tensor map (expert 0 of it) and its
// activation rows are P .. P+B-1.
__device__ __forceinline__ void seg_info(const EngineParams &p, int64_t it, int64_t end,
                                         SegInfo &s, int shared_g = -1) {
  s.gt = static_cast<int>(it / p.KB);
  s.kb0 = static_cast<int>(it - static_cast<int64_t>(s.gt) * p.KB);
  const int64_t tend = static_cast<int64_t>(s.gt + 1) * p.KB;
  const int64_t se = end < tend ? end : tend;
  s.kb1 = s.kb0 + static_cast<int>(se - it);
  const int g = s.gt / p.T;
  s.t = s.gt - g * p.T;
  int wbase;
  int e = 0;  // expert of a grouped launch
  if (p.grouped && g == shared_g) {
    s.xrow0 = p.P;
    s.ncols = min(p.B, p.slot_cols);
    wbase = 0;
  } else if (p.grouped) {
    // the route map comes from moe_front or the validating rebuild kernel; the clamps
    // only keep a corrupted map from steering loads or stores out of their buffers
    const int32_t *rm = p.route_map;
    e = min(max(rm[2 * p.E + 2 + 2 * p.P + g], 0), p.E - 1);
    s.xrow0 = min(max(rm[p.E + e], 0), p.P);
    s.ncols = min(max(rm[e], 0), min(p.slot_cols, p.P - s.xrow0));
    wbase = e * p.w_group_rows;
  } else {
    s.ncols = p.B;  // every batch column; wide projections split it into column groups
    s.xrow0 = 0;
    wbase = 0;
  }
  if (p.mode == MODE_GATEUP) {
    s.wrow0 = wbase + s.t * 64;                 // gate rows
    s.wrow1 = wbase + p.up_row_off + s.t * 64;  // matching up rows
  } else {
    s.wrow0 = wbase + s.t * 128;
    s.wrow1 = s.wrow0 + 64;
  }
  s.full = (s.kb0 == 0 && s.kb1 == p.KB);
  s.pblk = (e * p.T + s.t) * p.KB;
  s.cgrp = 0;
}

// Activation boxes (16 rows each) a segment needs: at least one.
__device__ __forceinline__ int seg_xboxes(const SegInfo &s) {
  return s.ncols > 16 ? (s.ncols + 15) >> 4 : 1;
}

// Bytes one stage receives: the 128-row weight tile plus the activation boxes.
__device__ __forceinline__ uint32_t stage_tx_bytes(const EngineParams &p, const SegInfo &s) {
  const int nxb = (16 * seg_xboxes(s) + p.xbox_rows - 1) / p.xbox_rows;
  return 16384u + static_cast<uint32_t>(nxb * p.xbox_rows) * 128u;
}

// Weight boxes of one k-block: one 128-row box, or the 64 gate rows and the 64 matching
// up rows (two boxes) in gate/up mode. A tile-packed W is mapped as rows of 128 bytes
// (64 k): the box of (expert, tile t, k-block kb) is the contiguous 16 KB block
// (expert*T + t)*KB + kb, whose rows land where the two gate/up boxes would.
__device__ __forceinline__ void load_weights(const EngineParams &p, const SegInfo &s,
                                             const CUtensorMap *wmap, uint8_t *dst,
                                             uint64_t *bar, int kb, uint64_t pol) {
  if (p.packed) {
    tma_load_2d_hint(dst, wmap, bar, 0, (s.pblk + kb) * TILE_N, pol);
    return;
  }
  tma_load_2d_hint(dst, wmap, bar, kb * TILE_K, s.wrow0, pol);
  if (p.wbox_rows == 64)
    tma_load_2d_hint(dst + 8192, wmap, bar, kb * TILE_K, s.wrow1, pol);
}

// Before the dependency wait, while the previous kernel of the stream is still
// finishing and HBM is underused, the producer warp asks L2 for the next l2pf_kb
// k-blocks of this CTA's weights beyond the ones already requested into shared memory
// (one bulk prefetch per weight row and segment; weights only, so this may precede the
// wait). The later TMA loads of those blocks then hit L2.
__device__ __forceinline__ void prefetch_weights_l2(const EngineParams &p, int64_t begin,
                                                    int64_t end, uint32_t skip, int lane) {
  if (p.l2pf_kb <= 0 || p.w_base == nullptr) return;
  const long long row_bytes = static_cast<long long>(p.K) * 2;
  int64_t it = begin + skip;
  int64_t stop = it + p.l2pf_kb;
  if (stop > end) stop = end;
  if (p.packed) {  // tile-packed W: each k-block of a segment is one contiguous 16 KB block
    for (int64_t i = it + lane; i < stop; i += 32) {
      SegInfo s;
      seg_info(p, i, i + 1, s);
      prefetch_l2_bulk(p.w_base + static_cast<long long>(s.pblk + s.kb0) * 16384, 16384u);
    }
    return;
  }
  while (it < stop) {
    SegInfo s;
    seg_info(p, it, stop, s);
    const long long k0 = static_cast<long long>(s.kb0) * TILE_K * 2;
    long long k1 = static_cast<long long>(s.kb1) * TILE_K * 2;
    if (k1 > row_bytes) k1 = row_bytes;
    if (k1 > k0) {
      for (int r = lane; r < TILE_N; r += 32) {
        const long long row = (r < 64) ? s.wrow0 + r
                                        : (p.wbox_rows == 64 ? s.wrow1 + (r - 64) : s.wrow0 + r);
        if (row < p.w_rows)
          prefetch_l2_bulk(p.w_base + row * row_bytes + k0, static_cast<uint32_t>(k1 - k0));
      }
    }
    it += s.kb1 - s.kb0;
  }
}

// TMA producer of both engines, run by one thread. The weight boxes of the first
// STAGES k-blocks do not depend on the previous kernel of the stream, so they are
// issued before griddep_wait (programmatic dependent launch) -- for a grouped launch
// only when its route map was complete before the previous kernel started (rm_ready),
// since the map picks the weights; the activation boxes only after it.
template <int STAGES, int STAGE_BYTES>
__device__ __forceinline__ void engine_produce(const EngineParams &p, const CUtensorMap *wmap,
                                               const CUtensorMap *xmap, uint8_t *stage_mem,
                                               uint64_t *full, uint64_t *empty,
                                               volatile int *flags, int64_t begin, int64_t end) {
  prefetch_tensormap(wmap);
  prefetch_tensormap(xmap);
  const uint64_t pol = policy_evict_first();  // weights are read once per launch
  uint32_t pre = 0;
  if (!p.grouped || p.rm_ready) {
    for (int64_t it = begin; it < end && pre < STAGES;) {
      SegInfo s;
      seg_info(p, it, end, s);
      const uint32_t bytes = stage_tx_bytes(p, s);
      for (int kb = s.kb0; kb < s.kb1 && pre < STAGES; ++kb, ++pre) {
        uint8_t *dst = stage_mem + pre * STAGE_BYTES;
        mbar_arrive_expect_tx(&full[pre], bytes);  // first use of the stage: it is empty
        load_weights(p, s, wmap, dst, &full[pre], kb, pol);
      }
      it += s.kb1 - s.kb0;
    }
  }
  griddep_wait();
  uint32_t q = 0;
  bool ok = true;
  for (int64_t it = begin; it < end && ok;) {
    SegInfo s;
    seg_info(p, it, end, s);
    const int nxb = (16 * seg_xboxes(s) + p.xbox_rows - 1) / p.xbox_rows;
    const uint32_t bytes = stage_tx_bytes(p, s);
    for (int kb = s.kb0; kb < s.kb1; ++kb, ++q) {
      const int st = static_cast<int>(q % STAGES);
      uint8_t *dst = stage_mem + st * STAGE_BYTES;
      if (q >= pre) {
        const uint32_t par = ((q / STAGES) & 1u) ^ 1u;
        if (!mbar_wait_bounded(&empty[st], par, p.status, flags, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[st], bytes);
        load_weights(p, s, wmap, dst, &full[st], kb, pol);
      }
      for (int i = 0; i < nxb; ++i)
        tma_load_2d(dst + 16384 + i * p.xbox_rows * 128, xmap, &full[st], kb * TILE_K,
                    s.xrow0 + p.xbox_rows * i);
    }
    it += s.kb1 - s.kb0;
  }
  // every weight and activation load of this CTA is issued: the next kernel of the
  // stream may be scheduled onto SMs as they free up
  griddep_launch_dependents();
  if (flags[0]) {
    // after a time-out: let this CTA's copies still in flight land before it exits
    const uint32_t q0 = q > STAGES ? q - STAGES : 0u;
    for (uint32_t qq = q0; qq < q; ++qq)
      (void)mbar_wait_drain(&full[qq % STAGES], (qq / STAGES) & 1u, 10000000ull);
  }
}

// Whole-tile schedule (p.dyn; grouped tensor-core launches). The launch's tiles are
// numbered in (group, tile) order. CTA w streams its static tiles [w*S, (w+1)*S) and then
// claims tiles G*S, G*S+1, ... one at a time from *p.dyn_ctr until none is left, so the
// CTAs on SMs that stream faster take more of the remainder (the SMs of a GB300 do not
// all read HBM at the same rate). Every tile is one segment over all of its k-blocks:
// no partial tiles, no reduction, and each output is accumulated in the same k order
// whichever CTA computes it.
__device__ __forceinline__ int dyn_static_tiles(const EngineParams &p, int ntiles) {
  return static_cast<int>((static_cast<int64_t>(ntiles) * p.dyn) / (256ll * p.G));
}

// Producer of the whole-tile schedule (one thread). Segment seg's tile, or -1 after the
// last one, goes to slot seg % 4 of `tslot` for the MMA and epilogue warps: tready[slot]
// completes a phase when the slot is written, tfree[slot] when both readers have taken
// it. As in engine_produce, the weight boxes of the first STAGES k-blocks (of static
// tiles) may be issued before griddep_wait; claims are made only after it (the counter
// is cleared by the launch before this one). The next claim is issued STAGES k-blocks
// before the current tile's last one, so its round trip overlaps the loads.
template <int STAGES, int STAGE_BYTES>
__device__ __forceinline__ void engine_produce_dyn(const EngineParams &p, const CUtensorMap *wmap,
                                                   const CUtensorMap *xmap, uint8_t *stage_mem,
                                                   uint64_t *full, uint64_t *empty,
                                                   volatile int *tslot, uint64_t *tready,
                                                   uint64_t *tfree, volatile int *flags,
                                                   int ntiles) {
  prefetch_tensormap(wmap);
  prefetch_tensormap(xmap);
  const uint64_t pol = policy_evict_first();
  const int S = dyn_static_tiles(p, ntiles);
  const int t0 = static_cast<int>(blockIdx.x) * S;
  uint32_t pre = 0;
  if (p.rm_ready) {
    for (int i = 0; i < S && pre < STAGES; ++i) {
      SegInfo s;
      const int64_t it = static_cast<int64_t>(t0 + i) * p.KB;
      seg_info(p, it, it + p.KB, s);
      const uint32_t bytes = stage_tx_bytes(p, s);
      for (int kb = 0; kb < p.KB && pre < STAGES; ++kb, ++pre) {
        mbar_arrive_expect_tx(&full[pre], bytes);  // first use of the stage: it is empty
        load_weights(p, s, wmap, stage_mem + pre * STAGE_BYTES, &full[pre], kb, pol);
      }
    }
  }
  griddep_wait();
  const int base = p.G * S;
  const int claim_kb = p.KB > STAGES ? p.KB - STAGES : 0;
  uint32_t q = 0;
  bool ok = true;
  int ahead = -1;  // the next dynamic tile, once claimed
  for (uint32_t seg = 0;; ++seg) {
    int tile;
    if (static_cast<int>(seg) < S) {
      tile = t0 + static_cast<int>(seg);
    } else {
      if (ahead < 0 && ok) ahead = base + atomicAdd(p.dyn_ctr, 1);
      tile = (ok && ahead < ntiles) ? ahead : -1;
      ahead = -1;
    }
    const int sl = static_cast<int>(seg & 3u);
    if (ok && !mbar_wait_bounded(&tfree[sl], ((seg >> 2) & 1u) ^ 1u, p.status, flags,
                                 p.wait_limit_ns)) {
      ok = false;
      tile = -1;
    }
    tslot[sl] = tile;
    mbar_arrive(&tready[sl]);
    if (tile < 0) break;
    SegInfo s;
    const int64_t it = static_cast<int64_t>(tile) * p.KB;
    seg_info(p, it, it + p.KB, s);
    const int nxb = (16 * seg_xboxes(s) + p.xbox_rows - 1) / p.xbox_rows;
    const uint32_t bytes = stage_tx_bytes(p, s);
    const bool next_dyn = static_cast<int>(seg) + 1 >= S;
    for (int kb = 0; kb < p.KB; ++kb, ++q) {
      if (kb == claim_kb && next_dyn) ahead = base + atomicAdd(p.dyn_ctr, 1);
      const int st = static_cast<int>(q % STAGES);
      uint8_t *dst = stage_mem + st * STAGE_BYTES;
      if (q >= pre) {
        const uint32_t par = ((q / STAGES) & 1u) ^ 1u;
        if (!mbar_wait_bounded(&empty[st], par, p.status, flags, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[st], bytes);
        load_weights(p, s, wmap, dst, &full[st], kb, pol);
      }
      for (int i = 0; i < nxb; ++i)
        tma_load_2d(dst + 16384 + i * p.xbox_rows * 128, xmap, &full[st], kb * TILE_K,
                    s.xrow0 + p.xbox_rows * i);
    }
  }
  griddep_launch_dependents();
  if (flags[0]) {
    // after a time-out: let this CTA's copies still in flight land before it exits
    const uint32_t q0 = q > STAGES ? q - STAGES : 0u;
    for (uint32_t qq = q0; qq < q; ++qq)
      (void)mbar_wait_drain(&full[qq % STAGES], (qq / STAGES) & 1u, 10000000ull);
  }
}

// 8 consecutive rows a, b (plus the residual run rr when has_r), rounded once to bf16,
// packed.
__device__ __forceinline__ uint4 pack_y8r(const float4 &a, const float4 &b, const uint4 &rr,
                                          bool has_r) {
  float y[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  if (has_r) {
    y[0] += bf16lo(rr.x);
    y[1] += bf16hi(rr.x);
    y[2] += bf16lo(rr.y);
    y[3] += bf16hi(rr.y);
    y[4] += bf16lo(rr.z);
    y[5] += bf16hi(rr.z);
    y[6] += bf16lo(rr.w);
    y[7] += bf16hi(rr.w);
  }
  uint4 o;
  o.x = f32_to_bf16_rn(y[0]) | (static_cast<uint32_t>(f32_to_bf16_rn(y[1])) << 16);
  o.y = f32_to_bf16_rn(y[2]) | (static_cast<uint32_t>(f32_to_bf16_rn(y[3])) << 16);
  o.z = f32_to_bf16_rn(y[4]) | (static_cast<uint32_t>(f32_to_bf16_rn(y[5])) << 16);
  o.w = f32_to_bf16_rn(y[6]) | (static_cast<uint32_t>(f32_to_bf16_rn(y[7])) << 16);
  return o;
}

// Y rows n0 .. n0+7 of batch column j: y (+ R) rounded once to bf16, one 16-byte store
// (or element by element for a ragged tail). Requires N % 8 == 0 and 16-byte aligned Y
// and R (p.vec_y).
__device__ __forceinline__ void store_y8(const EngineParams &p, int j, int n0, const float4 &a,
                                         const float4 &b) {
  float y[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  const size_t off = static_cast<size_t>(j) * p.N + n0;
  if (n0 + 8 <= p.N) {
    if (p.R != nullptr) {
      const uint4 rr = *reinterpret_cast<const uint4 *>(p.R + off);
      y[0] += bf16lo(rr.x);
      y[1] += bf16hi(rr.x);
      y[2] += bf16lo(rr.y);
      y[3] += bf16hi(rr.y);
      y[4] += bf16lo(rr.z);
      y[5] += bf16hi(rr.z);
      y[6] += bf16lo(rr.w);
      y[7] += bf16hi(rr.w);
    }
    uint4 o;
    o.x = f32_to_bf16_rn(y[0]) | (static_cast<uint32_t>(f32_to_bf16_rn(y[1])) << 16);
    o.y = f32_to_bf16_rn(y[2]) | (static_cast<uint32_t>(f32_to_bf16_rn(y[3])) << 16);
    o.z = f32_to_bf16_rn(y[4]) | (static_cast<uint32_t>(f32_to_bf16_rn(y[5])) << 16);
    o.w = f32_to_bf16_rn(y[6]) | (static_cast<uint32_t>(f32_to_bf16_rn(y[7])) << 16);
    *reinterpret_cast<uint4 *>(p.Y + off) = o;
  } else {
    for (int e = 0; e < 8 && n0 + e < p.N; ++e) {
      float ye = y[e];
      if (p.R != nullptr) ye += bf16_to_f32(p.R[off + e]);
      p.Y[off + e] = f32_to_bf16_rn(ye);
    }
  }
}

// Split-K reduction of one tile, run by the 128 threads that hold the segment's values
// (thread r holds row r, columns 0..ncols-1 in v). Returns true when v holds the final
// tile values on return (whole-tile segment, or this worker arrived last).
template <int MAXC>
__device__ __forceinline__ bool reduce_tile(const EngineParams &p, const SegInfo &s, int64_t total, int w,
                            int64_t begin, int r, float (&v)[MAXC], int bar_id,
                            volatile int *flags) {
  if (s.full && !p.defer) return true;
  const int64_t tb = static_cast<int64_t>(s.gt) * p.KB;
  const int which_me = (begin >= tb) ? 0 : 1;
  const size_t slot_floats = static_cast<size_t>(128) * p.slot_cols;
  // slot of (worker, which, column group); column groups only exist when p.ngrp > 1
  float *slot =
      p.partials + (static_cast<size_t>(w * 2 + which_me) * p.ngrp + s.cgrp) * slot_floats;
#pragma unroll
  for (int j = 0; j < MAXC; ++j)
    if (j < s.ncols) slot[j * 128 + r] = v[j];
  if (p.defer) return false;  // a dependent kernel adds the partials (front end)
  named_bar_sync(bar_id, 128);
  const int first = sk_worker_of(total, p.G, tb);
  const int last = sk_worker_of(total, p.G, tb + p.KB - 1);
  if (r == 0) {
    const int old = atom_add_acq_rel_gpu(&p.counters[s.gt * p.ngrp + s.cgrp], 1);
    flags[1] = (old == last - first) ? 1 : 0;
  }
  named_bar_sync(bar_id, 128);
  if (!flags[1]) return false;
  // Add the contributors' partials in worker order. Only the first contributor can
  // have started before this tile (its slot 1); every later one began inside it (slot
  // 0). Loads of RD contributors are issued before their adds so they overlap.
  constexpr int RD = MAXC >= 16 ? 1 : 16 / MAXC;
  const int which_first = (sk_start(total, p.G, first) >= tb) ? 0 : 1;
  float t[MAXC];
#pragma unroll
  for (int j = 0; j < MAXC; ++j) t[j] = 0.f;
  for (int wk0 = first; wk0 <= last; wk0 += RD) {
    float tmp[RD][MAXC];
#pragma unroll
    for (int d = 0; d < RD; ++d) {
      const int wk = wk0 + d;
      const int which = (wk == first) ? which_first : 0;
      const float *sl =
          p.partials + (static_cast<size_t>(wk * 2 + which) * p.ngrp + s.cgrp) * slot_floats;
      const bool other = (wk <= last) && (wk != w);
#pragma unroll
      for (int j = 0; j < MAXC; ++j)
        tmp[d][j] = (other && j < s.ncols) ? __ldcg(sl + j * 128 + r) : 0.f;
    }
#pragma unroll
    for (int d = 0; d < RD; ++d) {
      const int wk = wk0 + d;
      if (wk <= last) {
#pragma unroll
        for (int j = 0; j < MAXC; ++j) t[j] += (wk == w) ? v[j] : tmp[d][j];
      }
    }
  }
#pragma unroll
  for (int j = 0; j < MAXC; ++j) v[j] = t[j];
  if (r == 0) p.counters[s.gt * p.ngrp + s.cgrp] = 0;
  return true;
}

// Fused combine, after a down tile's rows are stored (128 threads, thread r = row r):
// every column's token counts one more contribution to its (token, block t) counter;
// the arrival that completes it (acquire-release, after a barrier over the 128 writers)
// computes Y[b, block] = bf16( sum_{j ascending} w[b,j] * Yp[pos[b,j]] (+ S[b]) ) in the
// same order and precision as the separate combine kernel, so the bits do not depend on
// which tile finishes a block, and resets the counter for the next call.
template <int MAXC>
__device__ __forceinline__ void combine_tail(const EngineParams &p, const SegInfo &s, int r,
                                             float *scratch, int bar_id) {
  int *last = reinterpret_cast<int *>(scratch);  // [MAXC]: token this tile finishes, or -1
  named_bar_sync(bar_id, 128);  // every row of this tile is stored
  if (r < s.ncols) {
    int b;
    if (p.grouped) {
      const int q = p.route_map[2 * p.E + 1 + min(max(s.xrow0 + r, 0), p.P - 1)];  // pairs
      b = q / p.topk;
    } else {
      b = s.xrow0 + r;
    }
    b = min(max(b, 0), p.B - 1);
    int *cnt = p.cmb_cnt + static_cast<size_t>(b) * p.T + s.t;
    const bool done = atom_add_acq_rel_gpu(cnt, 1) == p.cmb_need - 1;
    if (done) *cnt = 0;  // every contribution is in: nothing else touches it this call
    last[r] = done ? b : -1;
  }
  named_bar_sync(bar_id, 128);
  const int n = s.t * 128 + r;
  const int32_t *pos = p.route_map + 2 * p.E + 1 + p.P;
  for (int j = 0; j < s.ncols; ++j) {
    const int b = last[j];
    if (b < 0 || n >= p.N) continue;
    float y[MAX_TOPK];
#pragma unroll
    for (int k = 0; k < MAX_TOPK; ++k) {
      y[k] = 0.f;
      if (k < p.topk) {
        const int at = min(max(pos[b * p.topk + k], 0), p.P - 1);
        y[k] = __ldcg(p.cmb_yp + static_cast<size_t>(at) * p.N + n);
      }
    }
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < MAX_TOPK; ++k)
      if (k < p.topk) acc = fmaf(p.topk_w[b * p.topk + k], y[k], acc);
    if (p.cmb_s != nullptr) acc += __ldcg(p.cmb_s + static_cast<size_t>(b) * p.N + n);
    p.cmb_y[static_cast<size_t>(b) * p.N + n] = f32_to_bf16_rn(acc);
  }
}

// Epilogue of one finished tile, run by the same 128 threads. `scratch` holds at least
// 64 * MAXC floats and is free on entry.
template <int MAXC>
__device__ __forceinline__ void epilogue_rows(const EngineParams &p, const SegInfo &s, int r, float (&v)[MAXC],
                              float *scratch, int bar_id, volatile int *flags) {
  if (p.mode == MODE_LINEAR && p.vec_y) {
    // Through shared memory, half the columns at a time (scratch holds 128 x MAXC/2
    // fp32): thread r parks row r, then each thread adds R to and stores runs of 8 rows
    // of one column with 16-byte accesses. Per-lane 2-byte stores of 64 columns were
    // the slow part of a wide tile's epilogue. Every R run this thread adds is loaded
    // first: interleaved with the Y stores, each load would wait for the store before it
    // (the compiler cannot tell R and Y apart).
    constexpr int CW = MAXC >= 2 ? MAXC / 2 : 1;
    constexpr int NH = MAXC / CW;
    constexpr int NI = (CW * 16 + 127) / 128;  // runs per thread and half
    uint4 rr[NH][NI];
#pragma unroll
    for (int h = 0; h < NH; ++h)
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const int c = r + 128 * i;
        const int j = h * CW + (c >> 4), n0 = s.t * 128 + (c & 15) * 8;
        rr[h][i] = make_uint4(0u, 0u, 0u, 0u);
        if (p.R != nullptr && c < CW * 16 && j < s.ncols && n0 < p.N)
          rr[h][i] = *reinterpret_cast<const uint4 *>(
              p.R + static_cast<size_t>(s.xrow0 + j) * p.N + n0);
      }
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      named_bar_sync(bar_id, 128);
#pragma unroll
      for (int jj = 0; jj < CW; ++jj)
        if (h * CW + jj < s.ncols) scratch[jj * 128 + r] = v[h * CW + jj];
      named_bar_sync(bar_id, 128);
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const int c = r + 128 * i;
        const int jj = c >> 4, j = h * CW + jj;
        const int row8 = (c & 15) * 8, n0 = s.t * 128 + row8;
        if (c >= CW * 16 || j >= s.ncols || n0 >= p.N) continue;
        const float4 a = *reinterpret_cast<const float4 *>(scratch + jj * 128 + row8);
        const float4 b = *reinterpret_cast<const float4 *>(scratch + jj * 128 + row8 + 4);
        *reinterpret_cast<uint4 *>(p.Y + static_cast<size_t>(s.xrow0 + j) * p.N + n0) =
            pack_y8r(a, b, rr[h][i], p.R != nullptr);
      }
    }
  } else if (p.mode == MODE_LINEAR) {
    const int n = s.t * 128 + r;
    if (n < p.N) {
#pragma unroll
      for (int j = 0; j < MAXC; ++j) {
        if (j < s.ncols) {
          float y = v[j];
          const size_t off = static_cast<size_t>(s.xrow0 + j) * p.N + n;
          if (p.R != nullptr) y += bf16_to_f32(p.R[off]);
          p.Y[off] = f32_to_bf16_rn(y);
        }
      }
    }
  } else if (p.mode == MODE_GATEUP) {
    named_bar_sync(bar_id, 128);
    if (r >= 64) {
#pragma unroll
      for (int j = 0; j < MAXC; ++j)
        if (j < s.ncols) scratch[j * 64 + (r - 64)] = v[j];
    }
    named_bar_sync(bar_id, 128);
    if (r < 64) {
      const int i = s.t * 64 + r;
#pragma unroll
      for (int j = 0; j < MAXC; ++j) {
        if (j < s.ncols) {
          const float g = v[j];
          const float u = scratch[j * 64 + r];
          const float a = g / (1.f + expf(-g)) * u;
          p.A[static_cast<size_t>(s.xrow0 + j) * p.N + i] = f32_to_bf16_rn(a);
        }
      }
    }
  } else {  // MODE_DOWN
    const int n = s.t * 128 + r;
    if (n < p.N) {
#pragma unroll
      for (int j = 0; j < MAXC; ++j)
        if (j < s.ncols) p.Yp[static_cast<size_t>(s.xrow0 + j) * p.N + n] = v[j];
    }
    if (p.cmb_cnt != nullptr) combine_tail<MAXC>(p, s, r, scratch, bar_id);
  }
}

}  // namespace ssd
