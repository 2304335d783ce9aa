// routing.cuh -- softmax / top-k / renormalisation of router logits and the
// expert -> (token, slot) inverse map, as device functions run by one CTA.
//
// The routing step follows the router scores of "Hyper Optimizing Kimi K3 in vLLM",
// Part 1 / 3 "Improve MoE scheduling and overlap". The pages do not define it; the
// reading implemented here: softmax over the raw logits; the topk largest logits
// (compared in fp32) with ties to the lower expert index, listed by descending logit;
// weights renormalised over the chosen experts.
#pragma once

#include "common.cuh"

namespace ssd {

__device__ __forceinline__ float order_key_to_f32(uint32_t k) {
  return (k & 0x80000000u) ? __uint_as_float(k & 0x7FFFFFFFu) : __uint_as_float(~k);
}

// One warp routes token rows b = warp_id, warp_id + nwarps, ... of logits [B,E] (shared
// or global memory; L2_LOADS: global memory written by other CTAs of the same launch,
// read at L2). Writes topk_idx/topk_w (global) and, when given, probs (global)
// and sidx (shared copy of topk_idx for the route map). Register-only: every array
// index below is a compile-time constant after unrolling.
template <bool L2_LOADS = false>
__device__ __forceinline__ void route_tokens_warp(const float *logits, int B, int E, int topk,
                                                  int32_t *topk_idx, float *topk_w,
                                                  float *probs, int32_t *sidx, int warp_id,
                                                  int nwarps) {
  constexpr int VPL = MAX_E / 32;  // logits per lane
  const int lane = threadIdx.x & 31;
  const unsigned FULL = 0xFFFFFFFFu;
  for (int b = warp_id; b < B; b += nwarps) {
    const float *l = logits + static_cast<size_t>(b) * E;
    float v[VPL];
    uint32_t key[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      v[i] = (e < E) ? (L2_LOADS ? __ldcg(l + e) : l[e]) : -INFINITY;
      key[i] = (e < E) ? f32_order_key(v[i]) : 0u;  // 0: below every real key
    }
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPL; ++i) m = fmaxf(m, v[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));

    if (probs != nullptr) {
      float z = 0.f;
#pragma unroll
      for (int i = 0; i < VPL; ++i)
        if (lane + 32 * i < E) z += expf(v[i] - m);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(FULL, z, o);
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) probs[static_cast<size_t>(b) * E + e] = expf(v[i] - m) / z;
      }
    }

    // top-k: k rounds of a warp-wide arg-max on (logit desc, index asc). A lane keeps
    // the best of its remaining logits (bk, bi); a taken logit's key is zeroed and only
    // the lane that won the round rescans.
    uint32_t bk = 0;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (key[i] > bk) {  // strict: the lower index (smaller i) wins ties
        bk = key[i];
        bi = i;
      }
    int my_e = 0;
    float my_v = 0.f;
    for (int j = 0; j < topk; ++j) {
      const uint32_t kmax = __reduce_max_sync(FULL, bk);
      const uint32_t cand = (bk == kmax && bk != 0u) ? static_cast<uint32_t>(lane + 32 * bi)
                                                     : 0xFFFFFFFFu;
      const uint32_t win = __reduce_min_sync(FULL, cand);
      if (lane == static_cast<int>(win & 31u)) {
        const int wi = static_cast<int>(win >> 5);
        bk = 0;
        bi = 0;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          if (i == wi) key[i] = 0u;
          if (key[i] > bk) {
            bk = key[i];
            bi = i;
          }
        }
      }
      if (lane == j) {
        my_e = static_cast<int>(win);
        my_v = order_key_to_f32(kmax);
      }
    }
    float ex = (lane < topk) ? expf(my_v - m) : 0.f;
    float zs = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zs += __shfl_xor_sync(FULL, zs, o);
    if (lane < topk) {
      topk_idx[static_cast<size_t>(b) * topk + lane] = my_e;
      topk_w[static_cast<size_t>(b) * topk + lane] = ex / zs;
      if (sidx != nullptr) sidx[b * topk + lane] = my_e;
    }
  }
}

// Counting sort of the routing into the route-map layout of the public header, run by
// `nthreads` threads of one CTA (a multiple of 32, >= 32; `tid` = 0..nthreads-1, whole
// warps) that synchronise on named barrier `bar_id`. sidx: shared [B*topk] expert ids;
// smask: shared uint64 [E]; soff: shared int [E]. Requires B <= 64 (one bit per token).
__device__ __noinline__ static void build_route_map(const int32_t *sidx, int B, int topk, int E,
                                                    int32_t *rm, unsigned long long *smask,
                                                    int *soff, int nthreads, int bar_id,
                                                    int tid) {
  const int P = B * topk;
  int32_t *counts = rm;
  int32_t *offsets = rm + E;
  int32_t *pairs = rm + 2 * E + 1;
  int32_t *pos = pairs + P;
  int32_t *num_used = pos + P;
  int32_t *used = num_used + 1;

  for (int e = tid; e < E; e += nthreads) smask[e] = 0ull;
  named_bar_sync(bar_id, nthreads);
  for (int q = tid; q < P; q += nthreads)
    atomicOr(&smask[sidx[q]], 1ull << (q / topk));
  named_bar_sync(bar_id, nthreads);
  if (tid < 32) {
    const int lane = tid;
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int cnt = 0, nu = 0;
    for (int e = e0; e < e1; ++e) {
      const int c = __popcll(smask[e]);
      cnt += c;
      nu += (c > 0);
    }
    int icnt = cnt, inu = nu;  // inclusive scans across lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xFFFFFFFFu, icnt, o);
      const int c = __shfl_up_sync(0xFFFFFFFFu, inu, o);
      if (lane >= o) {
        icnt += a;
        inu += c;
      }
    }
    int run = icnt - cnt, runu = inu - nu;
    for (int e = e0; e < e1; ++e) {
      const int c = __popcll(smask[e]);
      counts[e] = c;
      offsets[e] = run;
      soff[e] = run;
      if (c > 0) used[runu++] = e;
      run += c;
    }
    if (lane == 31) {
      offsets[E] = icnt;
      *num_used = inu;
    }
  }
  named_bar_sync(bar_id, nthreads);
  for (int q = tid; q < P; q += nthreads) {
    const int e = sidx[q];
    const int b = q / topk;
    const int rank = __popcll(smask[e] & ((1ull << b) - 1ull));
    const int at = soff[e] + rank;
    pairs[at] = q;
    pos[q] = at;
  }
}

// The route map (layout of the public header) built by one warp without block
// barriers: token masks per expert by shared atomics, one warp-wide scan of the
// per-expert counts (each lane owns ceil(E/32) consecutive experts), then every
// (token, slot) entry placed by the rank of its token among the expert's tokens.
// sidx: shared [B*topk] expert ids (each in [0, E)); smask: shared uint64 [E]; soff:
// shared int [E]. Requires B <= 64. Run by all 32 lanes of one warp.
__device__ __noinline__ static void build_route_map_warp(const int32_t *sidx, int B, int topk,
                                                         int E, int32_t *rm,
                                                         unsigned long long *smask, int *soff) {
  const int lane = threadIdx.x & 31;
  const int P = B * topk;
  int32_t *counts = rm;
  int32_t *offsets = rm + E;
  int32_t *pairs = rm + 2 * E + 1;
  int32_t *pos = pairs + P;
  int32_t *num_used = pos + P;
  int32_t *used = num_used + 1;
  for (int e = lane; e < E; e += 32) smask[e] = 0ull;
  __syncwarp();
  for (int q = lane; q < P; q += 32) atomicOr(&smask[sidx[q]], 1ull << (q / topk));
  __syncwarp();
  const int per = (E + 31) / 32;
  const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
  int c = 0, u = 0;
  for (int e = e0; e < e1; ++e) {
    const int k = __popcll(smask[e]);
    c += k;
    u += (k > 0);
  }
  int ic = c, iu = u;  // inclusive scans across the lanes
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xFFFFFFFFu, ic, o);
    const int b = __shfl_up_sync(0xFFFFFFFFu, iu, o);
    if (lane >= o) {
      ic += a;
      iu += b;
    }
  }
  int run = ic - c, runu = iu - u;
  for (int e = e0; e < e1; ++e) {
    const int k = __popcll(smask[e]);
    counts[e] = k;
    offsets[e] = run;
    soff[e] = run;
    if (k > 0) used[runu++] = e;
    run += k;
  }
  if (lane == 31) {
    offsets[E] = ic;
    *num_used = iu;
  }
  __syncwarp();
  for (int q = lane; q < P; q += 32) {
    const int e = sidx[q];
    const int b = q / topk;
    const int at = soff[e] + __popcll(smask[e] & ((1ull << b) - 1ull));
    pairs[at] = q;
    pos[q] = at;
  }
}

}  // namespace ssd
