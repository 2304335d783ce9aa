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

// Token masks of the route-map builders: bit b of expert e's 64-bit mask lives in the
// 32-bit word 2e + b/32 (set with 32-bit shared atomics, far cheaper than 64-bit ones);
// every access goes through this 32-bit view.
__device__ __forceinline__ uint64_t token_mask(const unsigned *m32, int e) {
  return (static_cast<uint64_t>(m32[2 * e + 1]) << 32) | m32[2 * e];
}
__device__ __forceinline__ void token_mask_set(unsigned *m32, int e, int b) {
  atomicOr(m32 + 2 * e + (b >> 5), 1u << (b & 31));
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

  unsigned *m32 = reinterpret_cast<unsigned *>(smask);
  for (int e = tid; e < E; e += nthreads) m32[2 * e] = m32[2 * e + 1] = 0u;
  named_bar_sync(bar_id, nthreads);
  for (int q = tid; q < P; q += nthreads) token_mask_set(m32, sidx[q], q / topk);
  named_bar_sync(bar_id, nthreads);
  if (tid < 32) {
    const int lane = tid;
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int cnt = 0, nu = 0;
    for (int e = e0; e < e1; ++e) {
      const int c = __popcll(token_mask(m32, e));
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
      const int c = __popcll(token_mask(m32, e));
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
    const int rank = __popcll(token_mask(m32, e) & ((1ull << b) - 1ull));
    const int at = soff[e] + rank;
    pairs[at] = q;
    pos[q] = at;
  }
}

// ------------------------------------------------------------ one-launch front end --

// Composite routing key: the order key of the fp32 logit in the high word, the
// inverted expert index in the low word. A larger key is a larger logit or, for equal
// logits, a lower expert index; keys of distinct experts differ; 0 is below every real
// candidate.
__device__ __forceinline__ uint64_t route_key(float logit, uint32_t expert) {
  return (static_cast<uint64_t>(f32_order_key(logit)) << 32) | (0xFFFFFFFFu - expert);
}

// Routes one token with one warp: softmax, the topk largest logits (ties to the lower
// expert index, listed by descending logit), weights renormalised over the chosen k.
// Lane l holds experts l, l+32, ... (16 per lane, E <= 512), read from global memory at
// L2 (written by other CTAs of the launch). Each lane first sorts its 16 keys in
// registers (bitonic network); each of the k rounds then takes a warp-wide max of the
// lanes' heads and the lowest expert among equal heads, and the winning lane drops its
// head -- two warp reductions per round and no rescan.
// Outputs: idx/w [topk] (global), probs [E] (global, optional), sidx [topk] (shared,
// optional).
__device__ __forceinline__ void route_token_sorted(const float *logits, int E, int topk,
                                                   int32_t *idx, float *w, float *probs,
                                                   int32_t *sidx) {
  constexpr int V = 16;
  const int lane = threadIdx.x & 31;
  const unsigned FULL = 0xFFFFFFFFu;
  float v[V];
  uint64_t k[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? __ldcg(logits + e) : -INFINITY;
    k[i] = e < E ? route_key(v[i], static_cast<uint32_t>(e)) : 0ull;
  }
  if (probs != nullptr) {  // full softmax over the E logits
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < V; ++i) m = fmaxf(m, v[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i)
      if (lane + 32 * i < E) z += expf(v[i] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(FULL, z, o);
#pragma unroll
    for (int i = 0; i < V; ++i)
      if (lane + 32 * i < E) probs[lane + 32 * i] = expf(v[i] - m) / z;
  }
#pragma unroll
  for (int s = 2; s <= V; s <<= 1) {  // sort the lane's keys, descending
#pragma unroll
    for (int d = s >> 1; d > 0; d >>= 1) {
#pragma unroll
      for (int i = 0; i < V; ++i) {
        if ((i & d) == 0) {
          const bool desc = (i & s) == 0;
          const uint64_t a = k[i], b = k[i + d];
          const uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
          k[i] = desc ? hi : lo;
          k[i + d] = desc ? lo : hi;
        }
      }
    }
  }
  uint32_t my_e = 0;
  float my_v = 0.f;
  for (int j = 0; j < topk; ++j) {
    const uint32_t hk = static_cast<uint32_t>(k[0] >> 32);
    const uint32_t kmax = __reduce_max_sync(FULL, hk);
    const uint32_t cand = (hk == kmax && k[0] != 0ull) ? 0xFFFFFFFFu - static_cast<uint32_t>(k[0])
                                                       : 0xFFFFFFFFu;
    const uint32_t win = __reduce_min_sync(FULL, cand);  // lowest expert with the max logit
    if (lane == static_cast<int>(win & 31u)) {           // expert win lives in lane win % 32
#pragma unroll
      for (int i = 0; i < V - 1; ++i) k[i] = k[i + 1];
      k[V - 1] = 0ull;
    }
    if (lane == j) {
      my_e = win;
      my_v = order_key_to_f32(kmax);
    }
  }
  const float m0 = __shfl_sync(FULL, my_v, 0);  // the largest logit
  const float ex = lane < topk ? expf(my_v - m0) : 0.f;
  float zs = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) zs += __shfl_xor_sync(FULL, zs, o);
  if (lane < topk) {
    idx[lane] = static_cast<int32_t>(my_e);
    w[lane] = ex / zs;
    if (sidx != nullptr) sidx[lane] = static_cast<int32_t>(my_e);
  }
}

// k rounds over the sorted per-lane lists k[0..V) of a warp: each round takes the
// largest head logit and, among equal ones, the lowest expert; the winning lane drops
// its head. Lane j < topk ends with the j-th choice (expert, logit); a lane with no
// choice (fewer than topk real keys) keeps expert 0xFFFFFFFF.
template <int V>
__device__ __forceinline__ void warp_rounds(uint64_t (&k)[V], int topk, uint32_t &my_e,
                                            float &my_v) {
  const int lane = threadIdx.x & 31;
  const unsigned FULL = 0xFFFFFFFFu;
  my_e = 0xFFFFFFFFu;
  my_v = 0.f;
  for (int j = 0; j < topk; ++j) {
    const uint32_t hk = static_cast<uint32_t>(k[0] >> 32);
    const uint32_t kmax = __reduce_max_sync(FULL, hk);
    const uint32_t cand = (hk == kmax && k[0] != 0ull) ? 0xFFFFFFFFu - static_cast<uint32_t>(k[0])
                                                       : 0xFFFFFFFFu;
    const uint32_t win = __reduce_min_sync(FULL, cand);
    const uint32_t src = __ffs(__ballot_sync(FULL, cand == win && win != 0xFFFFFFFFu)) - 1;
    if (win != 0xFFFFFFFFu && lane == static_cast<int>(src)) {
#pragma unroll
      for (int i = 0; i < V - 1; ++i) k[i] = k[i + 1];
      k[V - 1] = 0ull;
    }
    if (lane == j) {
      my_e = win;
      my_v = order_key_to_f32(kmax);
    }
  }
}

template <int V>
__device__ __forceinline__ void sort_desc_lane(uint64_t (&k)[V]) {
#pragma unroll
  for (int s = 2; s <= V; s <<= 1) {
#pragma unroll
    for (int d = s >> 1; d > 0; d >>= 1) {
#pragma unroll
      for (int i = 0; i < V; ++i) {
        if ((i & d) == 0) {
          const bool desc = (i & s) == 0;
          const uint64_t a = k[i], b = k[i + d];
          const uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
          k[i] = desc ? hi : lo;
          k[i + d] = desc ? lo : hi;
        }
      }
    }
  }
}

// Candidates a warp keeps for the exact ranking of route_token_filtered (more: the token
// is routed by k warp rounds instead).
constexpr int RT_CMAX = 64;

// Routes one token with one warp: the topk largest logits (ties to the lower expert index,
// listed by descending logit), weights renormalised over the chosen k -- the same choices
// and the same weight arithmetic as route_token_sorted, without the full softmax. Lane l
// holds experts l, l+32, ... (E <= 512), read from global memory at L2 (written by other
// CTAs of the launch).
//   1. Lower bound: every lane's largest key is one candidate per lane; the topk-th
//      largest of those 32 heads (by logit) bounds the topk-th largest logit from below,
//      since the topk lanes with the largest heads hold topk distinct keys at or above it.
//   2. Filter: the keys whose logit reaches the bound (every chosen expert among them,
//      typically 8-16 of 384) are appended to a shared list in lane order (ballots).
//   3. Rank: each candidate counts the candidates above it; rank j < topk is choice j.
// No step waits on another lane's choice, unlike k rounds of warp reductions. With more
// than RT_CMAX candidates (many equal logits) the warp sorts its registers and takes k
// rounds, as route_token_sorted does.
// scratch: shared uint64 [RT_CMAX + MAX_TOPK] of this warp. Outputs: idx/w [topk]
// (global), sidx [topk] (shared, optional). trigger: once the logits are in registers,
// let the next kernel of the stream be scheduled (programmatic dependent launch).
// V: logits per lane, E <= 32 V (12 covers 384 experts; 16 the 512 maximum).
template <int V>
__device__ __forceinline__ void route_token_filtered(const float *logits, int E, int topk,
                                                     int32_t *idx, float *w, int32_t *sidx,
                                                     uint64_t *scratch, bool trigger = false) {
  static_assert(V >= 1 && V <= MAX_E / 32, "logits per lane");
  const int lane = threadIdx.x & 31;
  const unsigned FULL = 0xFFFFFFFFu;
  uint64_t k[V];
  uint32_t head = 0u;  // this lane's largest logit key (0: no expert)
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    k[i] = e < E ? route_key(__ldcg(logits + e), static_cast<uint32_t>(e)) : 0ull;
    head = max(head, static_cast<uint32_t>(k[i] >> 32));
  }
  if (trigger) {
    asm volatile("" ::"r"(head));  // every load of this lane has returned
    __syncwarp();
    if (lane == 0) griddep_launch_dependents();
  }
  // 1. the topk-th largest head: the smallest head with fewer than topk heads above it
  int above = 0;
#pragma unroll
  for (int h = 0; h < 32; ++h) above += __shfl_sync(FULL, head, h) > head;
  const uint32_t bound = __reduce_min_sync(FULL, above < topk ? head : 0xFFFFFFFFu);
  // 2. candidates in lane order
  uint64_t *cand = scratch, *slot = scratch + RT_CMAX;
  const unsigned lower = (1u << lane) - 1u;
  int C = 0;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const bool in = k[i] != 0ull && static_cast<uint32_t>(k[i] >> 32) >= bound;
    const unsigned bal = __ballot_sync(FULL, in);
    const int at = C + __popc(bal & lower);
    if (in && at < RT_CMAX) cand[at] = k[i];
    C += __popc(bal);
  }
  __syncwarp();
  uint32_t my_e = 0xFFFFFFFFu;
  float my_v = 0.f;
  if (C <= RT_CMAX) {
    // 3. exact ranks (keys of distinct experts differ)
    const uint64_t a0 = lane < C ? cand[lane] : 0ull;
    const uint64_t a1 = lane + 32 < C ? cand[lane + 32] : 0ull;
    int r0 = 0, r1 = 0;
#pragma unroll 4
    for (int j = 0; j < C; ++j) {
      const uint64_t x = cand[j];
      r0 += x > a0;
      r1 += x > a1;
    }
    if (lane < C && r0 < topk) slot[r0] = a0;
    if (lane + 32 < C && r1 < topk) slot[r1] = a1;
    __syncwarp();
    if (lane < topk) {
      const uint64_t kk = slot[lane];
      my_e = 0xFFFFFFFFu - static_cast<uint32_t>(kk);
      my_v = order_key_to_f32(static_cast<uint32_t>(kk >> 32));
    }
    __syncwarp();  // slots read before the scratch is reused
  } else {  // the sorting network wants a power of two: pad with empty keys
    uint64_t k16[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) k16[i] = i < V ? k[i] : 0ull;
    sort_desc_lane<16>(k16);
    warp_rounds<16>(k16, topk, my_e, my_v);
  }
  const float m0 = __shfl_sync(FULL, my_v, 0);  // the largest logit
  const float ex = lane < topk ? expf(my_v - m0) : 0.f;
  float zs = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) zs += __shfl_xor_sync(FULL, zs, o);
  if (lane < topk) {
    idx[lane] = static_cast<int32_t>(my_e);
    w[lane] = ex / zs;
    if (sidx != nullptr) sidx[lane] = static_cast<int32_t>(my_e);
  }
}

// The route map (layout of the public header) built by every thread of the CTA, each
// thread owning two consecutive experts (E <= 2 * blockDim.x): per-expert token masks by
// shared atomics; the counts scanned within each warp by shuffles and across warps from
// the warp totals in shared memory; counts / offsets / used written by their owners;
// every (token, slot) entry placed by the rank of its token among the expert's tokens.
// Four CTA barriers, no serial loop. sidx: shared [B*topk] expert ids in [0, E);
// scratch in shared memory: smask uint64 [E], soff int [E], swarp int [2 * warps].
// Requires B <= 64.
__device__ __noinline__ static void build_route_map_cta(const int32_t *sidx, int B, int topk,
                                                        int E, int32_t *rm,
                                                        unsigned long long *smask, int *soff,
                                                        int *swarp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = B * topk;
  int32_t *counts = rm;
  int32_t *offsets = rm + E;
  int32_t *pairs = rm + 2 * E + 1;
  int32_t *pos = pairs + P;
  int32_t *num_used = pos + P;
  int32_t *used = num_used + 1;
  const int e0 = 2 * tid, e1 = e0 + 1;
  unsigned *m32 = reinterpret_cast<unsigned *>(smask);
  if (e0 < E) m32[2 * e0] = m32[2 * e0 + 1] = 0u;
  if (e1 < E) m32[2 * e1] = m32[2 * e1 + 1] = 0u;
  __syncthreads();
  for (int q = tid; q < P; q += blockDim.x) token_mask_set(m32, sidx[q], q / topk);
  __syncthreads();
  const int c0 = e0 < E ? __popcll(token_mask(m32, e0)) : 0;
  const int c1 = e1 < E ? __popcll(token_mask(m32, e1)) : 0;
  const int c = c0 + c1, u = (c0 > 0) + (c1 > 0);
  int ic = c, iu = u;  // inclusive scans within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xFFFFFFFFu, ic, o);
    const int b = __shfl_up_sync(0xFFFFFFFFu, iu, o);
    if (lane >= o) {
      ic += a;
      iu += b;
    }
  }
  if (lane == 31) {
    swarp[2 * warp] = ic;
    swarp[2 * warp + 1] = iu;
  }
  __syncthreads();
  int bc = 0, bu = 0;  // totals of the warps before this one
  for (int w = 0; w < warp; ++w) {
    bc += swarp[2 * w];
    bu += swarp[2 * w + 1];
  }
  const int o0 = bc + ic - c, u0 = bu + iu - u;
  if (e0 < E) {
    counts[e0] = c0;
    offsets[e0] = o0;
    soff[e0] = o0;
    if (c0 > 0) used[u0] = e0;
  }
  if (e1 < E) {
    counts[e1] = c1;
    offsets[e1] = o0 + c0;
    soff[e1] = o0 + c0;
    if (c1 > 0) used[u0 + (c0 > 0)] = e1;
  }
  if (tid == blockDim.x - 1) {
    offsets[E] = o0 + c;
    *num_used = u0 + u;
  }
  __syncthreads();
  for (int q = tid; q < P; q += blockDim.x) {
    const int e = sidx[q];
    const int b = q / topk;
    const int at = soff[e] + __popcll(token_mask(m32, e) & ((1ull << b) - 1ull));
    pairs[at] = q;
    pos[q] = at;
  }
}

}  // namespace ssd
