// moe_aux.cu -- small kernels around the grouped expert GEMV, the L2 prefetch kernel,
// the weight packing kernel, the simulated communication phase and the bounded-wait
// self-test.
#include "common.cuh"
#include "internal.h"
#include "routing.cuh"

namespace ssd {

namespace {

// Copy the caller's topk_idx [B*topk] into shared `sidx` and check it (0 <= e < E,
// distinct within a token). Run by all 256 threads of the CTA; `bad` is a shared flag.
// Returns the same verdict in every thread.
__device__ __forceinline__ bool load_routing(const int32_t *topk_idx, int B, int topk, int E,
                                             int32_t *sidx, volatile int *bad) {
  if (threadIdx.x == 0) *bad = 0;
  __syncthreads();
  for (int q = threadIdx.x; q < B * topk; q += 256) {
    const int e = topk_idx[q];
    sidx[q] = e;
    if (e < 0 || e >= E) *bad = 1;
  }
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += 256)
    for (int i = 0; i < topk; ++i)
      for (int j = i + 1; j < topk; ++j)
        if (sidx[b * topk + i] == sidx[b * topk + j]) *bad = 1;
  __syncthreads();
  return *bad == 0;
}

// An invalid routing yields an empty map (no used expert, zeros elsewhere) and
// ST_BAD_ROUTING, so no later launch reads a weight or row out of range.
__device__ __forceinline__ void empty_route_map(int B, int topk, int E, int32_t *rm,
                                                unsigned *status) {
  const int n = 3 * E + 2 + 2 * B * topk;
  for (int i = threadIdx.x; i < n; i += 256) rm[i] = 0;
  if (threadIdx.x == 0) atomicOr(status, ST_BAD_ROUTING);
}

// Routed-expert gather for a caller without a route map, in one launch: every CTA
// validates topk_idx and builds the whole route map in shared memory with all 256
// threads (a few KB, cheaper than a second launch and its memory round trip), CTA 0
// publishes it to rm for the grouped launches and the combine, and every CTA copies its
// share of the rows
// Xg[q, :] = X[pairs[q] / topk, :] with UNR independent 16-byte loads in flight per thread.
__global__ void __launch_bounds__(256) gather_map_kernel(const uint16_t *X,
                                                         const int32_t *topk_idx, int B,
                                                         int topk, int E, int K, uint16_t *Xg,
                                                         int32_t *rm, unsigned *status,
                                                         int *dyn_reset, int nreset,
                                                         int shared_rows) {
  griddep_wait();
  griddep_launch_dependents();
  // the claim and ready counters of the routed launches that follow
  if (dyn_reset != nullptr && blockIdx.x == 0)
    for (int i = threadIdx.x; i < nreset; i += 256) dyn_reset[i] = 0;
  __shared__ int32_t sidx[MAX_B * MAX_TOPK];
  __shared__ unsigned long long smask[MAX_E];
  __shared__ int soff[MAX_E];
  __shared__ int32_t smap[3 * MAX_E + 2 + 2 * MAX_B * MAX_TOPK];
  __shared__ int swarp[16];
  __shared__ int bad;
  if (!load_routing(topk_idx, B, topk, E, sidx, &bad)) {
    if (blockIdx.x == 0) empty_route_map(B, topk, E, rm, status);
    return;
  }
  build_route_map_cta(sidx, B, topk, E, smap, smask, soff, swarp);
  __syncthreads();
  const int P = B * topk;
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < 3 * E + 2 + 2 * P; i += 256) rm[i] = smap[i];
  const int32_t *pairs = smap + 2 * E + 1;
  const int chunks = K / 8;  // 16-byte chunks per row
  const int64_t n = static_cast<int64_t>(P + shared_rows) * chunks;
  constexpr int UNR = 4;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * 256;
  for (int64_t i0 = blockIdx.x * 256ll + threadIdx.x; i0 < n; i0 += stride * UNR) {
    uint4 v[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < n) {
        const int q = static_cast<int>(i / chunks);
        const int c = static_cast<int>(i - static_cast<int64_t>(q) * chunks);
        const int b = q < P ? pairs[q] / topk : q - P;  // a valid map: 0 <= b < B
        v[u] = reinterpret_cast<const uint4 *>(X + static_cast<size_t>(b) * K)[c];
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < n) {
        const int q = static_cast<int>(i / chunks);
        const int c = static_cast<int>(i - static_cast<int64_t>(q) * chunks);
        reinterpret_cast<uint4 *>(Xg + static_cast<size_t>(q) * K)[c] = v[u];
      }
    }
  }
}

// Contributors of tile t of a split of `total` iterations (KB per tile) over G workers
// (each worker spans at most two tiles): workers first..last, and the slot that holds
// the first worker's part (0 when its range starts inside the tile, else 1; the later
// workers all start inside it).
struct TileContrib {
  int first, last, which_first;
};
__device__ __forceinline__ TileContrib tile_contrib(int t, int KB, int G, long long total) {
  const long long tb = static_cast<long long>(t) * KB;
  TileContrib c;
  c.first = static_cast<int>(((tb + 1) * G - 1) / total);
  c.last = static_cast<int>(((tb + KB) * G - 1) / total);
  c.which_first = (static_cast<long long>(c.first) * total / G >= tb) ? 0 : 1;
  return c;
}

// Sum in worker order of element `off` (column * 128 + row) of tile t's partial slots.
__device__ __forceinline__ float sum_partials(const float *partials, size_t slot_floats,
                                              const TileContrib &c, size_t off) {
  constexpr int D = 32;  // a front tile has ~G*KB/total + 1 contributors: all in flight
  float z = 0.f;
  for (int wk0 = c.first; wk0 <= c.last; wk0 += D) {
    float part[D];
#pragma unroll
    for (int d = 0; d < D; ++d) {
      const int wk = wk0 + d;
      const int which = (wk == c.first) ? c.which_first : 0;
      part[d] = (wk <= c.last)
                    ? __ldcg(partials + static_cast<size_t>(wk * 2 + which) * slot_floats + off)
                    : 0.f;
    }
#pragma unroll
    for (int d = 0; d < D; ++d)
      if (wk0 + d <= c.last) z += part[d];
  }
  return z;
}

// Second half of the MoE front end, launched programmatically after the router +
// latent product (which only stored its partial tiles). CTA (b, c) owns rows
// 512c .. 512c+511 of token b; thread i adds row 512c+i's partials of every worker of
// its tile in worker order (the product kernel's split, recomputed here) with all
// loads in flight. Latent rows go out as bf16. CTA (b, 0) holds all E <= 512 router
// logits of token b in shared memory and routes the token with one warp. Spread over
// B * ceil((E+L)/512) CTAs, the reduction costs one memory round trip.
// The route map needs every token's routing. With f.cluster (B <= 8), the B CTAs of
// chunk 0 form one thread-block cluster: each puts its token's expert ids into CTA 0's
// shared memory and CTA 0 builds the map after a cluster barrier -- no global round
// trip. Otherwise the CTA that routes the last token (acquire-release counter) reads
// every token's ids back and builds it.
__global__ void __launch_bounds__(512) front_finish_kernel(const FrontFinishParams f) {
  __shared__ float slog[MAX_E];
  __shared__ int32_t sidx[MAX_B * MAX_TOPK];
  __shared__ unsigned long long smask[MAX_E];
  __shared__ int soff[MAX_E];
  __shared__ int flag;
  const int b = blockIdx.x, c = blockIdx.y, i = threadIdx.x;
  // c is uniform over a cluster (clusters span tokens only)
  const bool clustered = f.cluster && c == 0;
  if (clustered) cluster_arrive_relaxed();
  griddep_wait();
  griddep_launch_dependents();
  const int n = c * 512 + i;
  const size_t slot_floats = static_cast<size_t>(128) * f.slot_cols;
  if (n < f.E + f.L) {
    const TileContrib tc = tile_contrib(n >> 7, f.KB, f.G, f.total);
    const float z =
        sum_partials(f.partials, slot_floats, tc, static_cast<size_t>(b) * 128 + (n & 127));
    if (n < f.E) {
      slog[n] = z;
      f.logits[static_cast<size_t>(b) * f.E + n] = z;
    } else {
      f.latent[static_cast<size_t>(b) * f.L + (n - f.E)] = f32_to_bf16_rn(z);
    }
  }
  if (c != 0) return;  // only the chunk holding the router rows routes (uniform per CTA)
  __syncthreads();
  if (i < 32)
    route_tokens_warp(slog, 1, f.E, f.topk, f.topk_idx + static_cast<size_t>(b) * f.topk,
                      f.topk_w + static_cast<size_t>(b) * f.topk,
                      f.probs ? f.probs + static_cast<size_t>(b) * f.E : nullptr,
                      clustered ? sidx : nullptr, 0, 1);
  if (clustered) {
    // rank b == token b: its ids go to sidx[b*topk ..] of rank 0 (rank 0 writes its own
    // ids onto themselves); every CTA of the cluster has started once the wait returns
    cluster_wait();
    if (i < f.topk)  // lane i wrote sidx[i] itself
      st_cluster_u32(cluster_map(sidx + b * f.topk + i, 0u), static_cast<uint32_t>(sidx[i]));
    cluster_sync_all();
    if (b != 0) return;
    build_route_map(sidx, f.B, f.topk, f.E, f.route_map, smask, soff, 512, 1, i);
    return;
  }
  if (f.route_map == nullptr) return;
  __syncthreads();
  if (i == 0) flag = (atom_add_acq_rel_gpu(f.all_done, 1) == f.B - 1);
  __syncthreads();
  if (!flag) return;
  for (int q = i; q < f.B * f.topk; q += 512) sidx[q] = __ldcg(f.topk_idx + q);
  __syncthreads();
  build_route_map(sidx, f.B, f.topk, f.E, f.route_map, smask, soff, 512, 1, i);
  if (i == 0) *f.all_done = 0;
}

// Second half of a deferred split-K projection (launched programmatically): CTA
// (t, cb) owns rows t*128 .. t*128+127 and batch columns 16cb .. 16cb+15; thread r adds
// row r's partials in worker order, adds the residual and rounds once to bf16.
__global__ void __launch_bounds__(128) linear_finish_kernel(const LinearFinishParams f) {
  griddep_wait();
  griddep_launch_dependents();
  const int t = blockIdx.x, j0 = blockIdx.y * 16, r = threadIdx.x;
  const int n = t * 128 + r;
  const TileContrib tc = tile_contrib(t, f.KB, f.G, f.total);
  const size_t slot_floats = static_cast<size_t>(128) * f.slot_cols;
  // columns j0..j0+15 lie in one group of 64 (wide projections keep a slot per group)
  const int g = j0 >> 6, jj0 = j0 & 63;
  float z[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) z[j] = 0.f;
  for (int wk = tc.first; wk <= tc.last; ++wk) {
    const int which = (wk == tc.first) ? tc.which_first : 0;
    const float *sl =
        f.partials + (static_cast<size_t>(wk * 2 + which) * f.ngrp + g) * slot_floats + r;
    float part[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      part[j] = (j0 + j < f.B) ? __ldcg(sl + static_cast<size_t>(jj0 + j) * 128) : 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) z[j] += part[j];
  }
  if (f.vec_y) {
    // transpose through shared memory: each thread then finishes 8 consecutive rows of
    // one column with 16-byte R loads and Y stores
    __shared__ __align__(16) float sz[16][128];
#pragma unroll
    for (int j = 0; j < 16; ++j) sz[j][r] = z[j];
    __syncthreads();
    // both runs' residuals first: interleaved with the Y stores, the second load would
    // wait for the first store (the compiler cannot tell R and Y apart)
    uint4 rq[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int c = r + 128 * q;
      const int j = c >> 4, n0 = t * 128 + (c & 15) * 8;
      rq[q] = make_uint4(0u, 0u, 0u, 0u);
      if (f.R != nullptr && j0 + j < f.B && n0 < f.N)
        rq[q] = *reinterpret_cast<const uint4 *>(f.R + static_cast<size_t>(j0 + j) * f.N + n0);
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int c = r + 128 * q;  // 16 columns x 16 runs of 8 rows
      const int j = c >> 4, row8 = (c & 15) * 8, n0 = t * 128 + row8;
      if (j0 + j >= f.B || n0 >= f.N) continue;
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = sz[j][row8 + e];
      const size_t off = static_cast<size_t>(j0 + j) * f.N + n0;  // N % 8 == 0: whole run
      if (f.R != nullptr) {
        const uint4 rr = rq[q];
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
      *reinterpret_cast<uint4 *>(f.Y + off) = o;
    }
    return;
  }
  if (n >= f.N) return;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j0 + j < f.B) {
      float y = z[j];
      if (f.R != nullptr) y += bf16_to_f32(f.R[static_cast<size_t>(j0 + j) * f.N + n]);
      f.Y[static_cast<size_t>(j0 + j) * f.N + n] = f32_to_bf16_rn(y);
    }
  }
}

// Xg[q, :] = X[pairs[q] / topk, :] -- the activation rows of every (token, slot) entry
// in expert order, so each expert's rows are contiguous for the TMA tile loads.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t *X, const int32_t *rm,
                                                          int B, int topk, int E, int K,
                                                          uint16_t *Xg, int *dyn_reset,
                                                          int nreset, int shared_rows) {
  griddep_wait();
  griddep_launch_dependents();
  // the claim and ready counters of the routed launches that follow
  if (dyn_reset != nullptr && blockIdx.x == 0)
    for (int i = threadIdx.x; i < nreset; i += 256) dyn_reset[i] = 0;
  const int P = B * topk;
  const int32_t *pairs = rm + 2 * E + 1;
  const int chunks = K / 8;  // 16-byte chunks per row
  const int64_t n = static_cast<int64_t>(P + shared_rows) * chunks;
  for (int64_t i = blockIdx.x * 256ll + threadIdx.x; i < n; i += gridDim.x * 256ll) {
    const int q = static_cast<int>(i / chunks);
    const int c = static_cast<int>(i - static_cast<int64_t>(q) * chunks);
    const int b = q < P ? min(max(pairs[q] / topk, 0), B - 1) : q - P;
    const uint4 v = reinterpret_cast<const uint4 *>(X + static_cast<size_t>(b) * K)[c];
    reinterpret_cast<uint4 *>(Xg + static_cast<size_t>(q) * K)[c] = v;
  }
}

// Y[b,h] = bf16( sum_{j ascending} w[b,j] * Yp[pos[b,j], h]  (+ S[b,h]) ), fp32.
__global__ void __launch_bounds__(256) combine_kernel(const float *topk_w, const int32_t *rm,
                                                      const float *Yp, const float *S, int B,
                                                      int topk, int E, int H, uint16_t *Y) {
  griddep_wait();
  griddep_launch_dependents();
  const int P = B * topk;
  const int32_t *pos = rm + 2 * E + 1 + P;
  const int H4 = H / 4;
  const int64_t n = static_cast<int64_t>(B) * H4;
  for (int64_t i = blockIdx.x * 256ll + threadIdx.x; i < n; i += gridDim.x * 256ll) {
    const int b = static_cast<int>(i / H4);
    const int h4 = static_cast<int>(i - static_cast<int64_t>(b) * H4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < topk; ++j) {
      const float wj = topk_w[b * topk + j];
      const int at = min(max(pos[b * topk + j], 0), P - 1);
      const float4 y = reinterpret_cast<const float4 *>(Yp + static_cast<size_t>(at) * H)[h4];
      acc.x = fmaf(wj, y.x, acc.x);
      acc.y = fmaf(wj, y.y, acc.y);
      acc.z = fmaf(wj, y.z, acc.z);
      acc.w = fmaf(wj, y.w, acc.w);
    }
    if (S != nullptr) {
      const float4 sv = reinterpret_cast<const float4 *>(S + static_cast<size_t>(b) * H)[h4];
      acc.x += sv.x;
      acc.y += sv.y;
      acc.z += sv.z;
      acc.w += sv.w;
    }
    uint2 o;
    o.x = static_cast<uint32_t>(f32_to_bf16_rn(acc.x)) |
          (static_cast<uint32_t>(f32_to_bf16_rn(acc.y)) << 16);
    o.y = static_cast<uint32_t>(f32_to_bf16_rn(acc.z)) |
          (static_cast<uint32_t>(f32_to_bf16_rn(acc.w)) << 16);
    reinterpret_cast<uint2 *>(Y + static_cast<size_t>(b) * H)[h4] = o;
  }
}

// Each thread issues bulk L2 prefetches of PF_CHUNK bytes over the range; nothing is
// written and nothing waits: the copies into L2 proceed after the kernel retires.
constexpr uint32_t PF_CHUNK = 32768;

__global__ void __launch_bounds__(128) l2_prefetch_kernel(const uint8_t *p, size_t bytes) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x * PF_CHUNK;
  for (size_t off = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) * PF_CHUNK;
       off < bytes; off += stride) {
    const size_t left = bytes - off;
    const uint32_t n = left < PF_CHUNK ? static_cast<uint32_t>(left) : PF_CHUNK;
    prefetch_l2_bulk(p + off, n);
  }
}

// Waits on an mbarrier that nothing arrives at; must give up after limit_ns.
__global__ void wait_selftest_kernel(unsigned *status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  (void)mbar_wait_bounded(&bar, 0u, status, &abort_flag, limit_ns);
}

// Occupies its stream for ns nanoseconds (globaltimer) while touching no memory: a
// stand-in for a communication phase that leaves HBM idle.
// HBM read-stream measurement (dec_read_stream): every CTA claims 256 KB chunks of the
// buffer from a counter (*next, zeroed before the launch) until none is left and streams
// each into RS_STAGES rotating 16 KB shared-memory stages with 1-D bulk copies, one
// thread issuing and the stage's mbarrier counting the bytes; nothing is written
// anywhere. Claiming, rather than a fixed share per CTA, keeps SMs that happen to stream
// slower in a given call from setting its end. Every wait is bounded; after a time-out
// the copies still in flight land before the CTA exits.
constexpr int RS_STAGES = 8;
constexpr int RS_CHUNK = 16384;
constexpr int RS_CLAIM = 16;  // 16 KB pieces per claimed chunk
__device__ unsigned long long g_rs_next;  // the current call's next chunk (one per device)
__global__ void __launch_bounds__(32) read_stream_kernel(const uint8_t *p, long long nchunks,
                                                         unsigned long long *next,
                                                         unsigned *status, uint64_t limit_ns) {
  extern __shared__ __align__(1024) uint8_t rs_stage[];
  __shared__ __align__(8) uint64_t bar[RS_STAGES];
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  for (int s = 0; s < RS_STAGES; ++s) mbar_init(&bar[s], 1);
  fence_mbar_init();
  long long chunk = 0, k = 0;  // k: pieces issued by this CTA
  int sub = RS_CLAIM;          // pieces of the current chunk already issued
  for (;;) {
    if (sub == RS_CLAIM) {
      chunk = static_cast<long long>(atomicAdd(next, 1ull));
      sub = 0;
    }
    if (chunk >= nchunks) break;
    const int s = static_cast<int>(k % RS_STAGES);
    // the stage's previous piece must have landed before it is reused
    if (k >= RS_STAGES &&
        !mbar_wait_bounded(&bar[s], static_cast<uint32_t>(((k / RS_STAGES) - 1) & 1), status,
                           &abort_flag, limit_ns))
      break;
    mbar_arrive_expect_tx(&bar[s], RS_CHUNK);
    bulk_load_1d(rs_stage + s * RS_CHUNK, p + (chunk * RS_CLAIM + sub) * RS_CHUNK, RS_CHUNK,
                 &bar[s]);
    ++sub;
    ++k;
  }
  // the last pieces in flight (bounded; without a status update after a time-out)
  for (long long d = k > RS_STAGES ? k - RS_STAGES : 0; d < k; ++d) {
    if (abort_flag)
      (void)mbar_wait_drain(&bar[d % RS_STAGES], static_cast<uint32_t>((d / RS_STAGES) & 1),
                            10000000ull);
    else if (!mbar_wait_bounded(&bar[d % RS_STAGES], static_cast<uint32_t>((d / RS_STAGES) & 1),
                                status, &abort_flag, limit_ns))
      continue;
  }
}

__global__ void comm_wait_kernel(uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < ns) __nanosleep(256);
}

// Row-major W [N,K] -> tile-packed Wp: 16 KB blocks of 128 rows x 64 k (rows of 128
// bytes), block (n/128, k/64) at index (n/128)*KB + k/64, KB = K/64. For a gate/up bank
// (gate_I > 0: W = [E, 2 gate_I, K], gate rows then up rows per expert) block row r of
// block-row t' = e * (gate_I/64) + t is gate row t*64 + r (r < 64) or up row
// gate_I + t*64 + r - 64 of expert e. One thread per 16-byte chunk of Wp (stores
// coalesced; eight threads read one 128-byte row piece). A plain copy: run once when the
// weights are loaded, not in the decode step.
__global__ void __launch_bounds__(256) pack_weight_kernel(const uint4 *W, uint4 *Wp, int K,
                                                          long long chunks, int gate_I) {
  const int KB = K >> 6;
  const long long row_chunks = K >> 3;
  for (long long i = blockIdx.x * 256ll + threadIdx.x; i < chunks;
       i += static_cast<long long>(gridDim.x) * 256) {
    const long long block = i >> 10;          // 1024 chunks of 16 bytes per block
    const int r = static_cast<int>((i >> 3) & 127), c = static_cast<int>(i & 7);
    const long long t = block / KB, kb = block - t * KB;
    long long row = t * 128 + r;
    if (gate_I > 0) {
      const long long tpe = gate_I >> 6;  // 64-row gate tiles per expert
      const long long e = t / tpe, te = t - e * tpe;
      row = e * 2 * gate_I + (r < 64 ? te * 64 + r : gate_I + te * 64 + (r - 64));
    }
    Wp[i] = __ldg(W + row * row_chunks + kb * 8 + c);
  }
}

}  // namespace

cudaError_t launch_pack_weight(const uint16_t *W, int N, int K, uint16_t *Wp, cudaStream_t s,
                               int gateup_I) {
  const long long chunks = static_cast<long long>(N) * K / 8;
  long long blocks = (chunks + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  pack_weight_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      reinterpret_cast<const uint4 *>(W), reinterpret_cast<uint4 *>(Wp), K, chunks, gateup_I);
  return cudaGetLastError();
}

size_t read_stream_claim_bytes() { return static_cast<size_t>(RS_CLAIM) * RS_CHUNK; }

cudaError_t launch_read_stream(const void *p, size_t bytes, int ctas, unsigned *status,
                               uint64_t limit_ns, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(RS_STAGES) * RS_CHUNK;
  cudaError_t e = cudaFuncSetAttribute(read_stream_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  void *next = nullptr;
  if ((e = cudaGetSymbolAddress(&next, g_rs_next)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(next, 0, sizeof(unsigned long long), s)) != cudaSuccess) return e;
  read_stream_kernel<<<ctas, 32, smem, s>>>(
      static_cast<const uint8_t *>(p), static_cast<long long>(bytes / read_stream_claim_bytes()),
      static_cast<unsigned long long *>(next), status, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_comm_wait(uint64_t ns, cudaStream_t s) {
  comm_wait_kernel<<<1, 32, 0, s>>>(ns);
  return cudaGetLastError();
}

cudaError_t launch_front_finish(const FrontFinishParams &f, cudaStream_t s) {
  const dim3 grid(f.B, (f.E + f.L + 511) / 512);
  if (f.cluster) return launch_pdl_cluster(front_finish_kernel, grid, dim3(512), 0, s, f.B, f);
  return launch_pdl(front_finish_kernel, grid, dim3(512), 0, s, f);
}

cudaError_t launch_linear_finish(const LinearFinishParams &f, cudaStream_t s) {
  return launch_pdl(linear_finish_kernel, dim3(f.T, (f.B + 15) / 16), dim3(128), 0, s, f);
}

cudaError_t launch_gather_map(const uint16_t *X, const int32_t *topk_idx, int B, int topk, int E,
                              int K, uint16_t *Xg, int32_t *route_map, unsigned *status,
                              int max_ctas, int *dyn_reset, int nreset, int shared_rows,
                              cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(B * topk + shared_rows) * (K / 8);
  int64_t need = (n + 1023) / 1024;  // 256 threads x 4 chunks per CTA and sweep
  int grid = static_cast<int>(need < max_ctas ? need : max_ctas);
  if (grid < 1) grid = 1;
  return launch_pdl(gather_map_kernel, dim3(grid), dim3(256), 0, s, X, topk_idx, B, topk, E, K,
                    Xg, route_map, status, dyn_reset, nreset, shared_rows);
}

cudaError_t launch_gather_rows(const uint16_t *X, const int32_t *route_map, int B, int topk,
                               int E, int K, uint16_t *Xg, int *dyn_reset, int nreset,
                               int shared_rows, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(B * topk + shared_rows) * (K / 8);
  int grid = static_cast<int>((n + 255) / 256);
  if (grid > 1024) grid = 1024;
  return launch_pdl(gather_rows_kernel, dim3(grid), dim3(256), 0, s, X, route_map, B, topk, E, K,
                    Xg, dyn_reset, nreset, shared_rows);
}

cudaError_t launch_combine(const float *topk_w, const int32_t *route_map, const float *Yp,
                           const float *S, int B, int topk, int E, int H, uint16_t *Y,
                           cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(B) * (H / 4);
  int grid = static_cast<int>((n + 255) / 256);
  if (grid > 1024) grid = 1024;
  return launch_pdl(combine_kernel, dim3(grid), dim3(256), 0, s, topk_w, route_map, Yp, S, B, topk,
                    E, H, Y);
}

cudaError_t launch_l2_prefetch(const void *p, size_t bytes, int ctas, cudaStream_t s) {
  const size_t per_cta = static_cast<size_t>(128) * PF_CHUNK;
  size_t need = (bytes + per_cta - 1) / per_cta;
  int grid = static_cast<int>(need < static_cast<size_t>(ctas) ? need : static_cast<size_t>(ctas));
  if (grid < 1) grid = 1;
  l2_prefetch_kernel<<<grid, 128, 0, s>>>(static_cast<const uint8_t *>(p), bytes);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(unsigned *status, uint64_t limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace ssd
