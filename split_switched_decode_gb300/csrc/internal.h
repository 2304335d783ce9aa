// internal.h -- interface between the library's translation units (not installed).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ssd {

// Parameters of one launch of the split-K engine (see engine.cuh). Passed by value.
struct EngineParams {
  int mode;          // EngineMode
  int N;             // epilogue output width: LINEAR/FRONT rows of W, GATEUP I, DOWN H
  int K;             // reduction length
  int T;             // tiles per group
  int KB;            // 64-wide k-blocks per tile
  int G;             // workers (== gridDim.x), G <= T*KB
  int grouped;       // 0: one group of B columns; 1: groups = used experts of a route map
  int rm_ready;      // grouped: the route map was complete before the previous kernel of
                     // the stream started, so it may be read before the dependency wait
  int B;             // columns of the single group
  int w_group_rows;  // W rows per group in the weight bank (grouped)
  int up_row_off;    // GATEUP: row offset of the up half inside a group (= I)
  int slot_cols;     // columns per partial slot (slot = 128 * slot_cols floats)
  int defer;         // 1: store every segment's partial tile and stop (MODE_FRONT)
  int vec_y;         // LINEAR: N % 8 == 0 and Y (and R) 16-byte aligned: 16-byte stores
  int packed;        // W tile-packed: contiguous 16 KB blocks of 128 rows x 64 k, block
                     // (expert, tile, k-block) at (expert * T + tile) * KB + k-block (gate/up:
                     // 64 gate rows then the 64 matching up rows)
  int pair;          // LINEAR, tensor cores: 2-CTA clusters, CTA pair (2t, 2t+1) holds the two
                     // k-halves of tile t and adds them through distributed shared memory
  int ngrp;          // LINEAR, tensor cores: groups of 64 batch columns sharing each weight
                     // tile (B > 64: up to 4); 1 everywhere else
  int dyn;           // grouped, tensor cores: whole-tile schedule. Of the launch's tiles,
                     // CTA w first takes [w*S, (w+1)*S), S = floor(dyn * tiles / (256 * G)),
                     // then claims the rest one tile at a time from *dyn_ctr. 0: stream-K
  int *dyn_ctr;      // this launch's claim counter, zero when the launch starts (the gather
                     // launch before the routed launches clears it)
  int with_shared;   // one launch for gate/up and down: one more group after the used
                     // experts, the shared expert (its own tensor maps; activation rows
                     // P .. P+B-1, all B tokens)
  int *ready;        // one launch for gate/up and down: per used expert, the gate/up tiles
                     // whose rows of A are stored (zero at the start, cleared with dyn_ctr;
                     // dyn_ctr[1] counts them over all experts)
  int wbox_rows;     // rows per weight TMA box: 128 (one box per tile) or 64 (gate/up)
  const uint8_t *w_base;  // weight matrix (raw pointer, for L2 prefetch)
  long long w_rows;       // rows of the weight matrix (all groups)
  int l2pf_kb;            // k-blocks beyond the smem ring prefetched to L2 before the wait
  int xbox_rows;     // rows per activation TMA box: 16, or 16 x boxes of the widest group
  int E;             // experts (grouped route map, FRONT router rows)
  int P;             // B * topk (grouped route map)
  const int32_t *route_map;  // grouped: counts | offsets | pairs | pos | num_used | used
  // MODE_LINEAR
  uint16_t *Y;
  const uint16_t *R;
  // MODE_GATEUP / MODE_DOWN: output row = group's first activation row + column
  uint16_t *A;  // [rows, N] bf16
  float *Yp;    // [rows, N] fp32
  // MODE_DOWN inside moe_experts with the combine fused in: the tile that completes the
  // last of a (token, 128-row block)'s contributions (its routed experts' down tiles and
  // the shared expert's) writes that block of Y. nullptr: no fused combine.
  int *cmb_cnt;          // [B][T] arrivals, zero between calls
  int cmb_need;          // contributions per (token, block): topk (+1 with a shared expert)
  int topk;
  const float *topk_w;   // [B, topk]
  const float *cmb_yp;   // routed down outputs [P, N] fp32, rows in route-map order
  const float *cmb_s;    // shared expert output [B, N] fp32, or nullptr
  uint16_t *cmb_y;       // Y [B, N] bf16
  // split-K reduction
  float *partials;  // [2*G][128*slot_cols]
  int *counters;    // one per (group, tile), zero between launches
  // error reporting
  unsigned *status;
  uint64_t wait_limit_ns;
};

// ------------------------------------------------------------------ launch --
// Programmatic dependent launch on or off for this process (DEC_PDL=0 turns it off).
bool pdl_enabled();

// cudaLaunchKernelEx with programmatic stream serialisation when enabled, so the kernel
// may start (and load weights) while the previous kernel of the stream finishes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// The same with thread-block clusters of `cluster_x` CTAs along x (co-scheduled; their
// shared memory is mutually addressable).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t s, int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_x);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// ------------------------------------------------------------- engine_cc.cu --
int engine_maxc_for(int ncols);                 // 2, 4, 8, 16, 32 or 64
cudaError_t launch_engine_cc(int maxc, const CUtensorMap &wmap, const CUtensorMap &xmap,
                             const EngineParams &p, cudaStream_t s);

// ----------------------------------------------------------- engine_pair.cu --
// Wide projections (MODE_LINEAR, one group of p.B <= ncol columns, p.KB >= 2) on CTA-pair
// tensor-core tiles: clusters of 4 CTAs per 256 rows of W ((p.T + 1) / 2 clusters), the
// two k-halves added inside the cluster; ncol = pair_cols(p.B) is 128..512. wmap
// has 128-row boxes (or tile-packed blocks), xmap boxes of pair_xbox_rows(ncol) rows. With
// p.vec_y, ymap and rmap (R, when given) map Y and R [B, N] without swizzle in boxes of
// 128 x ncol / 2 elements; otherwise they are not read. No workspace.
int pair_cols(int B);  // 128 up to 128 rows, else B rounded up to a multiple of 64
inline int pair_xbox_rows(int ncol) { return (ncol > 256 ? ncol / 2 : ncol) / 2; }
cudaError_t engine_pair_max_clusters(int ncol, int *n);
cudaError_t launch_engine_pair(int ncol, const CUtensorMap &wmap, const CUtensorMap &xmap,
                               const CUtensorMap &ymap, const CUtensorMap &rmap,
                               const EngineParams &p, cudaStream_t s);

// ------------------------------------------------------------- engine_tc.cu --
cudaError_t launch_engine_tc(int maxc, const CUtensorMap &wmap, const CUtensorMap &xmap,
                             const EngineParams &p, cudaStream_t s);
// The routed gate/up (p1: wmap1, xmap1) and down (p2: wmap2, xmap2) GEMVs of a grouped
// expert layer in one launch of p1.G CTAs: every tile claimed from p1.dyn_ctr, down tiles
// after their expert's gate/up tiles have published A (p1.ready).
// With p1.with_shared, the shared expert is one more group, its weights read through
// wmap1s (gate/up) and wmap2s (down).
cudaError_t launch_engine_tc_moe(int maxc, const CUtensorMap &wmap1, const CUtensorMap &xmap1,
                                 const CUtensorMap &wmap2, const CUtensorMap &xmap2,
                                 const CUtensorMap &wmap1s, const CUtensorMap &wmap2s,
                                 const EngineParams &p1, const EngineParams &p2,
                                 cudaStream_t s);

// ------------------------------------------------------------- gemv_tiny.cu --
constexpr int TINY_MAX_NB = 4;  // batch rows of the tiny kernel (1..4)
int gemv_tiny_grid(int N, int K, int num_sms);
// packed: W in the tile-packed layout of dec_pack_weight instead of row-major [N,K].
cudaError_t launch_gemv_tiny(const uint16_t *X, const uint16_t *W, const uint16_t *R,
                             uint16_t *Y, int B, int N, int K, int num_sms, cudaStream_t s,
                             bool packed = false);
// Row-major W [N,K] -> tile-packed Wp (N % 128 == 0, K % 64 == 0): 16 KB blocks of 128
// rows x 64 k, block (n/128, k/64) at index (n/128)*(K/64) + k/64 (moe_aux.cu).
// gateup_I > 0: W is a gate/up bank [E, 2*gateup_I, K]; each block holds 64 gate rows
// then the 64 matching up rows of one expert (N = E * 2 * gateup_I).
cudaError_t launch_pack_weight(const uint16_t *W, int N, int K, uint16_t *Wp, cudaStream_t s,
                               int gateup_I = 0);

// --------------------------------------------------------------- moe_aux.cu --
// Second half of the front end: adds the product's partial tiles in worker order,
// writes logits and latent, routes each token and builds the route map.
struct FrontFinishParams {
  const float *partials;
  int slot_cols, G, T, KB;
  long long total;
  int B, E, L, topk;
  float *logits;
  uint16_t *latent;
  int32_t *topk_idx;
  float *topk_w;
  float *probs;
  int32_t *route_map;
  int *all_done;  // [1], zero between launches
  int cluster;    // 1: chunk 0's B <= 8 CTAs form a cluster that builds the route map
};
cudaError_t launch_front_finish(const FrontFinishParams &f, cudaStream_t s);

// The whole front end in one launch (front_fused.cu): T tiles of 128 W_cat rows, one
// thread-block cluster of S CTAs per tile, CTA c of a cluster multiplying k-blocks
// [c*KB/S, (c+1)*KB/S); the partials are added in the token-owning CTA (token b -> CTA
// b % S) after transfers through distributed shared memory; router CTAs publish the
// token's logits, and arrival counters elect the CTAs that route (a warp per token) and
// build the route map.
struct FrontFusedParams {
  int B, E, L, KB, T, S, log2S, TR, topk;
  int nst;       // stage-ring depth (weight + activation boxes of one k-block per stage)
  int nsl;       // token slots per CTA: ceil(B / S)
  int single_b;  // up to this batch one CTA routes every token and builds the route map
  int trig_late; // router CTAs trigger the next kernel once routed, not at their start
  uint16_t *latent;     // [B, L] bf16
  int32_t *topk_idx;    // [B, topk]
  float *topk_w;        // [B, topk]
  float *probs;         // [B, E] or nullptr
  float *logits;        // [B, E] workspace: router logits, fp32
  int32_t *route_map;   // or nullptr
  int *counter;         // arrivals of the router CTAs; zero between calls
  unsigned *status;
  uint64_t wait_limit_ns;
};
// dynamic shared memory the one-launch front end may request (below the 227 KB opt-in
// limit per CTA, leaving room for the compiler's static shared memory)
constexpr size_t FRONT_FUSED_SMEM_MAX = 220 * 1024;
size_t front_fused_smem(int S, int nxb, int nst, int nsl);
// Thread-block clusters of S CTAs with `smem` bytes each that the device can hold at once
// (0: the configuration cannot be launched).
int front_fused_max_clusters(int S, int nxb, size_t smem);
cudaError_t launch_front_fused(const CUtensorMap &wmap, const CUtensorMap &xmap,
                               const FrontFusedParams &p, int nxb, size_t smem, cudaStream_t s);

// Second half of a deferred split-K projection: adds the partial tiles of every worker
// in worker order, adds R and rounds to bf16.
struct LinearFinishParams {
  const float *partials;
  int slot_cols, G, T, KB, ngrp, vec_y;
  long long total;
  int B, N;
  const uint16_t *R;
  uint16_t *Y;
};
cudaError_t launch_linear_finish(const LinearFinishParams &f, cudaStream_t s);
// Validates topk_idx, builds the route map (written to route_map) and gathers in one
// launch of at most max_ctas CTAs. Both gather launches also zero dyn_reset[0..nreset)
// (the claim and ready counters of the routed launches after them), unless it is nullptr,
// and with shared_rows = B append X's B rows after the P gathered ones (the shared
// expert's activation rows when it runs inside the routed launch).
cudaError_t launch_gather_map(const uint16_t *X, const int32_t *topk_idx, int B, int topk, int E,
                              int K, uint16_t *Xg, int32_t *route_map, unsigned *status,
                              int max_ctas, int *dyn_reset, int nreset, int shared_rows,
                              cudaStream_t s);
cudaError_t launch_comm_wait(uint64_t ns, cudaStream_t s);
// Read-stream measurement: `ctas` CTAs claim 256 KB chunks (read_stream_claim_bytes) of
// the first `bytes` of p and read them into shared memory (moe_aux.cu).
size_t read_stream_claim_bytes();
cudaError_t launch_read_stream(const void *p, size_t bytes, int ctas, unsigned *status,
                               uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_gather_rows(const uint16_t *X, const int32_t *route_map, int B, int topk,
                               int E, int K, uint16_t *Xg, int *dyn_reset, int nreset,
                               int shared_rows, cudaStream_t s);
cudaError_t launch_combine(const float *topk_w, const int32_t *route_map, const float *Yp,
                           const float *S, int B, int topk, int E, int H, uint16_t *Y,
                           cudaStream_t s);
cudaError_t launch_l2_prefetch(const void *p, size_t bytes, int ctas, cudaStream_t s);
cudaError_t launch_wait_selftest(unsigned *status, uint64_t limit_ns, cudaStream_t s);

}  // namespace ssd
