// api.cu -- host side of the C ABI declared in include/split_switched_decode.h:
// argument checks, the batch-size kernel switch, workspace planning, TMA descriptor
// encoding, side-stream scheduling of the shared expert, and error reporting.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/split_switched_decode.h"
#include "common.cuh"
#include "internal.h"

using namespace ssd;

namespace ssd {
bool pdl_enabled() {
  static const bool on = [] {
    const char *s = std::getenv("DEC_PDL");
    return !(s && s[0] == '0');
  }();
  return on;
}
}  // namespace ssd

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;

// Device status word: set by a kernel whose bounded wait ran out.
__device__ unsigned g_dec_status_word;

std::atomic<int> g_force_variant{-2};  // -2: not read from the environment yet
std::atomic<int> g_fault_inject{0};
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
thread_local int t_last_variant = DEC_VARIANT_NONE;

struct DeviceInfo {
  std::once_flag once;
  int num_sms = 0;
  unsigned *status = nullptr;
  cudaError_t err = cudaSuccess;
};
DeviceInfo g_dev[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Current device's info; nullptr (and *err set) when no device is usable.
DeviceInfo *device_info(cudaError_t *err) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = (e != cudaSuccess) ? e : cudaErrorInvalidDevice;
    return nullptr;
  }
  DeviceInfo &d = g_dev[dev];
  std::call_once(d.once, [&]() {
    d.err = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (d.err == cudaSuccess)
      d.err = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_dec_status_word);
  });
  if (d.err != cudaSuccess) {
    *err = d.err;
    return nullptr;
  }
  return &d;
}

int current_num_sms() {
  cudaError_t e;
  DeviceInfo *d = device_info(&e);
  return d ? d->num_sms : 0;
}

bool encoder_ready() {
  std::call_once(g_encode_once, []() {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode != nullptr;
}

// 2-D bf16 tensor [rows, inner] (inner contiguous), 128-byte swizzled boxes of
// 64 x box_rows elements.
bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows,
              uint32_t box_rows) {
  if (!encoder_ready()) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(TILE_K), box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A plain (unswizzled) 2-D map of a bf16 [rows, inner] tensor with boxes of box_inner x
// box_rows elements, for whole-tile TMA loads and stores of outputs.
bool make_map_plain(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows,
                    uint32_t box_inner, uint32_t box_rows) {
  if (!encoder_ready()) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int force_variant() {
  int v = g_force_variant.load();
  if (v == -2) {
    int init = DEC_VARIANT_NONE;
    if (const char *s = std::getenv("DEC_FORCE_VARIANT")) {
      if (!std::strcmp(s, "tiny")) init = DEC_VARIANT_TINY;
      else if (!std::strcmp(s, "splitk")) init = DEC_VARIANT_SPLITK;
      else if (!std::strcmp(s, "splitk_tc")) init = DEC_VARIANT_SPLITK_TC;
    }
    int expected = -2;
    g_force_variant.compare_exchange_strong(expected, init);
    v = g_force_variant.load();
  }
  return v;
}

// Host-side fault injection: true when this launch must be reported as failed.
bool consume_fault() {
  int n = g_fault_inject.load();
  while (n > 0) {
    if (g_fault_inject.compare_exchange_weak(n, n - 1)) return true;
  }
  return false;
}

dec_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DEC_OK : DEC_ERR_CUDA; }

// ------------------------------------------------------------ split-K planning --

struct SplitPlan {
  int T, KB, G, maxc, ngrp;  // ngrp: groups of 64 batch columns (B > 64: tensor cores only)
  size_t partial_bytes, counter_bytes, total;
};

// Batch from which a split-K projection with 2 * tiles >= 80 % of the SMs splits every
// tile into two halves instead of one equal range per SM (DEC_PAIR_SPLIT_MIN_B; 0 =
// never).
int pair_split_min_batch() {
  if (const char *s = std::getenv("DEC_PAIR_SPLIT_MIN_B")) {
    int v = std::atoi(s);
    return v >= 1 ? v : 1 << 30;
  }
  return 2;  // measured on the input projection: 0.8-3.4 us faster at B = 2..64
}

// Widest tile (batch columns, a power of two) whose two k-halves are added inside a
// 2-CTA cluster (DEC_PAIR_DSMEM_COLS; 0 = never, which leaves the halves to the
// last-arriver reduction through global memory). Measured on the input projection at
// B = 64: 22.8 instead of 25.5 us.
int pair_dsmem_max_cols() {
  if (const char *s = std::getenv("DEC_PAIR_DSMEM_COLS")) return std::atoi(s);
  return 64;
}

// Smallest share of the SMs (percent) that two workers per tile must cover for the
// two-halves split (DEC_PAIR_SPLIT_MIN_SM_PCT).
int pair_split_min_sm_pct() {
  if (const char *s = std::getenv("DEC_PAIR_SPLIT_MIN_SM_PCT")) return std::atoi(s);
  return 80;
}

// Whether a projection of this shape splits its tiles into two k-halves that run as
// 2-CTA clusters (the "pair" schedule; batch threshold aside).
bool pair_shape(int N, int K, int num_sms) {
  const int T = ceil_div(N, TILE_N), KB = ceil_div(K, TILE_K);
  return 2 * T <= num_sms && 200 * T >= pair_split_min_sm_pct() * num_sms && KB >= 2 &&
         KB % 2 == 0 && pair_dsmem_max_cols() >= 2;
}

// The batch-size switch's tiny-kernel range: B <= 2, except that a shape on the pair
// schedule takes tensor cores from B = 2 (measured on the input projection: 21.7
// instead of 22.6 us at B = 2; at B = 1 the tiny kernel stays ahead, 20.5 vs 21.8 us).
// The kernel takes up to 4 rows, but from 3 rows it is issue-bound (output projection
// 40.7 / 47.7 us at B = 3 / 4 against 41.2 / 41.1 us on tensor cores). DEC_TINY_MAX_B
// overrides (at most 4).
int tiny_max_batch(int N, int K, int num_sms) {
  if (const char *s = std::getenv("DEC_TINY_MAX_B")) return std::min(std::atoi(s), TINY_MAX_NB);
  return pair_shape(N, K, num_sms) && pair_split_min_batch() <= 2 ? 1 : 2;
}

// Workers: split_k == 0 -> one per SM (at most T*KB); S > 0 -> T*S (classic split-K).
bool plan_splitk(int B, int N, int K, int split_k, int num_sms, SplitPlan *pl) {
  pl->T = ceil_div(N, TILE_N);
  pl->KB = ceil_div(K, TILE_K);
  const int64_t iters = static_cast<int64_t>(pl->T) * pl->KB;
  if (split_k == 0) {
    pl->G = static_cast<int>(iters < num_sms ? iters : num_sms);
    // When two workers per tile still cover at least 80 % of the SMs, give every tile
    // exactly two k-halves: one partial to add instead of two or three, and on tensor
    // cores the two halves run as a 2-CTA cluster that adds them on chip.
    if (B >= pair_split_min_batch() && 2 * pl->T <= num_sms &&
        200 * pl->T >= pair_split_min_sm_pct() * num_sms && pl->KB >= 2)
      pl->G = 2 * pl->T;
  } else {
    if (split_k > pl->KB) return false;
    const int64_t g = static_cast<int64_t>(pl->T) * split_k;
    if (g > (1 << 20)) return false;
    pl->G = static_cast<int>(g);
  }
  if (pl->G < 1) return false;
  pl->ngrp = B > MAX_B ? (B <= 2 * MAX_B ? 2 : 4) : 1;
  pl->maxc = engine_maxc_for(B > MAX_B ? MAX_B : B);
  pl->partial_bytes = align_up(static_cast<size_t>(2) * pl->G * pl->ngrp * 128 * pl->maxc *
                               sizeof(float));
  pl->counter_bytes = align_up(static_cast<size_t>(pl->T) * pl->ngrp * sizeof(int));
  pl->total = pl->partial_bytes + pl->counter_bytes;
  return true;
}

// k-blocks of weights each worker prefetches to L2 before its dependency wait
// (DEC_L2PF_KB overrides; 0 turns it off).
int l2_prefetch_kblocks() {
  if (const char *s = std::getenv("DEC_L2PF_KB")) return std::atoi(s) < 0 ? 0 : std::atoi(s);
  return 0;  // measured: the projections slow down (prefetch traffic competes); off
}

// Activation box height for a launch whose groups have at most maxc columns: one box
// covers them all (fewer TMA instructions per stage). A wide projection's box holds
// every batch row (B <= 256 rows).
int xbox_rows_for(int maxc) { return 16 * ((maxc + 15) / 16); }
int xbox_rows_for(const SplitPlan &pl, int B) {
  return pl.ngrp > 1 ? 16 * ((B + 15) / 16) : xbox_rows_for(pl.maxc);
}

void fill_engine_common(EngineParams &p, const SplitPlan &pl, int mode, int N, int K, int B,
                        void *ws, const DeviceInfo *d) {
  std::memset(&p, 0, sizeof p);
  p.mode = mode;
  p.N = N;
  p.K = K;
  p.T = pl.T;
  p.KB = pl.KB;
  p.G = pl.G;
  p.B = B;
  p.slot_cols = pl.maxc;
  p.ngrp = pl.ngrp;
  p.wbox_rows = 128;
  p.xbox_rows = xbox_rows_for(pl, B);
  p.l2pf_kb = l2_prefetch_kblocks();
  p.partials = static_cast<float *>(ws);
  p.counters = reinterpret_cast<int *>(static_cast<char *>(ws) + pl.partial_bytes);
  p.status = d->status;
  p.wait_limit_ns = g_wait_limit_ns.load();
}

dec_status check_linear_args(const dec_bf16 *X, const dec_bf16 *W, dec_bf16 *Y, int B, int N,
                             int K) {
  if (!X || !W || !Y) return DEC_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || K < 1) return DEC_ERR_INVALID_ARG;
  if (B > MAX_ROWS) return DEC_ERR_UNSUPPORTED_SHAPE;
  if (K % 8 != 0) return DEC_ERR_MISALIGNED;
  if (!aligned16(X) || !aligned16(W)) return DEC_ERR_MISALIGNED;
  if (static_cast<int64_t>(N) * K > (int64_t(1) << 40)) return DEC_ERR_UNSUPPORTED_SHAPE;
  return DEC_OK;
}

// Batch at and above which split-K projections with K >= 12288 defer their reduction
// to a finishing kernel (DEC_DEFER_MIN_B overrides the batch; the K condition stays).
// With long K each tile's workers hold long ranges and the last worker's 32..64-column
// reduction is a visible tail; with short K the extra launch costs more than it saves.
int defer_min_batch() {
  if (const char *s = std::getenv("DEC_DEFER_MIN_B")) {
    int v = std::atoi(s);
    if (v >= 1) return v;
  }
  return 32;  // measured on the K = 16384 output projection: B = 32 and 64 gain 2-8 us
}

// Reduction depth (K) from which wide-batch projections defer (DEC_DEFER_MIN_K).
int defer_min_k() {
  if (const char *s = std::getenv("DEC_DEFER_MIN_K")) {
    int v = std::atoi(s);
    if (v >= 0) return v;
  }
  return 12288;
}

// Slack on the shared expert's share of the SMs next to the routed experts
// (DEC_SIDE_SLACK, 1.0 .. 2.0; default 1.25): its fair share is num_sms / (U + 1).
double side_slack() {
  if (const char *s = std::getenv("DEC_SIDE_SLACK")) {
    const double v = std::atof(s);
    if (v >= 1.0 && v <= 2.0) return v;
  }
  return 1.25;
}

// Whole-tile schedule of the routed-expert launches (tensor cores): the static share of
// the tiles, in 1/256 (DEC_EXPERT_DYN, 0 = stream-K ranges), and the expected tiles per
// CTA from which a launch uses it (DEC_EXPERT_DYN_MIN_TILES).
int expert_dyn() {
  if (const char *s = std::getenv("DEC_EXPERT_DYN")) {
    const int v = std::atoi(s);
    if (v >= 0 && v <= 256) return v;
  }
  return 230;
}
double expert_dyn_min_tiles() {
  if (const char *s = std::getenv("DEC_EXPERT_DYN_MIN_TILES")) {
    const double v = std::atof(s);
    if (v >= 0.0) return v;
  }
  return 6.5;
}

// Routed gate/up and down in one launch (tensor cores; DEC_EXPERT_ONE_LAUNCH=0: two
// launches, whole-tile or stream-K as above).
bool expert_one_launch() {
  if (const char *s = std::getenv("DEC_EXPERT_ONE_LAUNCH")) return std::atoi(s) != 0;
  return true;
}

// With the routed experts in one launch: the shared expert's tiles join that launch as
// one more group, claimed by every SM, instead of running on the side stream
// (DEC_SHARED_IN_ROUTED=0 keeps the side stream; a caller's side_max_ctas > 0 does too).
bool shared_in_routed() {
  if (const char *s = std::getenv("DEC_SHARED_IN_ROUTED")) return std::atoi(s) != 0;
  return true;
}

// Whether grouped launches whose route map is already complete read it, and issue their
// first weight loads, before the dependency wait (DEC_EARLY_ROUTE_MAP=0 turns it off).
bool early_route_map() {
  if (const char *s = std::getenv("DEC_EARLY_ROUTE_MAP")) return std::atoi(s) != 0;
  return true;
}

// Whether the front end's finishing kernel builds the route map inside one thread-block
// cluster over the tokens (B <= 8) instead of in the CTA that routes the last token
// (DEC_FRONT_CLUSTER=0 turns it off).
bool front_cluster() {
  if (const char *s = std::getenv("DEC_FRONT_CLUSTER")) return std::atoi(s) != 0;
  return true;
}

// Whether moe_experts, given a route map, adds the routed and shared outputs into Y
// inside the down launches' epilogues (the tile that completes a (token, block) does
// it) instead of in a separate combine launch (DEC_FUSED_COMBINE=0/1 overrides).
bool fused_combine() {
  if (const char *s = std::getenv("DEC_FUSED_COMBINE")) return std::atoi(s) != 0;
  return false;
}

// Wide projections (B > 64) defer their reduction to the finishing kernel unless
// DEC_WIDE_DEFER=0.
bool wide_defer() {
  if (const char *s = std::getenv("DEC_WIDE_DEFER")) return std::atoi(s) != 0;
  return true;
}

// The batch at and above which split-K work uses tensor-core tiles rather than CUDA-core
// tiles (dec_linear sends the smallest batches to the tiny kernel first).
int tc_min_batch() {
  if (const char *s = std::getenv("DEC_TC_MIN_B")) {
    int v = std::atoi(s);
    if (v >= 1) return v;
  }
  // measured: tensor-core tiles win at every batch -- projections from B = 2 (CUDA
  // cores are ALU-bound from B ~ 4), the front end at B = 1-2 (13.1 vs 13.8 us) and the
  // expert layer at B = 2 (232 vs 238 us)
  return 1;
}

// Rows of each launch of a projection call with B rows: B itself up to 256, else the
// call is cut into equal launches of at most 256 rows.
int rows_per_launch(int B) {
  const int n = (B + MAX_B_WIDE - 1) / MAX_B_WIDE;
  return (B + n - 1) / n;
}

dec_status run_splitk_rows(const dec_bf16 *X, const dec_bf16 *W, const dec_bf16 *R, dec_bf16 *Y,
                           int B, int N, int K, int split_k, int use_tc, void *ws,
                           size_t ws_bytes, cudaStream_t s, bool packed = false);

// Wide projections from DEC_WIDE_PAIR_MIN_B rows (default 65) up to 512 on CTA-pair
// tensor-core tiles, one launch per call (DEC_WIDE_PAIR_MMA=0: launches of at most 256
// rows on one-CTA tiles, each reading W). Up to 128 rows only where the clusters (4 CTAs
// per 256 rows of W) cover at least DEC_PAIR_SPLIT_MIN_SM_PCT of the SMs: measured on one
// box (us, CTA pairs -> one-CTA tiles), the input projection (128 CTAs) 22.5 -> 24.6 at 65
// rows and 23.0 -> 25.0 at 128, the output projection (112 CTAs) 43.4 -> 41.8 at 65 rows
// and 43.6 -> 43.5 at 128; from 129 rows the pair tiles win on both.
bool wide_pair_mma() {
  if (const char *s = std::getenv("DEC_WIDE_PAIR_MMA")) return std::atoi(s) != 0;
  return true;
}
int wide_pair_min_batch() {
  if (const char *s = std::getenv("DEC_WIDE_PAIR_MIN_B")) {
    const int v = std::atoi(s);
    if (v >= MAX_B + 1) return v;
  }
  return MAX_B + 1;
}

// 4-CTA clusters of the pair kernel the device holds at once, per device and column count.
std::atomic<int> g_pair_clusters[kMaxDevices][7];
std::once_flag g_pair_init_once;

int pair_clusters(int ncol) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::call_once(g_pair_init_once, []() {
    for (auto &d : g_pair_clusters)
      for (auto &v : d) v.store(-1);
  });
  std::atomic<int> &slot = g_pair_clusters[dev][ncol / 64 - 2];  // ncol = 128, 192, .. 512
  int n = slot.load();
  if (n < 0) {
    if (engine_pair_max_clusters(ncol, &n) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    slot.store(n);
  }
  return n;
}

// Whether a call of B rows takes the CTA-pair kernel: every 256-row slice of W needs one
// resident cluster (a second wave would double the time).
bool use_pair_kernel(int B, int N, int K, int split_k, int use_tc, int num_sms) {
  if (!use_tc || split_k != 0 || !wide_pair_mma() || B < wide_pair_min_batch() || B > MAX_ROWS)
    return false;
  if (ceil_div(K, TILE_K) < 2) return false;
  const int slices = (ceil_div(N, TILE_N) + 1) / 2;
  if (B <= 2 * MAX_B && 400 * slices < pair_split_min_sm_pct() * num_sms) return false;
  return pair_clusters(pair_cols(B)) >= slices;
}

// The CTA-pair launch. The workspace is checked as for the one-CTA launches (the same
// size contract whichever kernel runs); the pair kernel itself uses none of it.
dec_status run_pair_projection(const dec_bf16 *X, const dec_bf16 *W, const dec_bf16 *R,
                               dec_bf16 *Y, int B, int N, int K, void *ws, size_t ws_bytes,
                               cudaStream_t s, bool packed) {
  cudaError_t ce;
  DeviceInfo *d = device_info(&ce);
  if (!d) return DEC_ERR_CUDA;
  SplitPlan pl;
  if (!plan_splitk(rows_per_launch(B), N, K, 0, d->num_sms, &pl))
    return DEC_ERR_UNSUPPORTED_SHAPE;
  if (!ws) return DEC_ERR_INVALID_ARG;
  if (!aligned16(ws)) return DEC_ERR_MISALIGNED;
  if (ws_bytes < pl.total) return DEC_ERR_WORKSPACE_TOO_SMALL;
  CUtensorMap wmap, xmap;
  const bool wmap_ok = packed ? make_map(&wmap, W, TILE_K, static_cast<uint64_t>(N) * pl.KB, 128)
                              : make_map(&wmap, W, K, N, 128);
  const int ncol = pair_cols(B);
  if (!wmap_ok || !make_map(&xmap, X, K, B, pair_xbox_rows(ncol))) return DEC_ERR_CUDA;
  EngineParams p;
  std::memset(&p, 0, sizeof p);
  p.mode = MODE_LINEAR;
  p.N = N;
  p.K = K;
  p.T = pl.T;
  p.KB = pl.KB;
  p.G = 4 * ((pl.T + 1) / 2);
  p.B = B;
  p.ngrp = 1;
  p.Y = Y;
  p.R = R;
  p.vec_y = (N % 8 == 0 && aligned16(Y) && (R == nullptr || aligned16(R))) ? 1 : 0;
  p.packed = packed ? 1 : 0;
  p.status = d->status;
  p.wait_limit_ns = g_wait_limit_ns.load();
  // Y (and R) as whole tiles by TMA when their rows are 16-byte aligned (p.vec_y)
  CUtensorMap ymap, rmap;
  std::memset(&ymap, 0, sizeof ymap);
  std::memset(&rmap, 0, sizeof rmap);
  if (p.vec_y) {
    if (!make_map_plain(&ymap, Y, N, B, 128, ncol / 2)) return DEC_ERR_CUDA;
    if (R && !make_map_plain(&rmap, R, N, B, 128, ncol / 2)) return DEC_ERR_CUDA;
  }
  if (consume_fault()) return DEC_ERR_CUDA;
  ce = launch_engine_pair(ncol, wmap, xmap, ymap, rmap, p, s);
  if (ce == cudaErrorNotSupported) return DEC_ERR_UNSUPPORTED_SHAPE;
  if (ce != cudaSuccess) return DEC_ERR_CUDA;
  t_last_variant = DEC_VARIANT_SPLITK_TC_PAIR;
  return DEC_OK;
}

// A projection of 65..512 rows (speculative verification of up to 64 sequences x 8
// tokens) is one CTA-pair launch where use_pair_kernel allows; otherwise more than 256
// rows run as consecutive launches over row blocks, each reading W; on one stream, each
// launch's workspace use begins after the previous launch has finished with it (the
// stream order, or the dependency wait of a programmatic launch).
dec_status run_splitk(const dec_bf16 *X, const dec_bf16 *W, const dec_bf16 *R, dec_bf16 *Y,
                      int B, int N, int K, int split_k, int use_tc, void *ws, size_t ws_bytes,
                      cudaStream_t s, bool packed = false) {
  cudaError_t ce;
  DeviceInfo *d = device_info(&ce);
  if (!d) return DEC_ERR_CUDA;
  if (use_pair_kernel(B, N, K, split_k, use_tc, d->num_sms))
    return run_pair_projection(X, W, R, Y, B, N, K, ws, ws_bytes, s, packed);
  if (B <= MAX_B_WIDE)
    return run_splitk_rows(X, W, R, Y, B, N, K, split_k, use_tc, ws, ws_bytes, s, packed);
  if (!use_tc) return DEC_ERR_UNSUPPORTED_SHAPE;
  const int rows = rows_per_launch(B);
  for (int r0 = 0; r0 < B; r0 += rows) {
    const int rb = B - r0 < rows ? B - r0 : rows;
    const size_t xo = static_cast<size_t>(r0) * K, yo = static_cast<size_t>(r0) * N;
    const dec_status st = run_splitk_rows(X + xo, W, R ? R + yo : nullptr, Y + yo, rb, N, K,
                                          split_k, use_tc, ws, ws_bytes, s, packed);
    if (st != DEC_OK) return st;
  }
  return DEC_OK;
}

dec_status run_splitk_rows(const dec_bf16 *X, const dec_bf16 *W, const dec_bf16 *R, dec_bf16 *Y,
                           int B, int N, int K, int split_k, int use_tc, void *ws,
                           size_t ws_bytes, cudaStream_t s, bool packed) {
  cudaError_t ce;
  DeviceInfo *d = device_info(&ce);
  if (!d) return DEC_ERR_CUDA;
  if (B > MAX_B && !use_tc) return DEC_ERR_UNSUPPORTED_SHAPE;  // wide: tensor cores only
  SplitPlan pl;
  if (!plan_splitk(B, N, K, split_k, d->num_sms, &pl)) return DEC_ERR_UNSUPPORTED_SHAPE;
  if (!ws) return DEC_ERR_INVALID_ARG;
  if (!aligned16(ws)) return DEC_ERR_MISALIGNED;
  if (ws_bytes < pl.total) return DEC_ERR_WORKSPACE_TOO_SMALL;
  CUtensorMap wmap, xmap;
  // a tile-packed W is mapped as N*KB rows of 64 k (128 bytes): one box = one 16 KB block
  const bool wmap_ok = packed ? make_map(&wmap, W, TILE_K, static_cast<uint64_t>(N) * pl.KB, 128)
                              : make_map(&wmap, W, K, N, 128);
  if (!wmap_ok || !make_map(&xmap, X, K, B, xbox_rows_for(pl, B))) return DEC_ERR_CUDA;
  EngineParams p;
  fill_engine_common(p, pl, MODE_LINEAR, N, K, B, ws, d);
  p.Y = Y;
  p.R = R;
  p.vec_y = (N % 8 == 0 && aligned16(Y) && (R == nullptr || aligned16(R))) ? 1 : 0;
  p.packed = packed ? 1 : 0;
  // the optional L2 prefetch of later k-blocks (row-major rows or packed blocks)
  p.w_base = reinterpret_cast<const uint8_t *>(W);
  p.w_rows = N;
  // Every tile split into exactly two k-halves (G = 2 T, KB even): on tensor cores the
  // two workers of a tile run as a 2-CTA cluster and add their halves through
  // distributed shared memory, with no partial tiles in global memory and no counter.
  const bool pair_ok = use_tc && pl.G == 2 * pl.T && pl.KB % 2 == 0 &&
                       (pl.ngrp > 1 ? pair_dsmem_max_cols() >= MAX_B
                                    : pl.maxc <= pair_dsmem_max_cols());
  // Otherwise, for large batches, the product kernel only stores partial tiles and a
  // finishing kernel over (tile, 16 columns) adds them, instead of each tile's last
  // worker adding 64-wide partials at the end of the product (the product's tail).
  // Needs workers that span at most two tiles.
  if (pair_ok)
    p.defer = 0;
  else if (pl.ngrp > 1)  // wide: four 64-column reductions per tile are too long a tail
    p.defer = (pl.G >= pl.T && wide_defer()) ? 1 : 0;
  else
    p.defer = (B >= defer_min_batch() && K >= defer_min_k() && pl.G >= pl.T) ? 1 : 0;
  p.pair = pair_ok ? 1 : 0;
  if (consume_fault()) return DEC_ERR_CUDA;
  ce = use_tc ? launch_engine_tc(pl.maxc, wmap, xmap, p, s)
              : launch_engine_cc(pl.maxc, wmap, xmap, p, s);
  if (ce == cudaErrorNotSupported) return DEC_ERR_UNSUPPORTED_SHAPE;
  if (ce != cudaSuccess) return DEC_ERR_CUDA;
  if (p.defer) {
    LinearFinishParams f;
    f.partials = p.partials;
    f.slot_cols = p.slot_cols;
    f.G = p.G;
    f.T = p.T;
    f.KB = p.KB;
    f.ngrp = p.ngrp;
    f.vec_y = p.vec_y;
    f.total = static_cast<long long>(p.T) * p.KB;
    f.B = B;
    f.N = N;
    f.R = R;
    f.Y = Y;
    if (launch_linear_finish(f, s) != cudaSuccess) return DEC_ERR_CUDA;
  }
  t_last_variant = use_tc ? DEC_VARIANT_SPLITK_TC : DEC_VARIANT_SPLITK;
  return DEC_OK;
}

// ------------------------------------------------------------- MoE planning --

struct FrontPlan {
  SplitPlan sk;
  size_t done_off, logits_off;  // done_off: the route-map counter of the two-launch path
  size_t fcnt_off;              // one-launch path: arrival counters
  size_t total;
};

// k-splits per front tile (0 = one worker per SM). Fewer splits mean fewer partial
// tiles for each tile's last worker to add, which dominates at large B.
int front_splits(int B, int E, int L, int num_sms) {
  int s = 0;
  if (const char *e = std::getenv("DEC_FRONT_SPLIT")) s = std::atoi(e);
  (void)B;
  if (s <= 0) return 0;
  const int T = ceil_div(E + L, TILE_N);
  if (s * T > num_sms) s = num_sms / T;
  return s < 1 ? 1 : s;
}

bool plan_front(int B, int E, int L, int K, int num_sms, FrontPlan *fp, int splits = 0) {
  if (!plan_splitk(B, E + L, K, splits, num_sms, &fp->sk)) return false;
  fp->done_off = fp->sk.total;
  fp->logits_off = fp->done_off + kAlign;
  fp->fcnt_off = fp->logits_off + align_up(static_cast<size_t>(B) * E * sizeof(float));
  fp->total = fp->fcnt_off + kAlign;
  return true;
}

// Whether moe_front with B tokens runs as one launch (front_fused.cu) where the device
// can schedule it (measured at least as fast as the product kernel + finishing kernel
// at every batch: 11.6 vs 12.8 us at B = 1, 16.4 vs 17.1 us at B = 64); up to
// DEC_FRONT_FUSED_MAX_B tokens (default 64); DEC_FRONT_FUSED=0/1 turns it off / on at
// every batch.
bool front_fused_enabled(int B) {
  if (const char *s = std::getenv("DEC_FRONT_FUSED")) return std::atoi(s) != 0;
  int max_b = MAX_B;
  if (const char *s = std::getenv("DEC_FRONT_FUSED_MAX_B")) max_b = std::atoi(s);
  return B <= max_b;
}

// Stage-ring depth of the one-launch front end (DEC_FRONT_STAGES; default 8, cut to what
// fits in shared memory). Even, because the two MMA-issuing warps each own every other
// stage. A ring at least as deep as a CTA's k-range (7 k-blocks at K = 7168) loads all
// its weights before the dependency wait: measured 0.3-1.2 us faster per call than 4
// stages, although the next call's CTAs can then no longer sit on the same SMs early.
int front_stages_override() {
  if (const char *s = std::getenv("DEC_FRONT_STAGES")) {
    const int v = std::atoi(s) & ~1;
    return v >= 2 && v <= 12 ? v : 0;
  }
  return 0;
}

// Largest batch whose tokens the one-launch front end routes in one CTA (a warp per
// token, one arrival counter; DEC_FRONT_SINGLE_B, default 8). Larger batches route each
// token group in its own CTA and elect the route-map builder with a second counter.
int front_single_batch() {
  if (const char *s = std::getenv("DEC_FRONT_SINGLE_B")) {
    const int v = std::atoi(s);
    if (v >= 0 && v <= MAX_B) return v;
  }
  return 8;
}

// Largest batch for which the one-launch front end's router CTAs hold back the trigger
// of the next kernel until their routing has read the logits (DEC_FRONT_LATE_TRIGGER_B).
// The next kernel's weight loads, issued before its dependency wait, otherwise flood L2
// while the routing CTA reads the freshly published logits (measured at B = 1: 2.0 us
// for those reads, 0.6 us without the burst). Default 8: a chain of front
// ends measured 8.3-8.6 us per call at B = 1-8 with it, 8.8-9.9 us without.
int front_late_trigger_batch() {
  if (const char *s = std::getenv("DEC_FRONT_LATE_TRIGGER_B")) {
    const int v = std::atoi(s);
    if (v >= 0 && v <= MAX_B) return v;
  }
  return 8;
}

struct FusedFrontPlan {
  int S, log2S, nxb, nst, nsl;
  size_t smem;
};

// The deepest even ring, at most `want` stages, that fits in shared memory.
int fit_stages(int S, int nxb, int nsl, int want) {
  int nst = want;
  while (nst > 2 && front_fused_smem(S, nxb, nst, nsl) > FRONT_FUSED_SMEM_MAX) nst -= 2;
  return nst;
}

// Clusters of S CTAs of the one-launch front end the device holds at once, per device,
// activation-box count and cluster size, queried once with the largest shared-memory
// footprint of that configuration (64 tokens, the ring cut to fit).
std::atomic<int> g_ff_clusters[kMaxDevices][3][5];
std::once_flag g_ff_init_once;

int fused_front_clusters(int S, int nxb, int want) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::call_once(g_ff_init_once, []() {
    for (auto &d : g_ff_clusters)
      for (auto &a : d)
        for (auto &v : a) v.store(-1);
  });
  const int xi = nxb == 1 ? 0 : (nxb == 2 ? 1 : 2);
  int si = 0;
  while ((1 << si) < S) ++si;
  std::atomic<int> &slot = g_ff_clusters[dev][xi][si];
  int n = slot.load();
  if (n < 0) {
    const int nsl_max = (MAX_B + S - 1) / S;
    const int nst = fit_stages(S, nxb, nsl_max, want);
    n = front_fused_max_clusters(S, nxb, front_fused_smem(S, nxb, nst, nsl_max));
    slot.store(n);
  }
  return n;
}

// Cluster size S: the largest power of two <= min(16, k-blocks) that the device can
// schedule; every CTA of a cluster then owns KB/S (+-1) k-blocks of its tile.
bool plan_front_fused(int B, int K, FusedFrontPlan *f) {
  const int KB = ceil_div(K, TILE_K);
  f->nxb = B <= 16 ? 1 : (B <= 32 ? 2 : 4);
  const int ovr = front_stages_override();
  const int want = ovr > 0 ? ovr : 8;
  int S = 16;
  while (S > KB) S >>= 1;
  for (; S >= 1; S >>= 1)
    if (fused_front_clusters(S, f->nxb, want) >= 1) break;
  if (S < 1) return false;
  f->S = S;
  f->log2S = 0;
  while ((1 << f->log2S) < S) ++f->log2S;
  // 16-CTA clusters send every slot of a destination with one vector store
  f->nsl = S == 16 ? f->nxb : (B + S - 1) / S;
  f->nst = fit_stages(S, f->nxb, f->nsl, want);
  f->smem = front_fused_smem(S, f->nxb, f->nst, f->nsl);
  return f->smem <= FRONT_FUSED_SMEM_MAX;
}

struct ExpertsPlan {
  int maxc, Tg, Td, KBg, KBd;
  size_t rm_off, xg_off, a_off, yp_off, as_off, s_off;
  size_t main_part_off, main_cnt_off, side_part_off, side_cnt_off, cmb_off, dyn_off, total;
};

bool plan_experts(int B, int E, int topk, int H, int I, int num_sms, ExpertsPlan *ep) {
  const size_t P = static_cast<size_t>(B) * topk;
  ep->maxc = engine_maxc_for(B);
  ep->Tg = I / 64;
  ep->Td = H / TILE_N;
  ep->KBg = ceil_div(H, TILE_K);
  ep->KBd = ceil_div(I, TILE_K);
  size_t o = 0;
  ep->rm_off = o;
  o += align_up(moe_route_map_ints(B, E, topk) * sizeof(int32_t));
  // P gathered rows, then B more for the shared expert when it runs in the routed launch
  const size_t PB = P + static_cast<size_t>(B);
  ep->xg_off = o;
  o += align_up(PB * H * 2);
  ep->a_off = o;
  o += align_up(PB * I * 2);
  ep->yp_off = o;
  o += align_up(PB * H * sizeof(float));
  ep->as_off = o;
  o += align_up(static_cast<size_t>(B) * I * 2);
  ep->s_off = o;
  o += align_up(static_cast<size_t>(B) * H * sizeof(float));
  const size_t part = align_up(static_cast<size_t>(2) * num_sms * 128 * ep->maxc * sizeof(float));
  const int tmax = ep->Tg > ep->Td ? ep->Tg : ep->Td;
  ep->main_part_off = o;
  o += part;
  ep->main_cnt_off = o;
  o += align_up(static_cast<size_t>(E) * tmax * sizeof(int));
  ep->side_part_off = o;
  o += part;
  ep->side_cnt_off = o;
  o += align_up(static_cast<size_t>(tmax) * sizeof(int));
  ep->cmb_off = o;  // fused combine: one arrival counter per (token, 128-row block of H)
  o += align_up(static_cast<size_t>(B) * ep->Td * sizeof(int));
  ep->dyn_off = o;  // routed launches: counters [4], then a ready count per group (E + 1)
  o += align_up((5 + static_cast<size_t>(E)) * sizeof(int));
  ep->total = o;
  return true;
}

// Two events per (host thread, device) for the main/side fork and join.
struct StreamEvents {
  cudaEvent_t fork = nullptr, join = nullptr;
};
thread_local StreamEvents t_events[kMaxDevices];

dec_status get_events(StreamEvents **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DEC_ERR_CUDA;
  StreamEvents &ev = t_events[dev];
  if (!ev.fork) {
    if (cudaEventCreateWithFlags(&ev.fork, cudaEventDisableTiming) != cudaSuccess)
      return DEC_ERR_CUDA;
    if (cudaEventCreateWithFlags(&ev.join, cudaEventDisableTiming) != cudaSuccess)
      return DEC_ERR_CUDA;
  }
  *out = &ev;
  return DEC_OK;
}

dec_status run_front(const dec_bf16 *X, const dec_bf16 *Wcat, int B, int K, int E, int L,
                     int topk, dec_bf16 *latent, int32_t *topk_idx, float *topk_w,
                     float *probs_opt, int32_t *route_map_opt, void *ws, size_t ws_bytes,
                     int sms, cudaStream_t s);

}  // namespace

// =================================================================== C ABI ====

extern "C" {

const char *dec_status_string(int status) {
  switch (status) {
    case DEC_OK: return "ok";
    case DEC_ERR_INVALID_ARG: return "invalid argument";
    case DEC_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (use the standard path)";
    case DEC_ERR_MISALIGNED: return "misaligned pointer or length";
    case DEC_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case DEC_ERR_CUDA: return "CUDA error";
    case DEC_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

const char *dec_variant_name(int variant) {
  switch (variant) {
    case DEC_VARIANT_TINY: return "tiny";
    case DEC_VARIANT_SPLITK: return "splitk";
    case DEC_VARIANT_SPLITK_TC: return "splitk_tc";
    case DEC_VARIANT_FRONT_ONE_LAUNCH: return "front_one_launch";
    case DEC_VARIANT_SPLITK_TC_PAIR: return "splitk_tc_pair";
    default: return "none";
  }
}

int dec_last_variant(void) { return t_last_variant; }

int dec_version(void) { return 100; }

dec_status dec_set_force_variant(int variant) {
  if (variant < DEC_VARIANT_NONE || variant > DEC_VARIANT_SPLITK_TC) return DEC_ERR_INVALID_ARG;
  g_force_variant.store(variant);
  return DEC_OK;
}

dec_status dec_set_fault_inject(int count) {
  if (count < 0) return DEC_ERR_INVALID_ARG;
  g_fault_inject.store(count);
  return DEC_OK;
}

dec_status dec_set_wait_limit_ns(uint64_t ns) {
  if (ns < 1000000ull) return DEC_ERR_INVALID_ARG;
  g_wait_limit_ns.store(ns);
  return DEC_OK;
}

dec_status dec_sync_status(dec_stream_t s) {
  cudaError_t ce;
  DeviceInfo *d = device_info(&ce);
  if (!d) return DEC_ERR_CUDA;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(s)) != cudaSuccess) return DEC_ERR_CUDA;
  unsigned word = 0, zero = 0;
  if (cudaMemcpy(&word, d->status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return DEC_ERR_CUDA;
  if (word != 0 && cudaMemcpy(d->status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
    return DEC_ERR_CUDA;
  if (word & ST_TIMEOUT) return DEC_ERR_TIMEOUT;
  if (word & ST_BAD_ROUTING) return DEC_ERR_INVALID_ARG;
  return DEC_OK;
}

dec_status dec_debug_wait_timeout(uint64_t limit_ns, dec_stream_t s) {
  if (limit_ns < 1000000ull || limit_ns > 10000000000ull) return DEC_ERR_INVALID_ARG;
  cudaError_t ce;
  DeviceInfo *d = device_info(&ce);
  if (!d) return DEC_ERR_CUDA;
  return cuda_status(launch_wait_selftest(d->status, limit_ns, reinterpret_cast<cudaStream_t>(s)));
}

// ------------------------------------------------------------- projection ----

}  // extern "C"

namespace {

// Below this K the batch switch keeps the tiny kernel for packed weights (see linear_impl).
constexpr int kPackedTinyMaxK = 12288;

// A tile-packed weight needs whole 128-row tiles and 64-wide k-blocks.
dec_status check_packed_shape(int N, int K) {
  return (N % TILE_N == 0 && K % TILE_K == 0) ? DEC_OK : DEC_ERR_UNSUPPORTED_SHAPE;
}

dec_status gemv_impl(const dec_bf16 *X, const dec_bf16 *W, const dec_bf16 *R, dec_bf16 *Y, int B,
                     int N, int K, dec_stream_t s, bool packed) {
  dec_status st = check_linear_args(X, W, Y, B, N, K);
  if (st == DEC_OK && packed) st = check_packed_shape(N, K);
  if (st != DEC_OK) return st;
  if (B > TINY_MAX_NB) return DEC_ERR_UNSUPPORTED_SHAPE;
  cudaError_t ce;
  DeviceInfo *d = device_info(&ce);
  if (!d) return DEC_ERR_CUDA;
  if (consume_fault()) return DEC_ERR_CUDA;
  ce = launch_gemv_tiny(X, W, R, Y, B, N, K, d->num_sms, reinterpret_cast<cudaStream_t>(s),
                        packed);
  if (ce != cudaSuccess) return DEC_ERR_CUDA;
  t_last_variant = DEC_VARIANT_TINY;
  return DEC_OK;
}

dec_status splitk_impl(const dec_bf16 *X, const dec_bf16 *W, const dec_bf16 *R, dec_bf16 *Y,
                       int B, int N, int K, int split_k, int use_tc, void *ws, size_t ws_bytes,
                       dec_stream_t s, bool packed) {
  dec_status st = check_linear_args(X, W, Y, B, N, K);
  if (st == DEC_OK && packed) st = check_packed_shape(N, K);
  if (st != DEC_OK) return st;
  if (split_k < 0 || (use_tc != 0 && use_tc != 1)) return DEC_ERR_INVALID_ARG;
  return run_splitk(X, W, R, Y, B, N, K, split_k, use_tc, ws, ws_bytes,
                    reinterpret_cast<cudaStream_t>(s), packed);
}

dec_status linear_impl(const dec_bf16 *X, const dec_bf16 *W, const dec_bf16 *R, dec_bf16 *Y,
                       int B, int N, int K, void *ws, size_t ws_bytes, dec_stream_t s,
                       bool packed) {
  dec_status st = check_linear_args(X, W, Y, B, N, K);
  if (st == DEC_OK && packed) st = check_packed_shape(N, K);
  if (st != DEC_OK) return st;
  int v = force_variant();
  if (v == DEC_VARIANT_NONE) {
    cudaError_t ce;
    const DeviceInfo *d = device_info(&ce);
    if (!d) return DEC_ERR_CUDA;
    // On packed weights the tiny kernel's reads are strided by the 16 KB blocks; from
    // K = 12288 the split-K tiles, which stream whole blocks, are faster already at B = 1
    // (the 16384 -> 7168 projection: 37.9 / 38.3 us at B = 1 / 2 against 38.9 / 45.9).
    if (B <= tiny_max_batch(N, K, d->num_sms) && !(packed && K >= kPackedTinyMaxK))
      v = DEC_VARIANT_TINY;
    else if (B <= 2 || B >= tc_min_batch() || B > MAX_B)  // B <= 2 here: a pair shape
      v = DEC_VARIANT_SPLITK_TC;
    else
      v = DEC_VARIANT_SPLITK;
  }
  if (v == DEC_VARIANT_TINY) return gemv_impl(X, W, R, Y, B, N, K, s, packed);
  return run_splitk(X, W, R, Y, B, N, K, 0, v == DEC_VARIANT_SPLITK_TC ? 1 : 0, ws, ws_bytes,
                    reinterpret_cast<cudaStream_t>(s), packed);
}

}  // namespace

extern "C" {

dec_status dec_gemv(const dec_bf16 *X, const dec_bf16 *W, const dec_bf16 *R, dec_bf16 *Y, int B,
                    int N, int K, dec_stream_t s) {
  return gemv_impl(X, W, R, Y, B, N, K, s, false);
}

dec_status dec_gemv_packed(const dec_bf16 *X, const dec_bf16 *Wp, const dec_bf16 *R, dec_bf16 *Y,
                           int B, int N, int K, dec_stream_t s) {
  return gemv_impl(X, Wp, R, Y, B, N, K, s, true);
}

size_t dec_splitk_workspace_bytes(int B, int N, int K, int split_k) {
  if (B < 1 || B > MAX_ROWS || N < 1 || K < 1 || split_k < 0) return 0;
  B = rows_per_launch(B);  // every launch of the call reuses the workspace
  SplitPlan pl;
  const int sms = current_num_sms();
  if (sms <= 0 || !plan_splitk(B, N, K, split_k, sms, &pl)) return 0;
  return pl.total;
}

dec_status dec_splitk_gemm(const dec_bf16 *X, const dec_bf16 *W, const dec_bf16 *R, dec_bf16 *Y,
                           int B, int N, int K, int split_k, int use_tc, void *ws,
                           size_t ws_bytes, dec_stream_t s) {
  return splitk_impl(X, W, R, Y, B, N, K, split_k, use_tc, ws, ws_bytes, s, false);
}

dec_status dec_splitk_gemm_packed(const dec_bf16 *X, const dec_bf16 *Wp, const dec_bf16 *R,
                                  dec_bf16 *Y, int B, int N, int K, int split_k, int use_tc,
                                  void *ws, size_t ws_bytes, dec_stream_t s) {
  return splitk_impl(X, Wp, R, Y, B, N, K, split_k, use_tc, ws, ws_bytes, s, true);
}

size_t dec_linear_workspace_bytes(int B, int N, int K) {
  return dec_splitk_workspace_bytes(B, N, K, 0);
}

dec_status dec_linear(const dec_bf16 *X, const dec_bf16 *W, const dec_bf16 *R, dec_bf16 *Y, int B,
                      int N, int K, void *ws, size_t ws_bytes, dec_stream_t s) {
  return linear_impl(X, W, R, Y, B, N, K, ws, ws_bytes, s, false);
}

dec_status dec_linear_packed(const dec_bf16 *X, const dec_bf16 *Wp, const dec_bf16 *R, dec_bf16 *Y,
                             int B, int N, int K, void *ws, size_t ws_bytes, dec_stream_t s) {
  return linear_impl(X, Wp, R, Y, B, N, K, ws, ws_bytes, s, true);
}

dec_status dec_pack_weight(const dec_bf16 *W, int N, int K, dec_bf16 *Wp, dec_stream_t s) {
  if (!W || !Wp || N < 1 || K < 1) return DEC_ERR_INVALID_ARG;
  if (check_packed_shape(N, K) != DEC_OK) return DEC_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(W) || !aligned16(Wp)) return DEC_ERR_MISALIGNED;
  if (static_cast<int64_t>(N) * K > (int64_t(1) << 40)) return DEC_ERR_UNSUPPORTED_SHAPE;
  const uint16_t *wb = W, *end = W + static_cast<size_t>(N) * K;  // no overlap allowed
  if (Wp < end && wb < Wp + static_cast<size_t>(N) * K) return DEC_ERR_INVALID_ARG;
  cudaError_t ce;
  if (!device_info(&ce)) return DEC_ERR_CUDA;
  return cuda_status(launch_pack_weight(W, N, K, Wp, reinterpret_cast<cudaStream_t>(s)));
}

// ------------------------------------------------------------------- MoE ----

size_t moe_route_map_ints(int B, int E, int topk) {
  if (B < 1 || E < 1 || topk < 1) return 0;
  return static_cast<size_t>(3) * E + 2 + static_cast<size_t>(2) * B * topk;
}

size_t moe_front_workspace_bytes(int B, int E, int L, int K) {
  if (B < 1 || B > MAX_B || E < 1 || E > MAX_E || L < 0 || K < 1) return 0;
  const int sms = current_num_sms();
  FrontPlan fp;
  if (sms <= 0 || !plan_front(B, E, L, K, sms, &fp)) return 0;
  return fp.total;
}

dec_status moe_front(const dec_bf16 *X, const dec_bf16 *Wcat, int B, int K, int E, int L,
                     int topk, dec_bf16 *latent, int32_t *topk_idx, float *topk_w,
                     float *probs_opt, int32_t *route_map_opt, void *ws, size_t ws_bytes,
                     dec_stream_t s) {
  if (!X || !Wcat || !topk_idx || !topk_w || !ws) return DEC_ERR_INVALID_ARG;
  if (L > 0 && !latent) return DEC_ERR_INVALID_ARG;
  if (B < 1 || K < 1 || E < 1 || L < 0 || topk < 1) return DEC_ERR_INVALID_ARG;
  if (B > MAX_B || E > MAX_E || topk > MAX_TOPK || topk > E) return DEC_ERR_UNSUPPORTED_SHAPE;
  if (K % 8 != 0 || !aligned16(X) || !aligned16(Wcat) || !aligned16(ws)) return DEC_ERR_MISALIGNED;
  cudaError_t ce;
  DeviceInfo *d = device_info(&ce);
  if (!d) return DEC_ERR_CUDA;
  return run_front(X, Wcat, B, K, E, L, topk, latent, topk_idx, topk_w, probs_opt, route_map_opt,
                   ws, ws_bytes, d->num_sms, reinterpret_cast<cudaStream_t>(s));
}

}  // extern "C"

namespace {

// The front end (product + finishing kernel) on at most `sms` workers, arguments
// already checked.
dec_status run_front(const dec_bf16 *X, const dec_bf16 *Wcat, int B, int K, int E, int L,
                     int topk, dec_bf16 *latent, int32_t *topk_idx, float *topk_w,
                     float *probs_opt, int32_t *route_map_opt, void *ws, size_t ws_bytes,
                     int sms, cudaStream_t s) {
  cudaError_t ce;
  DeviceInfo *d = device_info(&ce);
  if (!d) return DEC_ERR_CUDA;
  FrontPlan fp;
  int splits = front_splits(B, E, L, sms);
  if (splits > ceil_div(K, TILE_K)) splits = ceil_div(K, TILE_K);
  if (!plan_front(B, E, L, K, sms, &fp, splits)) return DEC_ERR_UNSUPPORTED_SHAPE;
  if (ws_bytes < fp.total) return DEC_ERR_WORKSPACE_TOO_SMALL;
  CUtensorMap wmap, xmap;
  if (!make_map(&wmap, Wcat, K, E + L, 128) ||
      !make_map(&xmap, X, K, B, xbox_rows_for(fp.sk.maxc)))
    return DEC_ERR_CUDA;
  char *wsb = static_cast<char *>(ws);
  const int fv = force_variant();
  FusedFrontPlan ffp;
  if (front_fused_enabled(B) && fv != DEC_VARIANT_SPLITK && plan_front_fused(B, K, &ffp)) {
    CUtensorMap xmap1;
    if (!make_map(&xmap1, X, K, B, 16 * ffp.nxb)) return DEC_ERR_CUDA;
    FrontFusedParams f;
    std::memset(&f, 0, sizeof f);
    f.B = B;
    f.E = E;
    f.L = L;
    f.KB = ceil_div(K, TILE_K);
    f.T = ceil_div(E + L, TILE_N);
    f.S = ffp.S;
    f.log2S = ffp.log2S;
    f.TR = ceil_div(E, TILE_N);
    f.topk = topk;
    f.nst = ffp.nst;
    f.nsl = ffp.nsl;
    f.single_b = front_single_batch();
    f.trig_late = B <= front_late_trigger_batch() ? 1 : 0;
    f.latent = latent;
    f.topk_idx = topk_idx;
    f.topk_w = topk_w;
    f.probs = probs_opt;
    f.logits = reinterpret_cast<float *>(wsb + fp.logits_off);
    f.route_map = route_map_opt;
    f.counter = reinterpret_cast<int *>(wsb + fp.fcnt_off);
    f.status = d->status;
    f.wait_limit_ns = g_wait_limit_ns.load();
    if (consume_fault()) return DEC_ERR_CUDA;
    ce = launch_front_fused(wmap, xmap1, f, ffp.nxb, ffp.smem, s);
    if (ce != cudaSuccess) return DEC_ERR_CUDA;
    t_last_variant = DEC_VARIANT_FRONT_ONE_LAUNCH;
    return DEC_OK;
  }
  EngineParams p;
  fill_engine_common(p, fp.sk, MODE_FRONT, E + L, K, B, ws, d);
  if (fp.sk.G < fp.sk.T) return DEC_ERR_UNSUPPORTED_SHAPE;  // a worker may span 2 tiles at most
  p.w_base = reinterpret_cast<const uint8_t *>(Wcat);
  p.w_rows = E + L;
  p.defer = 1;  // partial tiles only; front_finish adds them
  if (consume_fault()) return DEC_ERR_CUDA;
  const bool tc = (fv == DEC_VARIANT_SPLITK_TC) || (fv == DEC_VARIANT_NONE && B >= tc_min_batch());
  ce = tc ? launch_engine_tc(fp.sk.maxc, wmap, xmap, p, s)
          : launch_engine_cc(fp.sk.maxc, wmap, xmap, p, s);
  if (ce == cudaErrorNotSupported) return DEC_ERR_UNSUPPORTED_SHAPE;
  if (ce != cudaSuccess) return DEC_ERR_CUDA;
  FrontFinishParams f;
  f.partials = p.partials;
  f.slot_cols = p.slot_cols;
  f.G = p.G;
  f.T = p.T;
  f.KB = p.KB;
  f.total = static_cast<long long>(p.T) * p.KB;
  f.B = B;
  f.E = E;
  f.L = L;
  f.topk = topk;
  f.logits = reinterpret_cast<float *>(wsb + fp.logits_off);
  f.latent = latent;
  f.topk_idx = topk_idx;
  f.topk_w = topk_w;
  f.probs = probs_opt;
  f.route_map = route_map_opt;
  f.all_done = reinterpret_cast<int *>(wsb + fp.done_off);
  f.cluster = (route_map_opt != nullptr && B <= 8 && front_cluster()) ? 1 : 0;
  ce = launch_front_finish(f, s);
  if (ce != cudaSuccess) return DEC_ERR_CUDA;
  t_last_variant = tc ? DEC_VARIANT_SPLITK_TC : DEC_VARIANT_SPLITK;
  return DEC_OK;
}

// A front end launched by moe_layer between the shared expert's and the routed
// experts' launches.
struct FrontCall {
  const dec_bf16 *Wcat;
  int L;
  dec_bf16 *latent;
  void *ws;
  size_t ws_bytes;
};

dec_status moe_experts_impl(const dec_bf16 *X, const int32_t *topk_idx, const float *topk_w,
                            const int32_t *route_map, const dec_bf16 *Wgu, const dec_bf16 *Wd,
                            int E, const dec_bf16 *Wgu_shared, const dec_bf16 *Wd_shared, int B,
                            int H, int I, int topk, dec_bf16 *Y, void *ws, size_t ws_bytes,
                            dec_stream_t main_stream, dec_stream_t side_stream,
                            int side_max_ctas, const FrontCall *fc, bool packed);

}  // namespace

extern "C" {

size_t moe_experts_workspace_bytes(int B, int E, int topk, int H, int I) {
  if (B < 1 || B > MAX_B || E < 1 || E > MAX_E || topk < 1 || topk > MAX_TOPK || H < 1 || I < 1)
    return 0;
  const int sms = current_num_sms();
  ExpertsPlan ep;
  if (sms <= 0 || !plan_experts(B, E, topk, H, I, sms, &ep)) return 0;
  return ep.total;
}

dec_status moe_experts(const dec_bf16 *X, const int32_t *topk_idx, const float *topk_w,
                       const int32_t *route_map, const dec_bf16 *Wgu, const dec_bf16 *Wd, int E,
                       const dec_bf16 *Wgu_shared, const dec_bf16 *Wd_shared, int B, int H,
                       int I, int topk, dec_bf16 *Y, void *ws, size_t ws_bytes,
                       dec_stream_t main_stream, dec_stream_t side_stream, int side_max_ctas) {
  return moe_experts_impl(X, topk_idx, topk_w, route_map, Wgu, Wd, E, Wgu_shared, Wd_shared, B,
                          H, I, topk, Y, ws, ws_bytes, main_stream, side_stream, side_max_ctas,
                          nullptr, false);
}

dec_status moe_experts_packed(const dec_bf16 *X, const int32_t *topk_idx, const float *topk_w,
                              const int32_t *route_map, const dec_bf16 *Wgu_p,
                              const dec_bf16 *Wd_p, int E, const dec_bf16 *Wgu_shared_p,
                              const dec_bf16 *Wd_shared_p, int B, int H, int I, int topk,
                              dec_bf16 *Y, void *ws, size_t ws_bytes, dec_stream_t main_stream,
                              dec_stream_t side_stream, int side_max_ctas) {
  return moe_experts_impl(X, topk_idx, topk_w, route_map, Wgu_p, Wd_p, E, Wgu_shared_p,
                          Wd_shared_p, B, H, I, topk, Y, ws, ws_bytes, main_stream, side_stream,
                          side_max_ctas, nullptr, true);
}

dec_status dec_pack_expert_weights(const dec_bf16 *Wgu, const dec_bf16 *Wd, int E, int H, int I,
                                   dec_bf16 *Wgu_p, dec_bf16 *Wd_p, dec_stream_t s) {
  if (!Wgu || !Wd || !Wgu_p || !Wd_p || E < 1 || H < 1 || I < 1) return DEC_ERR_INVALID_ARG;
  if (H % TILE_N != 0 || I % TILE_K != 0 || H % TILE_K != 0) return DEC_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(Wgu) || !aligned16(Wd) || !aligned16(Wgu_p) || !aligned16(Wd_p))
    return DEC_ERR_MISALIGNED;
  const size_t n = static_cast<size_t>(E) * H * I;  // elements of Wd; Wgu has 2n
  if (n > (size_t(1) << 40)) return DEC_ERR_UNSUPPORTED_SHAPE;
  auto overlap = [](const dec_bf16 *a, size_t na, const dec_bf16 *b, size_t nb) {
    return a < b + nb && b < a + na;
  };
  // no destination may overlap a source or the other destination
  if (overlap(Wgu, 2 * n, Wgu_p, 2 * n) || overlap(Wd, n, Wd_p, n) ||
      overlap(Wgu_p, 2 * n, Wd_p, n) || overlap(Wgu, 2 * n, Wd_p, n) ||
      overlap(Wd, n, Wgu_p, 2 * n))
    return DEC_ERR_INVALID_ARG;
  cudaError_t ce;
  if (!device_info(&ce)) return DEC_ERR_CUDA;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
  ce = launch_pack_weight(Wgu, E * 2 * I, H, Wgu_p, cs, I);
  if (ce == cudaSuccess) ce = launch_pack_weight(Wd, E * H, I, Wd_p, cs);
  return cuda_status(ce);
}

size_t moe_layer_workspace_bytes(int B, int E, int L, int H, int I, int topk) {
  const size_t e = moe_experts_workspace_bytes(B, E, topk, H, I);
  const size_t f = moe_front_workspace_bytes(B, E, L, H);
  return (e == 0 || f == 0) ? 0 : align_up(e) + f;
}

}  // extern "C"

namespace {

dec_status moe_layer_impl(const dec_bf16 *X, const dec_bf16 *Wcat, int E, int L, int topk,
                          const dec_bf16 *Wgu, const dec_bf16 *Wd, const dec_bf16 *Wgu_shared,
                          const dec_bf16 *Wd_shared, int B, int H, int I, dec_bf16 *latent,
                          int32_t *topk_idx, float *topk_w, int32_t *route_map_opt, dec_bf16 *Y,
                          void *ws, size_t ws_bytes, dec_stream_t main_stream,
                          dec_stream_t side_stream, int side_max_ctas, bool packed) {
  if (!X || !Wcat || !ws) return DEC_ERR_INVALID_ARG;
  if (L < 0 || (L > 0 && !latent)) return DEC_ERR_INVALID_ARG;
  if (!aligned16(Wcat)) return DEC_ERR_MISALIGNED;
  const size_t e = moe_experts_workspace_bytes(B, E, topk, H, I);
  const size_t f = moe_front_workspace_bytes(B, E, L, H);
  if (e == 0 || f == 0) {
    if (B < 1 || E < 1 || topk < 1 || H < 1 || I < 1) return DEC_ERR_INVALID_ARG;
    return DEC_ERR_UNSUPPORTED_SHAPE;
  }
  if (ws_bytes < align_up(e) + f) return DEC_ERR_WORKSPACE_TOO_SMALL;
  if (H % 8 != 0) return DEC_ERR_MISALIGNED;
  FrontCall fc;
  fc.Wcat = Wcat;
  fc.L = L;
  fc.latent = latent;
  fc.ws = static_cast<char *>(ws) + align_up(e);
  fc.ws_bytes = f;
  return moe_experts_impl(X, topk_idx, topk_w, route_map_opt, Wgu, Wd, E, Wgu_shared, Wd_shared,
                          B, H, I, topk, Y, ws, align_up(e), main_stream, side_stream,
                          side_max_ctas, &fc, packed);
}

}  // namespace

extern "C" {

dec_status moe_layer(const dec_bf16 *X, const dec_bf16 *Wcat, int E, int L, int topk,
                     const dec_bf16 *Wgu, const dec_bf16 *Wd, const dec_bf16 *Wgu_shared,
                     const dec_bf16 *Wd_shared, int B, int H, int I, dec_bf16 *latent,
                     int32_t *topk_idx, float *topk_w, int32_t *route_map_opt, dec_bf16 *Y,
                     void *ws, size_t ws_bytes, dec_stream_t main_stream,
                     dec_stream_t side_stream, int side_max_ctas) {
  return moe_layer_impl(X, Wcat, E, L, topk, Wgu, Wd, Wgu_shared, Wd_shared, B, H, I, latent,
                        topk_idx, topk_w, route_map_opt, Y, ws, ws_bytes, main_stream,
                        side_stream, side_max_ctas, false);
}

dec_status moe_layer_packed(const dec_bf16 *X, const dec_bf16 *Wcat, int E, int L, int topk,
                            const dec_bf16 *Wgu_p, const dec_bf16 *Wd_p,
                            const dec_bf16 *Wgu_shared_p, const dec_bf16 *Wd_shared_p, int B,
                            int H, int I, dec_bf16 *latent, int32_t *topk_idx, float *topk_w,
                            int32_t *route_map_opt, dec_bf16 *Y, void *ws, size_t ws_bytes,
                            dec_stream_t main_stream, dec_stream_t side_stream,
                            int side_max_ctas) {
  return moe_layer_impl(X, Wcat, E, L, topk, Wgu_p, Wd_p, Wgu_shared_p, Wd_shared_p, B, H, I,
                        latent, topk_idx, topk_w, route_map_opt, Y, ws, ws_bytes, main_stream,
                        side_stream, side_max_ctas, true);
}

}  // extern "C"

namespace {

dec_status moe_experts_impl(const dec_bf16 *X, const int32_t *topk_idx, const float *topk_w,
                            const int32_t *route_map, const dec_bf16 *Wgu, const dec_bf16 *Wd,
                            int E, const dec_bf16 *Wgu_shared, const dec_bf16 *Wd_shared, int B,
                            int H, int I, int topk, dec_bf16 *Y, void *ws, size_t ws_bytes,
                            dec_stream_t main_stream, dec_stream_t side_stream,
                            int side_max_ctas, const FrontCall *fc, bool packed) {
  if (!X || !topk_idx || !topk_w || !Wgu || !Wd || !Y || !ws) return DEC_ERR_INVALID_ARG;
  if ((Wgu_shared == nullptr) != (Wd_shared == nullptr)) return DEC_ERR_INVALID_ARG;
  if (B < 1 || E < 1 || H < 1 || I < 1 || topk < 1 || side_max_ctas < 0)
    return DEC_ERR_INVALID_ARG;
  if (B > MAX_B || E > MAX_E || topk > MAX_TOPK || topk > E) return DEC_ERR_UNSUPPORTED_SHAPE;
  if (H % TILE_N != 0 || I % 64 != 0) return DEC_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(X) || !aligned16(Wgu) || !aligned16(Wd) || !aligned16(ws) ||
      (Wgu_shared && (!aligned16(Wgu_shared) || !aligned16(Wd_shared))) || !aligned16(Y) ||
      (reinterpret_cast<uintptr_t>(topk_w) & 3u) || (reinterpret_cast<uintptr_t>(topk_idx) & 3u))
    return DEC_ERR_MISALIGNED;
  cudaError_t ce;
  DeviceInfo *d = device_info(&ce);
  if (!d) return DEC_ERR_CUDA;
  ExpertsPlan ep;
  if (!plan_experts(B, E, topk, H, I, d->num_sms, &ep)) return DEC_ERR_UNSUPPORTED_SHAPE;
  if (ws_bytes < ep.total) return DEC_ERR_WORKSPACE_TOO_SMALL;
  StreamEvents *ev = nullptr;
  dec_status st = get_events(&ev);
  if (st != DEC_OK) return st;

  cudaStream_t ms = reinterpret_cast<cudaStream_t>(main_stream);
  cudaStream_t ss = reinterpret_cast<cudaStream_t>(side_stream);
  const bool shared = (Wgu_shared != nullptr);
  // The fused combine counts every (token, block)'s contributions, so it needs a routing
  // that is valid by construction: a route map from the caller (moe_front) or moe_layer.
  const bool fused = (route_map != nullptr || fc != nullptr) && fused_combine();
  // tensor-core tiles for the expert GEMVs from the same batch threshold as dec_linear
  const int fv = force_variant();
  const bool tc = (fv == DEC_VARIANT_SPLITK_TC) || (fv == DEC_VARIANT_NONE && B >= tc_min_batch());
  // the shared expert as one more group of the one-launch routed experts (every SM claims
  // its tiles too), unless the caller capped its CTAs or the combine is fused
  const bool merged = shared && tc && expert_one_launch() && shared_in_routed() && !fused &&
                      side_max_ctas == 0;
  const bool overlap = shared && !merged && (ss != ms);
  const int P = B * topk;
  char *wsb = static_cast<char *>(ws);
  int32_t *rm = route_map ? const_cast<int32_t *>(route_map)
                          : reinterpret_cast<int32_t *>(wsb + ep.rm_off);
  uint16_t *Xg = reinterpret_cast<uint16_t *>(wsb + ep.xg_off);
  uint16_t *A = reinterpret_cast<uint16_t *>(wsb + ep.a_off);
  float *Yp = reinterpret_cast<float *>(wsb + ep.yp_off);
  uint16_t *As = reinterpret_cast<uint16_t *>(wsb + ep.as_off);
  float *S = reinterpret_cast<float *>(wsb + ep.s_off);

  // CTA split between the routed experts (main) and the shared expert (side): in
  // proportion to the weight bytes each reads, using the expected number of distinct
  // experts for this batch, unless the caller caps the side.
  double miss = 1.0;
  for (int b = 0; b < B; ++b) miss *= 1.0 - static_cast<double>(topk) / E;
  const double u_exp = E * (1.0 - miss);  // expected distinct experts of the batch
  int g_side = 0;
  if (overlap) {
    if (side_max_ctas > 0) {
      g_side = side_max_ctas;
    } else {
      // a fair bandwidth share is num_sms/(U+1) SMs; round up with some slack so the
      // shared expert (88 MB at the Kimi shape) never becomes the critical path
      g_side = static_cast<int>(std::ceil(side_slack() * d->num_sms / (1.0 + u_exp)));
      if (g_side < 2) g_side = 2;
    }
    if (g_side < 1) g_side = 1;
    if (g_side > d->num_sms / 2) g_side = d->num_sms / 2;
  }
  const int g_main = d->num_sms - g_side;

  CUtensorMap m_wgu, m_wd, m_xg, m_a;
  // grouped launches keep 16-row activation boxes: most experts have few tokens
  // tile-packed banks are mapped as rows of 64 k (128 bytes): one box = one 16 KB block
  const uint64_t gu_rows = static_cast<uint64_t>(E) * 2 * I, d_rows = static_cast<uint64_t>(E) * H;
  if (!(packed ? make_map(&m_wgu, Wgu, TILE_K, gu_rows * (H / TILE_K), 128)
               : make_map(&m_wgu, Wgu, H, gu_rows, 64)) ||
      !(packed ? make_map(&m_wd, Wd, TILE_K, d_rows * (I / TILE_K), 128)
               : make_map(&m_wd, Wd, I, d_rows, 128)) ||
      !make_map(&m_xg, Xg, H, P + (merged ? B : 0), XBOX_ROWS) ||
      !make_map(&m_a, A, I, P + (merged ? B : 0), XBOX_ROWS))
    return DEC_ERR_CUDA;
  CUtensorMap m_wgus, m_wds, m_x, m_as;
  const int xb_shared = xbox_rows_for(ep.maxc);
  if (shared && (!(packed ? make_map(&m_wgus, Wgu_shared, TILE_K,
                                    static_cast<uint64_t>(2) * I * (H / TILE_K), 128)
                           : make_map(&m_wgus, Wgu_shared, H, 2 * I, 64)) ||
                 !(packed ? make_map(&m_wds, Wd_shared, TILE_K,
                                     static_cast<uint64_t>(H) * (I / TILE_K), 128)
                          : make_map(&m_wds, Wd_shared, I, H, 128)) ||
                 !make_map(&m_x, X, H, B, xb_shared) || !make_map(&m_as, As, I, B, xb_shared)))
    return DEC_ERR_CUDA;

  if (consume_fault()) return DEC_ERR_CUDA;

  auto engine = [&](const CUtensorMap &wm, const CUtensorMap &xm, EngineParams &p,
                    cudaStream_t st_) -> cudaError_t {
    return tc ? launch_engine_tc(p.slot_cols, wm, xm, p, st_)
              : launch_engine_cc(p.slot_cols, wm, xm, p, st_);
  };
  auto base = [&](EngineParams &p, int mode, int N, int K, int T, int KB, int G, int grouped,
                  size_t part_off, size_t cnt_off) {
    std::memset(&p, 0, sizeof p);
    p.packed = packed ? 1 : 0;
    p.mode = mode;
    p.N = N;
    p.K = K;
    p.T = T;
    p.KB = KB;
    p.G = G;
    p.grouped = grouped;
    p.B = B;
    p.slot_cols = ep.maxc;
    p.ngrp = 1;
    p.wbox_rows = (mode == MODE_GATEUP) ? 64 : 128;
    p.xbox_rows = grouped ? XBOX_ROWS : xb_shared;
    p.E = E;
    p.P = P;
    p.route_map = rm;
    p.partials = reinterpret_cast<float *>(wsb + part_off);
    p.counters = reinterpret_cast<int *>(wsb + cnt_off);
    p.status = d->status;
    p.wait_limit_ns = g_wait_limit_ns.load();
  };

  auto set_combine = [&](EngineParams &p) {
    p.cmb_cnt = reinterpret_cast<int *>(wsb + ep.cmb_off);
    p.cmb_need = topk + (shared ? 1 : 0);
    p.topk = topk;
    p.topk_w = topk_w;
    p.cmb_yp = Yp;
    p.cmb_s = shared ? S : nullptr;
    p.cmb_y = reinterpret_cast<uint16_t *>(Y);
  };

  // ---- shared expert, side stream (or main when no second stream was given), unless
  // it runs inside the routed launch
  if (shared && !merged) {
    cudaStream_t sst = overlap ? ss : ms;
    const int gs = overlap ? g_side : d->num_sms;
    if (overlap) {
      if ((ce = cudaEventRecord(ev->fork, ms)) != cudaSuccess) return DEC_ERR_CUDA;
      if ((ce = cudaStreamWaitEvent(ss, ev->fork, 0)) != cudaSuccess) return DEC_ERR_CUDA;
    }
    EngineParams p;
    base(p, MODE_GATEUP, I, H, ep.Tg, ep.KBg, gs < ep.Tg * ep.KBg ? gs : ep.Tg * ep.KBg, 0,
         overlap ? ep.side_part_off : ep.main_part_off, overlap ? ep.side_cnt_off : ep.main_cnt_off);
    p.w_group_rows = 2 * I;
    p.up_row_off = I;
    p.A = As;
    p.w_base = packed ? nullptr : reinterpret_cast<const uint8_t *>(Wgu_shared);
    p.w_rows = 2LL * I;
    p.l2pf_kb = l2_prefetch_kblocks();
    if ((ce = engine(m_wgus, m_x, p, sst)) != cudaSuccess) return DEC_ERR_CUDA;
    base(p, MODE_DOWN, H, I, ep.Td, ep.KBd, gs < ep.Td * ep.KBd ? gs : ep.Td * ep.KBd, 0,
         overlap ? ep.side_part_off : ep.main_part_off, overlap ? ep.side_cnt_off : ep.main_cnt_off);
    p.w_group_rows = H;
    p.Yp = S;
    if (fused) set_combine(p);
    p.w_base = packed ? nullptr : reinterpret_cast<const uint8_t *>(Wd_shared);
    p.w_rows = H;
    p.l2pf_kb = l2_prefetch_kblocks();
    if ((ce = engine(m_wds, m_as, p, sst)) != cudaSuccess) return DEC_ERR_CUDA;
    if (overlap && (ce = cudaEventRecord(ev->join, ss)) != cudaSuccess) return DEC_ERR_CUDA;
  }

  // ---- moe_layer: the front end runs now, while the shared expert streams its
  // weights on the side stream, on the SMs the routed experts will use; it writes the
  // routing and the route map the routed launches read
  if (fc != nullptr) {
    st = run_front(X, fc->Wcat, B, H, E, fc->L, topk, fc->latent, const_cast<int32_t *>(topk_idx),
                   const_cast<float *>(topk_w), nullptr, rm, fc->ws, fc->ws_bytes, g_main, ms);
    if (st != DEC_OK) return st;
  }
  const bool have_map = route_map != nullptr || fc != nullptr;

  // ---- routed experts, main stream
  // without a route map the gather launch validates topk_idx and builds it
  int *dyn_ctr = reinterpret_cast<int *>(wsb + ep.dyn_off);
  const int xrows = merged ? B : 0;  // X's rows after the gathered ones: the shared expert's
  ce = have_map ? launch_gather_rows(X, rm, B, topk, E, H, Xg, dyn_ctr, 5 + E, xrows, ms)
                : launch_gather_map(X, topk_idx, B, topk, E, H, Xg, rm, d->status,
                                    2 * d->num_sms, dyn_ctr, 5 + E, xrows, ms);
  if (ce != cudaSuccess) return DEC_ERR_CUDA;
  {
    EngineParams p;
    // G <= T*KB keeps every worker range non-empty even with a single used expert
    const int gg = g_main < ep.Tg * ep.KBg ? g_main : ep.Tg * ep.KBg;
    const int gd = g_main < ep.Td * ep.KBd ? g_main : ep.Td * ep.KBd;
    // The gather launch waits for whatever wrote the route map and only then lets the
    // gate/up launch start; so when the map is not the gather's own output, it is
    // complete before gate/up starts, and likewise before down starts: both may then
    // read it, and issue their first weight loads, before their dependency wait.
    if (tc && expert_one_launch()) {
      // gate/up and down in one launch: whole tiles claimed at run time, each down tile
      // after its expert's gate/up tiles have stored A
      EngineParams p2;
      base(p, MODE_GATEUP, I, H, ep.Tg, ep.KBg, g_main, 1, ep.main_part_off, ep.main_cnt_off);
      p.w_group_rows = 2 * I;
      p.up_row_off = I;
      p.A = A;
      p.rm_ready = (have_map && early_route_map()) ? 1 : 0;
      p.dyn_ctr = dyn_ctr;
      p.ready = dyn_ctr + 4;
      p.with_shared = merged ? 1 : 0;
      p.w_base = packed ? reinterpret_cast<const uint8_t *>(Wgu) : nullptr;
      base(p2, MODE_DOWN, H, I, ep.Td, ep.KBd, g_main, 1, ep.main_part_off, ep.main_cnt_off);
      p2.w_group_rows = H;
      p2.Yp = Yp;
      if (fused) set_combine(p2);
      p2.rm_ready = p.rm_ready;
      p2.with_shared = p.with_shared;
      p2.w_base = packed ? reinterpret_cast<const uint8_t *>(Wd) : nullptr;
      if ((ce = launch_engine_tc_moe(ep.maxc, m_wgu, m_xg, m_wd, m_a, merged ? m_wgus : m_wgu,
                                     merged ? m_wds : m_wd, p, p2, ms)) != cudaSuccess)
        return DEC_ERR_CUDA;
    } else {
    // Whole-tile schedule once the CTAs expect enough tiles each that the last claims
    // even out the SMs' different read rates (tiles per CTA from the expected number of
    // distinct experts; with fewer, whole tiles are too coarse and stream-K ranges win).
    const int dyn = tc ? expert_dyn() : 0;
    const double dyn_min = expert_dyn_min_tiles();
    base(p, MODE_GATEUP, I, H, ep.Tg, ep.KBg, gg, 1, ep.main_part_off, ep.main_cnt_off);
    p.w_group_rows = 2 * I;
    p.up_row_off = I;
    p.A = A;
    p.rm_ready = (have_map && early_route_map()) ? 1 : 0;
    if (dyn > 0 && u_exp * ep.Tg >= dyn_min * gg) {
      p.dyn = dyn;
      p.dyn_ctr = dyn_ctr;
    }
    if ((ce = engine(m_wgu, m_xg, p, ms)) != cudaSuccess) return DEC_ERR_CUDA;
    base(p, MODE_DOWN, H, I, ep.Td, ep.KBd, gd, 1, ep.main_part_off, ep.main_cnt_off);
    p.w_group_rows = H;
    p.Yp = Yp;
    if (fused) set_combine(p);
    p.rm_ready = early_route_map() ? 1 : 0;
    if (dyn > 0 && u_exp * ep.Td >= dyn_min * gd) {
      p.dyn = dyn;
      p.dyn_ctr = dyn_ctr + 1;
    }
    if ((ce = engine(m_wd, m_a, p, ms)) != cudaSuccess) return DEC_ERR_CUDA;
    }
  }
  // Y is complete once both streams are done: the main stream waits for the side one
  if (overlap && (ce = cudaStreamWaitEvent(ms, ev->join, 0)) != cudaSuccess) return DEC_ERR_CUDA;
  if (!fused &&
      (ce = launch_combine(topk_w, rm, Yp,
                           shared ? (merged ? Yp + static_cast<size_t>(P) * H : S) : nullptr, B,
                           topk, E, H, Y, ms)) !=
          cudaSuccess)
    return DEC_ERR_CUDA;
  return DEC_OK;
}

}  // namespace

extern "C" {

// ------------------------------------------------------------- L2 prefetch ----

dec_status l2_prefetch(const void *p, size_t bytes, int max_ctas, dec_stream_t s) {
  if (!p || max_ctas < 0) return DEC_ERR_INVALID_ARG;
  if (!aligned16(p)) return DEC_ERR_MISALIGNED;
  bytes &= ~static_cast<size_t>(15);
  if (bytes == 0) return DEC_OK;
  if (consume_fault()) return DEC_ERR_CUDA;
  const int ctas = max_ctas == 0 ? 8 : max_ctas;
  return cuda_status(launch_l2_prefetch(p, bytes, ctas, reinterpret_cast<cudaStream_t>(s)));
}

dec_status dec_sim_comm_wait(uint64_t ns, dec_stream_t s) {
  if (ns < 1000ull || ns > 1000000000ull) return DEC_ERR_INVALID_ARG;
  if (consume_fault()) return DEC_ERR_CUDA;
  return cuda_status(launch_comm_wait(ns, reinterpret_cast<cudaStream_t>(s)));
}

size_t dec_read_stream_bytes(size_t bytes) {
  const size_t c = read_stream_claim_bytes();
  return (bytes / c) * c;
}

dec_status dec_read_stream(const void *p, size_t bytes, dec_stream_t s) {
  if (!p) return DEC_ERR_INVALID_ARG;
  if (!aligned16(p)) return DEC_ERR_MISALIGNED;
  cudaError_t ce;
  DeviceInfo *d = device_info(&ce);
  if (!d) return DEC_ERR_CUDA;
  if (bytes < read_stream_claim_bytes()) return DEC_OK;  // less than one chunk: nothing
  return cuda_status(launch_read_stream(p, bytes, d->num_sms, d->status,
                                        g_wait_limit_ns.load(),
                                        reinterpret_cast<cudaStream_t>(s)));
}

}  // extern "C"

// ======================================================= no-allocation variant ====
//
// Some callers cannot hand this library a workspace: code running inside a host
// program that owns the GPU memory pool and forbids allocation after start-up (a
// plugin inside another inference runtime, a serving loop whose memory was frozen
// after warm-up), or code that must not call cudaMalloc at all. dec_splitk_gemm_noalloc
// gives them the split-K projection with its scratch (per-worker partial tiles and
// per-tile arrival counters) in the fixed device array below, which every GPU that
// loads this library keeps until the process exits.

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch per device, looked up on the first call made with
// that device current. A failed lookup is not cached, so a later call can succeed (for
// example once a stream capture that made the first attempt fail has ended).
std::mutex g_noalloc_mu;
void *g_noalloc_addr[kMaxDevices] = {};

}  // namespace

extern "C" dec_status dec_splitk_gemm_noalloc(const dec_bf16 *X, const dec_bf16 *W,
                                              const dec_bf16 *R, dec_bf16 *Y, int B, int N,
                                              int K, int use_tc, dec_stream_t s) {
  dec_status st = check_linear_args(X, W, Y, B, N, K);
  if (st != DEC_OK) return st;
  if (use_tc != 0 && use_tc != 1) return DEC_ERR_INVALID_ARG;
  if (B > MAX_B && !use_tc) return DEC_ERR_UNSUPPORTED_SHAPE;  // wide: tensor cores only
  if (B > MAX_B_WIDE) return DEC_ERR_UNSUPPORTED_SHAPE;          // one launch only
  cudaError_t ce;
  DeviceInfo *d = device_info(&ce);
  if (!d) return DEC_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DEC_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DEC_ERR_CUDA;
  void *scratch = nullptr;
  {
    // The name g_noalloc_scratch is only a host-side stand-in: the array's device
    // address on this device (current here) comes from the runtime.
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr &&
        cudaGetSymbolAddress(&g_noalloc_addr[dev], g_noalloc_scratch) != cudaSuccess) {
      g_noalloc_addr[dev] = nullptr;
      return DEC_ERR_CUDA;
    }
    scratch = g_noalloc_addr[dev];
  }
  SplitPlan pl;
  if (!plan_splitk(B, N, K, 0, d->num_sms, &pl)) return DEC_ERR_UNSUPPORTED_SHAPE;
  if (pl.total > kNoAllocScratchBytes) return DEC_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
  // 129..256 rows: the CTA-pair launch, as dec_splitk_gemm takes it (it uses no scratch)
  if (use_pair_kernel(B, N, K, 0, use_tc, d->num_sms))
    return run_pair_projection(X, W, R, Y, B, N, K, scratch, kNoAllocScratchBytes, cs, false);
  // The arrival counters must start at zero. Every call that completes leaves them at
  // zero, and the array starts zeroed, but a call whose kernel gave up on a bounded
  // wait can leave some set; clearing them here makes the next call correct anyway.
  // The partial tiles are always written before they are read.
  if (cudaMemsetAsync(static_cast<char *>(scratch) + pl.partial_bytes, 0, pl.counter_bytes,
                      cs) != cudaSuccess)
    return DEC_ERR_CUDA;
  // The same planning, schedule choice (two-halves clusters, deferred finish) and
  // kernels as dec_splitk_gemm with split_k = 0, so the bits are the same too.
  return run_splitk_rows(X, W, R, Y, B, N, K, 0, use_tc, scratch, kNoAllocScratchBytes, cs);
}
