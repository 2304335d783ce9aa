// engine_cc.cu -- split-K engine with CUDA-core tiles.
//
// One CTA per SM: warp 8 lane 0 is the TMA producer, warps 0..7 compute. Weight tiles
// (128 rows x 64 k, two 64-row boxes) and activation tiles (16-row boxes) arrive by TMA
// with the 128-byte swizzle into an 8-deep ring of shared-memory stages guarded by
// full/empty mbarriers. Consumer thread (r, h) owns tile row r and k-half h: per stage
// it unpacks its 32 weights once and multiplies them with every batch column
// (broadcast reads of the activation row), accumulating in fp32 registers. At the end
// of a segment the two k-halves are added (h0 + h1) and the shared reduction and
// epilogue of engine.cuh run.
#include <atomic>

#include "engine.cuh"

namespace ssd {

namespace {

constexpr int CC_THREADS = 288;  // 8 consumer warps + 1 producer warp
constexpr int SMEM_LIMIT = 232448;

template <int MAXC>
struct CCConfig {
  static constexpr int NXB = (MAXC + 15) / 16;
  static constexpr int STAGE_BYTES = 16384 + NXB * 2048;
  static constexpr int SCRATCH_BYTES = 128 * MAXC * 4;
  static constexpr int BUDGET = SMEM_LIMIT - 1024 - 256;
  static constexpr int FIT = (BUDGET - SCRATCH_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = FIT > 8 ? 8 : FIT;
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + SCRATCH_BYTES + 256;
  static_assert(STAGES >= 4, "pipeline too shallow");
};

template <int MAXC>
__device__ __forceinline__ void cc_compute(const uint8_t *st, int r, int h, int ncols,
                                           float (&acc)[MAXC]) {
  float wf[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = h * 4 + i;
    const uint4 u = *reinterpret_cast<const uint4 *>(st + r * 128 + ((c ^ (r & 7)) << 4));
    wf[8 * i + 0] = bf16lo(u.x);
    wf[8 * i + 1] = bf16hi(u.x);
    wf[8 * i + 2] = bf16lo(u.y);
    wf[8 * i + 3] = bf16hi(u.y);
    wf[8 * i + 4] = bf16lo(u.z);
    wf[8 * i + 5] = bf16hi(u.z);
    wf[8 * i + 6] = bf16lo(u.w);
    wf[8 * i + 7] = bf16hi(u.w);
  }
  const uint8_t *xt = st + 16384;
#pragma unroll
  for (int j = 0; j < MAXC; ++j) {
    if (j < ncols) {
      float a = acc[j];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = h * 4 + i;
        const uint4 u =
            *reinterpret_cast<const uint4 *>(xt + j * 128 + ((c ^ (j & 7)) << 4));
        a = fmaf(wf[8 * i + 0], bf16lo(u.x), a);
        a = fmaf(wf[8 * i + 1], bf16hi(u.x), a);
        a = fmaf(wf[8 * i + 2], bf16lo(u.y), a);
        a = fmaf(wf[8 * i + 3], bf16hi(u.y), a);
        a = fmaf(wf[8 * i + 4], bf16lo(u.z), a);
        a = fmaf(wf[8 * i + 5], bf16hi(u.z), a);
        a = fmaf(wf[8 * i + 6], bf16lo(u.w), a);
        a = fmaf(wf[8 * i + 7], bf16hi(u.w), a);
      }
      acc[j] = a;
    }
  }
}

template <int MAXC>
__global__ void __launch_bounds__(CC_THREADS, 1)
    engine_cc_kernel(const __grid_constant__ CUtensorMap wmap,
                     const __grid_constant__ CUtensorMap xmap, const EngineParams p) {
  using C = CCConfig<MAXC>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *stage_mem = smem;
  float *scratch = reinterpret_cast<float *>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::STAGES * C::STAGE_BYTES +
                                                C::SCRATCH_BYTES);
  uint64_t *empty = full + C::STAGES;
  volatile int *flags = reinterpret_cast<volatile int *>(empty + C::STAGES);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int w = blockIdx.x;
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
      mbar_init(&empty[s], 8);
    }
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 8) {
    // ---------------------------------------------------------------- producer
    if (!p.grouped) prefetch_weights_l2(p, begin, end, C::STAGES, lane);
    if (lane == 0)
      engine_produce<C::STAGES, C::STAGE_BYTES>(p, &wmap, &xmap, stage_mem, full, empty, flags,
                                                begin, end);
    else
      griddep_wait();
  } else {
    // --------------------------------------------------------------- consumers
    griddep_wait();
    const int r = tid & 127, h = tid >> 7;
    uint32_t q = 0;
    for (int64_t it = begin; it < end;) {
      SegInfo s;
      seg_info(p, it, end, s);
      float acc[MAXC];
#pragma unroll
      for (int j = 0; j < MAXC; ++j) acc[j] = 0.f;
      for (int kb = s.kb0; kb < s.kb1; ++kb, ++q) {
        const int st = static_cast<int>(q % C::STAGES);
        const uint32_t par = (q / C::STAGES) & 1u;
        if (!mbar_wait_bounded(&full[st], par, p.status, flags, p.wait_limit_ns)) break;
        cc_compute<MAXC>(stage_mem + st * C::STAGE_BYTES, r, h, s.ncols, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
      named_bar_sync(1, 256);
      if (flags[0]) break;  // uniform across the 256 consumers after the barrier
      if (h == 1) {
#pragma unroll
        for (int j = 0; j < MAXC; ++j)
          if (j < s.ncols) scratch[j * 128 + r] = acc[j];
      }
      named_bar_sync(1, 256);
      if (h == 0) {
#pragma unroll
        for (int j = 0; j < MAXC; ++j)
          if (j < s.ncols) acc[j] += scratch[j * 128 + r];
        if (reduce_tile<MAXC>(p, s, total, w, begin, r, acc, 2, flags))
          epilogue_rows<MAXC>(p, s, r, acc, scratch, 2, flags);
      }
      it += s.kb1 - s.kb0;
    }
  }
  __syncthreads();
}

// The shared-memory opt-in is a per-device function attribute: set it on the first
// launch on each device (outside any later stream capture), not on every launch.
template <int MAXC>
cudaError_t launch_t(const CUtensorMap &wmap, const CUtensorMap &xmap, const EngineParams &p,
                     cudaStream_t s) {
  using C = CCConfig<MAXC>;
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(engine_cc_kernel<MAXC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  return launch_pdl(engine_cc_kernel<MAXC>, dim3(p.G), dim3(CC_THREADS), C::SMEM, s, wmap, xmap, p);
}

}  // namespace

int engine_maxc_for(int ncols) {
  int m = 2;
  while (m < ncols) m *= 2;
  return m;
}

cudaError_t launch_engine_cc(int maxc, const CUtensorMap &wmap, const CUtensorMap &xmap,
                             const EngineParams &p, cudaStream_t s) {
  if (p.ngrp != 1) return cudaErrorInvalidValue;  // wide projections: tensor cores only
  if (p.dyn) return cudaErrorInvalidValue;        // whole-tile schedule: tensor cores only
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
