// gemv_tiny.cu -- tiny-matrix projection for decode batches of 1 to 4.
//
// "Hyper Optimizing Kimi K3 in vLLM", Part 1 / 1 "Tune shapes for the workload": at
// batch sizes 1-2 the projections use a dedicated small-matrix kernel.
//
//     Y[b,n] = bf16( sum_k X[b,k] W[n,k] (+ R[b,n]) ),  b < NB in 1..4
//
// Design (GB300): the op moves N*K*2 bytes of weights and does 2*NB flops per weight,
// so at NB = 1-2 it is bound by HBM bandwidth (from NB = 3 on, by instruction issue:
// bf16 unpacking plus NB fp32 FMAs per weight). Each CTA owns a contiguous block of rows; its 8
// warps split every row into P k-pieces and cover the rows in R row-slots
// (8 = P * R). A lane streams 16-byte weight chunks with the non-coherent,
// no-L1-allocate load (16 loads in flight per lane: 4 rows x 4 chunks), multiplies
// them with the matching activation chunks (coherent loads, L1-resident), and keeps
// NB x 4 fp32 partial sums in registers. A warp reduces them with shuffles; the P
// piece sums of a row are added in piece order from shared memory. The result does
// not depend on launch timing: every sum has a fixed order. Under programmatic
// dependent launch the first weight loads are issued before griddepcontrol.wait and
// every activation load after it (asm volatile loads with a memory clobber, so the
// compiler cannot hoist them above the wait).
//
// A tile-packed W (dec_pack_weight: 16 KB blocks of 128 rows x 64 k, block (n/128, k/64)
// at index (n/128)*(K/64) + k/64, rows of 128 bytes inside) has its own kernel below: a
// warp's load covers 4 adjacent rows x 128 bytes of one block (512 contiguous bytes)
// instead of 512 bytes along one row.
#include "common.cuh"
#include "internal.h"

namespace ssd {

namespace {

constexpr int TINY_THREADS = 256;
constexpr int TINY_WARPS = TINY_THREADS / 32;
constexpr int TINY_RG = 4;   // rows per warp iteration
constexpr int TINY_JU = 4;   // 16-byte chunks per lane per row per iteration
constexpr int TINY_MAX_ROWS_PER_CTA = 512;

// Coherent 128-bit activation load, kept after any preceding wait by asm volatile.
__device__ __forceinline__ uint4 ld_act_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ float dot8(const uint4 &w, const uint4 &x, float acc) {
  acc = fmaf(bf16lo(w.x), bf16lo(x.x), acc);
  acc = fmaf(bf16hi(w.x), bf16hi(x.x), acc);
  acc = fmaf(bf16lo(w.y), bf16lo(x.y), acc);
  acc = fmaf(bf16hi(w.y), bf16hi(x.y), acc);
  acc = fmaf(bf16lo(w.z), bf16lo(x.z), acc);
  acc = fmaf(bf16hi(w.z), bf16hi(x.z), acc);
  acc = fmaf(bf16lo(w.w), bf16lo(x.w), acc);
  acc = fmaf(bf16hi(w.w), bf16hi(x.w), acc);
  return acc;
}

template <int NB>
__global__ void __launch_bounds__(TINY_THREADS, 2)
    gemv_tiny_kernel(const uint16_t *X, const uint16_t *__restrict__ W, const uint16_t *R,
                     uint16_t *Y, int N, int K, int P, int early_trigger) {
  extern __shared__ float red[];  // [rows of this CTA][P][NB]
  const int C = K >> 3;           // 16-byte chunks per row
  const int G = gridDim.x;
  const int r0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * N / G);
  const int r1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * N / G);
  const int nrows = r1 - r0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = TINY_WARPS / P;  // row slots
  const int piece = warp % P, slot = warp / P;
  const int cb = static_cast<int>(static_cast<int64_t>(piece) * C / P);
  const int ce = static_cast<int>(static_cast<int64_t>(piece + 1) * C / P);
  const uint8_t *Wb = reinterpret_cast<const uint8_t *>(W);
  const uint8_t *Xb = reinterpret_cast<const uint8_t *>(X);
  const size_t row_bytes = static_cast<size_t>(K) * 2;
  bool waited = false;  // the first weight loads go out before the dependency wait

  for (int rl = slot; rl < nrows; rl += S * TINY_RG) {
    float acc[TINY_RG][NB];
#pragma unroll
    for (int g = 0; g < TINY_RG; ++g)
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[g][b] = 0.f;

    for (int c = cb + lane; c < ce; c += 32 * TINY_JU) {
      uint4 wv[TINY_RG][TINY_JU];
#pragma unroll
      for (int g = 0; g < TINY_RG; ++g) {
        const int row = rl + g * S;
#pragma unroll
        for (int u = 0; u < TINY_JU; ++u) {
          const int cc = c + 32 * u;
          if (cc < ce && row < nrows)
            wv[g][u] = ld_weight_stream(Wb + static_cast<size_t>(r0 + row) * row_bytes +
                                        static_cast<size_t>(cc) * 16);
          else
            wv[g][u] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if (!waited) {  // activations are written by the previous kernel of the stream
        griddep_wait();
        waited = true;
        // small matrices: every weight load of this CTA is out, let the next kernel of the
        // stream start on the half of the SM this one leaves free (see gemv_tiny_grid)
        if (early_trigger) griddep_launch_dependents();
      }
#pragma unroll
      for (int u = 0; u < TINY_JU; ++u) {
        const int cc = c + 32 * u;
        if (cc < ce) {
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const uint4 xv = ld_act_v4(Xb + static_cast<size_t>(b) * row_bytes +
                                       static_cast<size_t>(cc) * 16);
#pragma unroll
            for (int g = 0; g < TINY_RG; ++g) acc[g][b] = dot8(wv[g][u], xv, acc[g][b]);
          }
        }
      }
    }
#pragma unroll
    for (int g = 0; g < TINY_RG; ++g) {
      const int row = rl + g * S;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float v = acc[g][b];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
        if (lane == 0 && row < nrows) red[(row * P + piece) * NB + b] = v;
      }
    }
  }
  griddep_launch_dependents();  // all weight loads of this CTA are done
  griddep_wait();               // before the residual read and the output write
  __syncthreads();
  for (int i = threadIdx.x; i < nrows * NB; i += TINY_THREADS) {
    const int row = i / NB, b = i - row * NB;
    float s = 0.f;
    for (int pc = 0; pc < P; ++pc) s += red[(row * P + pc) * NB + b];
    const int n = r0 + row;
    if (R != nullptr) s += bf16_to_f32(R[static_cast<size_t>(b) * N + n]);
    Y[static_cast<size_t>(b) * N + n] = f32_to_bf16_rn(s);
  }
}

// Tile-packed W. The CTA owns whole quads of rows (4 consecutive rows, never across a
// 128-row tile); lane l handles row 4q + l/8 of a quad and the 16-byte chunk l%8 of a
// 64-wide k-block, so one load instruction of a warp reads 4 rows x 128 bytes, contiguous
// in the packed block. Warp (piece, slot) covers k-blocks [KB*piece/P, KB*(piece+1)/P)
// of RG quads per iteration, quads slot, slot + S, ... interleaved over the S slots as
// the row-major kernel interleaves rows (RG x JU = 16 loads in flight per lane); the
// eight lanes of a row are added with three shuffles, the P pieces in piece order.
template <int NB>
__global__ void __launch_bounds__(TINY_THREADS, 2)
    gemv_tiny_packed_kernel(const uint16_t *X, const uint16_t *__restrict__ W, const uint16_t *R,
                            uint16_t *Y, int N, int K, int P, int early_trigger) {
  extern __shared__ float red[];  // [rows of this CTA][P][NB]
  const int KB = K >> 6;
  const int Q = N >> 2;  // quads
  const int G = gridDim.x;
  const int q0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * Q / G);
  const int q1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * Q / G);
  const int nq = q1 - q0, r0 = 4 * q0, nrows = 4 * nq;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r4 = lane >> 3, c8 = lane & 7;
  const int S = TINY_WARPS / P;
  const int piece = warp % P, slot = warp / P;
  const int kbb = static_cast<int>(static_cast<int64_t>(piece) * KB / P);
  const int kbe = static_cast<int>(static_cast<int64_t>(piece + 1) * KB / P);
  const uint8_t *Wb = reinterpret_cast<const uint8_t *>(W);
  const uint8_t *Xb = reinterpret_cast<const uint8_t *>(X);
  const size_t row_bytes = static_cast<size_t>(K) * 2;
  bool waited = false;

  for (int qq = slot; qq < nq; qq += S * TINY_RG) {
    float acc[TINY_RG][NB];
#pragma unroll
    for (int g = 0; g < TINY_RG; ++g)
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[g][b] = 0.f;

    for (int kb = kbb; kb < kbe; kb += TINY_JU) {
      uint4 wv[TINY_RG][TINY_JU];
#pragma unroll
      for (int g = 0; g < TINY_RG; ++g) {
        const int n = r0 + 4 * (qq + g * S) + r4;  // global row
#pragma unroll
        for (int u = 0; u < TINY_JU; ++u) {
          if (kb + u < kbe && qq + g * S < nq) {
            const size_t blk = static_cast<size_t>(n >> 7) * KB + static_cast<size_t>(kb + u);
            wv[g][u] = ld_weight_stream(Wb + ((blk << 7) + static_cast<size_t>(n & 127)) * 128 +
                                        static_cast<size_t>(c8) * 16);
          } else {
            wv[g][u] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      if (!waited) {  // activations are written by the previous kernel of the stream
        griddep_wait();
        waited = true;
        if (early_trigger) griddep_launch_dependents();
      }
#pragma unroll
      for (int u = 0; u < TINY_JU; ++u) {
        if (kb + u < kbe) {
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const uint4 xv = ld_act_v4(Xb + static_cast<size_t>(b) * row_bytes +
                                       static_cast<size_t>((kb + u) * 8 + c8) * 16);
#pragma unroll
            for (int g = 0; g < TINY_RG; ++g) acc[g][b] = dot8(wv[g][u], xv, acc[g][b]);
          }
        }
      }
    }
#pragma unroll
    for (int g = 0; g < TINY_RG; ++g) {
      const int row = 4 * (qq + g * S) + r4;  // local row
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float v = acc[g][b];
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
        if (c8 == 0 && qq + g * S < nq) red[(row * P + piece) * NB + b] = v;
      }
    }
  }
  griddep_launch_dependents();
  griddep_wait();
  __syncthreads();
  for (int i = threadIdx.x; i < nrows * NB; i += TINY_THREADS) {
    const int row = i / NB, b = i - row * NB;
    float s = 0.f;
    for (int pc = 0; pc < P; ++pc) s += red[(row * P + pc) * NB + b];
    const int n = r0 + row;
    if (R != nullptr) s += bf16_to_f32(R[static_cast<size_t>(b) * N + n]);
    Y[static_cast<size_t>(b) * N + n] = f32_to_bf16_rn(s);
  }
}

int tiny_pieces(int K) {
  const int C = K / 8;
  int P = 1;
  while (P < TINY_WARPS && C / (2 * P) >= 64) P *= 2;
  return P;
}


// Weight matrices up to this size get one CTA per SM instead of two: all of a CTA's
// loads are in flight at once anyway, and the other half of each SM is left to the next
// kernel of the stream, which then loads its own weights while this one finishes
// (triggered right after the first weight loads).
constexpr size_t TINY_SMALL_BYTES = size_t(16) << 20;

bool tiny_small(int N, int K) { return static_cast<size_t>(N) * K * 2 <= TINY_SMALL_BYTES; }

}  // namespace

int gemv_tiny_grid(int N, int K, int num_sms) {
  int g = tiny_small(N, K) ? num_sms : 2 * num_sms;
  const int need = (N + TINY_MAX_ROWS_PER_CTA - 1) / TINY_MAX_ROWS_PER_CTA;
  if (g < need) g = need;
  if (g > N) g = N;
  return g;
}

template <int NB>
cudaError_t launch_tiny_nb(const uint16_t *X, const uint16_t *W, const uint16_t *R, uint16_t *Y,
                           int N, int K, int G, int P, int early, size_t smem, bool packed,
                           cudaStream_t s) {
  return packed ? launch_pdl(gemv_tiny_packed_kernel<NB>, dim3(G), dim3(TINY_THREADS), smem, s, X,
                             W, R, Y, N, K, P, early)
                : launch_pdl(gemv_tiny_kernel<NB>, dim3(G), dim3(TINY_THREADS), smem, s, X, W, R,
                             Y, N, K, P, early);
}

cudaError_t launch_gemv_tiny(const uint16_t *X, const uint16_t *W, const uint16_t *R,
                             uint16_t *Y, int B, int N, int K, int num_sms, cudaStream_t s,
                             bool packed) {
  int G = gemv_tiny_grid(N, K, num_sms);
  if (packed && G > N / 4) G = N / 4;  // whole quads of rows per CTA
  const int P = tiny_pieces(K);
  const int early = tiny_small(N, K) ? 1 : 0;
  // rows of the largest CTA: whole quads when packed
  const int rows = packed ? 4 * ((N / 4 + G - 1) / G) : (N + G - 1) / G;
  const size_t smem = static_cast<size_t>(rows) * P * B * sizeof(float);
  switch (B) {
    case 1: return launch_tiny_nb<1>(X, W, R, Y, N, K, G, P, early, smem, packed, s);
    case 2: return launch_tiny_nb<2>(X, W, R, Y, N, K, G, P, early, smem, packed, s);
    case 3: return launch_tiny_nb<3>(X, W, R, Y, N, K, G, P, early, smem, packed, s);
    case 4: return launch_tiny_nb<4>(X, W, R, Y, N, K, G, P, early, smem, packed, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ssd
