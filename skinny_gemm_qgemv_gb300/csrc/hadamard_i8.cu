// Block-32 randomized Hadamard transform + per-row symmetric int8, and the
// exact W8A8 int32 product.
//
// Uzu article, section "How Uzu optimizes bytes and tokens per pass":
// activations are quantized to 8 bits at run time; before that a block-
// diagonal randomized Hadamard transform (random sign flips, then a +-1
// Hadamard on every 32-value block, matching a 32-wide SIMD group) spreads
// outliers over the block; it is exactly invertible. Both int8 operands then
// feed an integer matrix product.
//
// GB300 mapping: one 32-element block is one warp, one element per lane; the
// five butterfly stages are __shfl_xor_sync exchanges with plain fp32 add/sub
// (no FMA), spans 1, 2, 4, 8, 16 in that order, so every rounding matches the
// fixed reference order. The row maximum goes through shared memory, then
// s = max / 127 and q = rint(z / s) use IEEE division and round-half-even.
#include <cuda_runtime.h>

#include <algorithm>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

__global__ void __launch_bounds__(256) hadamard32_quant_i8_kernel(const uint16_t* __restrict__ x,
                                                                  const uint32_t* __restrict__ sign_bits,
                                                                  int8_t* __restrict__ q, float* __restrict__ scale,
                                                                  int K) {
  extern __shared__ float zrow[];  // [K]
  __shared__ float wmax[8];
  pdl_wait();
  const int m = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = K / 32;
  float amax = 0.f;
  for (int b = warp; b < nb; b += 8) {
    float v = bf16_bits_to_f32(x[(size_t)m * K + 32 * b + lane]);
    if ((sign_bits[b] >> lane) & 1u) v = -v;
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
      const float p = __shfl_xor_sync(0xffffffffu, v, h);
      v = (lane & h) ? __fsub_rn(p, v) : __fadd_rn(v, p);
    }
    zrow[32 * b + lane] = v;
    amax = fmaxf(amax, fabsf(v));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) wmax[warp] = amax;
  __syncthreads();
  float mx = wmax[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) mx = fmaxf(mx, wmax[w]);
  const float s = __fdiv_rn(mx, 127.0f);
  if (threadIdx.x == 0) scale[m] = s;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    int8_t code = 0;
    if (s > 0.f) {
      float r = rintf(__fdiv_rn(zrow[k], s));
      r = fminf(fmaxf(r, -127.f), 127.f);
      code = (int8_t)(int)r;
    }
    q[(size_t)m * K + k] = code;
  }
}

cudaError_t launch_hadamard32_quant_i8(const uint16_t* x, const uint32_t* sign_bits, int8_t* q, float* scale,
                                       int M, int K, cudaStream_t stream, bool pdl) {
  const size_t smem = sizeof(float) * (size_t)K;
  cudaError_t e = allow_max_smem(hadamard32_quant_i8_kernel);
  if (e != cudaSuccess) return e;
  return launch_kernel(hadamard32_quant_i8_kernel, dim3(M), dim3(256), smem, stream, pdl, x, sign_bits, q, scale,
                       K);
}

// ---------------------------------------------------------------------------
// W8A8: C[m][n] = sum_k a[m][k] w[n][k], exact in int32 (dp4a, integer adds).
// One warp per output column n; 16-byte weight loads; activations via L1.
// ---------------------------------------------------------------------------
template <int MMAX>
__global__ void __launch_bounds__(256) w8a8_dp4a_kernel(const int8_t* __restrict__ a, const int8_t* __restrict__ w,
                                                        int32_t* __restrict__ c, int M, int N, int K) {
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + warp;
  if (n >= N) return;
  int acc[MMAX];
#pragma unroll
  for (int m = 0; m < MMAX; ++m) acc[m] = 0;
  for (int k = lane * 16; k < K; k += 512) {
    const uint4 wv = ldg_stream128(w + (size_t)n * K + k);
#pragma unroll
    for (int m = 0; m < MMAX; ++m) {
      if (m < M) {
        const int4 av = __ldg(reinterpret_cast<const int4*>(a + (size_t)m * K + k));
        acc[m] = __dp4a((int)wv.x, av.x, acc[m]);
        acc[m] = __dp4a((int)wv.y, av.y, acc[m]);
        acc[m] = __dp4a((int)wv.z, av.z, acc[m]);
        acc[m] = __dp4a((int)wv.w, av.w, acc[m]);
      }
    }
  }
#pragma unroll
  for (int m = 0; m < MMAX; ++m) {
    if (m < M) {
      int v = acc[m];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) c[(size_t)m * N + n] = v;
    }
  }
}

// Tiled W8A8 for the skinny shapes: a producer warp streams the weights and
// the activations of each 1024-k chunk through shared memory (cp.async.bulk,
// one row segment per copy) and each consumer lane keeps NC columns x MMAX rows
// of int32 sums in registers, so one 16-byte activation load feeds NC columns
// (the one-warp-per-column kernel above loads every activation once per
// column, from L1). Tile: 8 warps x NC columns x the whole K.
constexpr int kW8Warps = 8;
constexpr int kW8Chunk = 1024;  // k per stage
// stages in flight (weights + activations of a chunk per stage, <= 216 KB)
constexpr int w8_stages(int nc) { return nc >= 8 ? 3 : 4; }

template <int MMAX, int NC>
__global__ void __launch_bounds__(32 * (kW8Warps + 1), 1)
    w8a8_tile_kernel(const int8_t* __restrict__ a, const int8_t* __restrict__ w, int32_t* __restrict__ c, int M,
                     int N, int K, uint32_t* err) {
  constexpr int kCols = kW8Warps * NC;  // columns per tile
  constexpr uint32_t kActOff = kCols * kW8Chunk;  // the chunk's activations [MMAX][1024] after its weights
  constexpr uint32_t kStage = (kCols + MMAX) * kW8Chunk;
  constexpr int kW8Stages = w8_stages(NC);
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kW8Stages * kStage);
  uint64_t* empty = full + kW8Stages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kW8Stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kW8Warps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  const int ntiles = (N + kCols - 1) / kCols, nchunk = (K + kW8Chunk - 1) / kW8Chunk;
  if (warp == kW8Warps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const int n0 = t * kCols, cols = min(kCols, N - n0);
        for (int kc = 0; kc < nchunk; ++kc, ++it) {
          const int st = it % kW8Stages;
          if (it >= kW8Stages) ok = mbar_wait(&empty[st], ((it / kW8Stages) & 1) ^ 1, err, kErrGemvEmptyWait);
          if (!ok) break;
          const uint32_t len = (uint32_t)min(kW8Chunk, K - kc * kW8Chunk);
          mbar_arrive_expect_tx(&full[st], (uint32_t)(cols + M) * len);
          for (int j = 0; j < cols; ++j)
            bulk_g2s_evict_first(smem + (size_t)st * kStage + (size_t)j * kW8Chunk,
                                 w + (size_t)(n0 + j) * K + (size_t)kc * kW8Chunk, len, &full[st], pol);
          for (int m = 0; m < M; ++m)
            bulk_g2s(smem + (size_t)st * kStage + kActOff + (size_t)m * kW8Chunk,
                     a + (size_t)m * K + (size_t)kc * kW8Chunk, len, &full[st]);
        }
      }
      for (int j = max(0, it - kW8Stages); j < it; ++j)
        mbar_wait(&full[j % kW8Stages], (j / kW8Stages) & 1, err, kErrGemvDrain);
    }
    return;
  }
  // ------------------------------------------------------------------ consumers
  int it = 0;
  for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int n0 = t * kCols;
    int acc[NC * MMAX];
#pragma unroll
    for (int q = 0; q < NC * MMAX; ++q) acc[q] = 0;
    for (int kc = 0; kc < nchunk; ++kc, ++it) {
      const int st = it % kW8Stages;
      if (!mbar_wait(&full[st], (it / kW8Stages) & 1, err, kErrGemvFullWait)) break;
      const uint32_t sb = smem_u32(smem + (size_t)st * kStage + (size_t)warp * NC * kW8Chunk);
      const uint32_t sa = smem_u32(smem + (size_t)st * kStage + kActOff);
#pragma unroll
      for (int i = 0; i < kW8Chunk / 512; ++i) {
        const int kl = 16 * lane + 512 * i, k = kc * kW8Chunk + kl;
        if (k < K) {
          uint4 wv[NC];
#pragma unroll
          for (int j = 0; j < NC; ++j) wv[j] = lds128(sb + j * kW8Chunk + kl);
#pragma unroll
          for (int m = 0; m < MMAX; ++m) {
            if (m < M) {
              const uint4 av = lds128(sa + m * kW8Chunk + kl);
#pragma unroll
              for (int j = 0; j < NC; ++j) {
                int v = acc[j * MMAX + m];
                v = __dp4a((int)wv[j].x, (int)av.x, v);
                v = __dp4a((int)wv[j].y, (int)av.y, v);
                v = __dp4a((int)wv[j].z, (int)av.z, v);
                v = __dp4a((int)wv[j].w, (int)av.w, v);
                acc[j * MMAX + m] = v;
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    // lane sums of the NC x MMAX values, 32 at a time (exact integer adds)
#pragma unroll
    for (int h = 0; h < NC * MMAX; h += 32) {
      int v[32];
#pragma unroll
      for (int q = 0; q < 32; ++q) v[q] = acc[h + q];
      const int tot = transposed_warp_sum<32>(v, lane);
      const int q = h + transposed_row<32>(lane);
      const int j = q / MMAX, m = q % MMAX, n = n0 + warp * NC + j;
      if (m < M && n < N) c[(size_t)m * N + n] = tot;
    }
  }
}

template <int MMAX, int NC>
static cudaError_t launch_w8a8_tile(const int8_t* a, const int8_t* w, int32_t* c, int M, int N, int K,
                                    uint32_t* err, cudaStream_t stream, bool pdl) {
  auto kern = w8a8_tile_kernel<MMAX, NC>;
  const size_t smem = (size_t)w8_stages(NC) * (kW8Warps * NC + MMAX) * kW8Chunk + 2 * w8_stages(NC) * 8;
  cudaError_t e = allow_max_smem(kern);
  if (e != cudaSuccess) return e;
  const int ntiles = (N + kW8Warps * NC - 1) / (kW8Warps * NC);
  const int grid = std::min(ntiles, device_sm_count());
  return launch_kernel(kern, dim3(grid), dim3(32 * (kW8Warps + 1)), smem, stream, pdl, a, w, c, M, N, K, err);
}

cudaError_t launch_w8a8_i32(const int8_t* a, const int8_t* w, int32_t* c, int M, int N, int K, uint32_t* err,
                            cudaStream_t stream, bool pdl) {
  // M <= 16 with K a multiple of 512: the tensor cores through exact fp16 operands
  if (err && w8a8_mma_ok(M, N, K)) return launch_w8a8_mma(a, w, c, M, N, K, err, stream, pdl);
  // other wide matrices: the tiled kernel (NC x MMAX = 64 sums per lane); else one warp per column
  if (err && N >= 4 * kW8Warps * device_sm_count() / 4) {
    if (M <= 8) return launch_w8a8_tile<8, 8>(a, w, c, M, N, K, err, stream, pdl);
    if (M <= 16) return launch_w8a8_tile<16, 4>(a, w, c, M, N, K, err, stream, pdl);
    return launch_w8a8_tile<32, 2>(a, w, c, M, N, K, err, stream, pdl);
  }
  dim3 grid((N + 7) / 8), block(256);
  if (M <= 4) return launch_kernel(w8a8_dp4a_kernel<4>, grid, block, 0, stream, pdl, a, w, c, M, N, K);
  if (M <= 8) return launch_kernel(w8a8_dp4a_kernel<8>, grid, block, 0, stream, pdl, a, w, c, M, N, K);
  if (M <= 16) return launch_kernel(w8a8_dp4a_kernel<16>, grid, block, 0, stream, pdl, a, w, c, M, N, K);
  return launch_kernel(w8a8_dp4a_kernel<32>, grid, block, 0, stream, pdl, a, w, c, M, N, K);
}

}  // namespace qg
