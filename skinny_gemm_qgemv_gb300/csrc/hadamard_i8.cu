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

cudaError_t launch_w8a8_i32(const int8_t* a, const int8_t* w, int32_t* c, int M, int N, int K,
                            cudaStream_t stream, bool pdl) {
  dim3 grid((N + 7) / 8), block(256);
  if (M <= 4) return launch_kernel(w8a8_dp4a_kernel<4>, grid, block, 0, stream, pdl, a, w, c, M, N, K);
  if (M <= 8) return launch_kernel(w8a8_dp4a_kernel<8>, grid, block, 0, stream, pdl, a, w, c, M, N, K);
  if (M <= 16) return launch_kernel(w8a8_dp4a_kernel<16>, grid, block, 0, stream, pdl, a, w, c, M, N, K);
  return launch_kernel(w8a8_dp4a_kernel<32>, grid, block, 0, stream, pdl, a, w, c, M, N, K);
}

}  // namespace qg
