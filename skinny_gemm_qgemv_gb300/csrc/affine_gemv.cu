// Affine quantized GEMV / skinny GEMM at any of the widths of the affine
// format: 2, 3, 4, 5, 6 or 8 bits, groups of 32, 64 or 128 codes.
//
// "MLX Runner: An Inference Engine You Can Read", section "Architecture: one
// command buffer per token": weights are stored as integer codes plus one
// scale and one bias per group (weight = scale x code + bias) at 2, 3, 4, 5, 6
// or 8 bits and group sizes 32, 64 or 128, and the kernels multiply against the
// packed codes directly, with no dequantized copy.
//
// Layout: the codes of a row form one little-endian bit stream (code k in bits
// [bits*k, bits*k + bits), bit j in bit j % 32 of word j / 32); at 4 bits this
// is the W4A16 layout. This is the generic path, one warp per output row: lane
// l takes codes l, l + 32, ..., reads the one or two words holding its code,
// dequantizes in fp32 and accumulates for every activation row. The 4-bit g64
// case has its own fast kernels (qgemv_w4a16, qgemm_w4a16_skinny).
#include <cuda_runtime.h>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

template <int MMAX>
__global__ void __launch_bounds__(256) affine_generic_kernel(const uint32_t* __restrict__ wq, int bits,
                                                             const uint16_t* __restrict__ scales,
                                                             const uint16_t* __restrict__ biases,
                                                             const uint16_t* __restrict__ x, float* __restrict__ y,
                                                             int M, int N, int K, int lg_group) {
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + warp;
  if (n >= N) return;
  const uint32_t words = (uint32_t)(((uint64_t)K * bits) >> 5);
  const uint32_t* row = wq + (size_t)n * words;
  const int groups = K >> lg_group;
  const uint32_t mask = (1u << bits) - 1u;
  float acc[MMAX];
#pragma unroll
  for (int m = 0; m < MMAX; ++m) acc[m] = 0.f;
  for (int k = lane; k < K; k += 32) {
    const uint64_t bit = (uint64_t)bits * (uint64_t)k;
    const uint32_t wi = (uint32_t)(bit >> 5), sh = (uint32_t)(bit & 31u);
    const uint64_t two = (uint64_t)__ldg(row + wi) | (wi + 1 < words ? (uint64_t)__ldg(row + wi + 1) << 32 : 0ull);
    const uint32_t q = (uint32_t)(two >> sh) & mask;
    const int g = k >> lg_group;
    const float wt = fmaf(f16_bits_to_f32(__ldg(scales + (size_t)n * groups + g)), (float)q,
                          f16_bits_to_f32(__ldg(biases + (size_t)n * groups + g)));
#pragma unroll
    for (int m = 0; m < MMAX; ++m)
      if (m < M) acc[m] = fmaf(wt, bf16_bits_to_f32(__ldg(x + (size_t)m * K + k)), acc[m]);
  }
#pragma unroll
  for (int m = 0; m < MMAX; ++m) {
    if (m < M) {
      const float t = warp_sum(acc[m]);
      if (lane == 0) y[(size_t)m * N + n] = t;
    }
  }
}

cudaError_t launch_affine_generic(const uint32_t* wq, int bits, const uint16_t* sc, const uint16_t* bi,
                                  const uint16_t* x, float* y, int M, int N, int K, int group, cudaStream_t stream,
                                  bool pdl) {
  if (group != 32 && group != 64 && group != 128) return cudaErrorInvalidValue;
  if (bits != 2 && bits != 3 && bits != 4 && bits != 5 && bits != 6 && bits != 8) return cudaErrorInvalidValue;
  if (M < 1 || M > 32 || N < 1 || K < 32 || K % 32 || K % group) return cudaErrorInvalidValue;
  const int lg = group == 32 ? 5 : (group == 64 ? 6 : 7);
  const dim3 grid((N + 7) / 8), block(256);
  if (M <= 1)
    return launch_kernel(affine_generic_kernel<1>, grid, block, 0, stream, pdl, wq, bits, sc, bi, x, y, M, N, K, lg);
  if (M <= 4)
    return launch_kernel(affine_generic_kernel<4>, grid, block, 0, stream, pdl, wq, bits, sc, bi, x, y, M, N, K, lg);
  if (M <= 8)
    return launch_kernel(affine_generic_kernel<8>, grid, block, 0, stream, pdl, wq, bits, sc, bi, x, y, M, N, K, lg);
  if (M <= 16)
    return launch_kernel(affine_generic_kernel<16>, grid, block, 0, stream, pdl, wq, bits, sc, bi, x, y, M, N, K,
                         lg);
  return launch_kernel(affine_generic_kernel<32>, grid, block, 0, stream, pdl, wq, bits, sc, bi, x, y, M, N, K, lg);
}

}  // namespace qg
