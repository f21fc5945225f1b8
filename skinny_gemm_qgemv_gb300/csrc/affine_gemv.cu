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
//
// Up to 4 activation rows take affine_fast_kernel instead: lane l of a warp
// takes whole 32-code chunks (BITS consecutive words: exactly 32 codes, so a
// chunk never shares a word with the next one, and a warp reads 32 BITS words
// contiguously), extracts the codes with constant shifts (a funnel shift where
// a code spans two words), and folds the affine group per chunk as
// s * sum(q x) + b * sum(x), the chunk sums of x computed once per CTA.
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

namespace {

// the BITS words of 32-code chunk c of a row (little-endian bit stream)
template <int BITS>
__device__ __forceinline__ void load_chunk(const uint32_t* __restrict__ p, uint32_t (&w)[BITS + 1]) {
  if (BITS == 2) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
    w[0] = v.x, w[1] = v.y;
  } else if (BITS == 4) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
  } else if (BITS == 8) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p)), u = __ldg(reinterpret_cast<const uint4*>(p) + 1);
    w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w, w[4] = u.x, w[5] = u.y, w[6] = u.z, w[7] = u.w;
  } else if (BITS == 6) {
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(p) + i);
      w[2 * i] = v.x, w[2 * i + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < BITS; ++i) w[i] = __ldg(p + i);
  }
  w[BITS] = 0u;
}

// code j of a chunk (compile-time position)
template <int BITS, int J>
__device__ __forceinline__ uint32_t chunk_code(const uint32_t (&w)[BITS + 1]) {
  constexpr int bit = BITS * J, wi = bit >> 5, sh = bit & 31;
  constexpr uint32_t mask = (1u << BITS) - 1u;
  if (sh + BITS <= 32) return (w[wi] >> sh) & mask;
  return __funnelshift_r(w[wi], w[wi + 1], sh) & mask;
}

template <int BITS, int MM, int J>
struct ChunkDot {
  __device__ __forceinline__ static void run(const uint32_t (&w)[BITS + 1], const uint32_t (&xv)[MM][16],
                                             float (&dot)[MM]) {
    const float q = (float)chunk_code<BITS, J>(w);
#pragma unroll
    for (int m = 0; m < MM; ++m) {
      const uint32_t u = xv[m][J >> 1];
      const float xf = __uint_as_float((J & 1) ? (u & 0xFFFF0000u) : (u << 16));  // bf16 -> fp32
      dot[m] = fmaf(q, xf, dot[m]);
    }
    ChunkDot<BITS, MM, J + 1>::run(w, xv, dot);
  }
};
template <int BITS, int MM>
struct ChunkDot<BITS, MM, 32> {
  __device__ __forceinline__ static void run(const uint32_t (&)[BITS + 1], const uint32_t (&)[MM][16], float (&)[MM]) {}
};

}  // namespace

// One warp per output row, 8 rows per CTA; MM >= M activation rows.
template <int BITS, int MM>
__global__ void __launch_bounds__(256) affine_fast_kernel(const uint32_t* __restrict__ wq,
                                                          const uint16_t* __restrict__ scales,
                                                          const uint16_t* __restrict__ biases,
                                                          const uint16_t* __restrict__ x, float* __restrict__ y,
                                                          int M, int N, int K, int lg_group) {
  extern __shared__ float sxs[];  // [M][K / 32]: the sum of x over each 32-code chunk
  pdl_wait();
  const int nch = K >> 5;
  for (int i = threadIdx.x; i < M * nch; i += blockDim.x) {
    const int m = i / nch, c = i - m * nch;
    const uint4* xp = reinterpret_cast<const uint4*>(x + (size_t)m * K + 32 * c);
    float t = 0.f;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 u = __ldg(xp + v);
      const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) t += __uint_as_float(uu[j] << 16) + __uint_as_float(uu[j] & 0xFFFF0000u);
    }
    sxs[i] = t;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + warp;
  if (n >= N) return;
  const uint32_t* row = wq + (size_t)n * nch * BITS;
  const int groups = K >> lg_group, gpc = lg_group - 5;  // chunks per group: 2^gpc
  float acc[MM];
#pragma unroll
  for (int m = 0; m < MM; ++m) acc[m] = 0.f;
  for (int c = lane; c < nch; c += 32) {
    uint32_t w[BITS + 1];
    load_chunk<BITS>(row + (size_t)BITS * c, w);
    uint32_t xv[MM][16];
#pragma unroll
    for (int m = 0; m < MM; ++m) {
      const uint4* xp = reinterpret_cast<const uint4*>(x + (size_t)(m < M ? m : 0) * K + 32 * c);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint4 u = __ldg(xp + v);
        xv[m][4 * v] = u.x, xv[m][4 * v + 1] = u.y, xv[m][4 * v + 2] = u.z, xv[m][4 * v + 3] = u.w;
      }
    }
    const int g = c >> gpc;
    const float sc = f16_bits_to_f32(__ldg(scales + (size_t)n * groups + g));
    const float bi = f16_bits_to_f32(__ldg(biases + (size_t)n * groups + g));
    float dot[MM];
#pragma unroll
    for (int m = 0; m < MM; ++m) dot[m] = 0.f;
    ChunkDot<BITS, MM, 0>::run(w, xv, dot);
#pragma unroll
    for (int m = 0; m < MM; ++m)
      if (m < M) acc[m] = fmaf(sc, dot[m], fmaf(bi, sxs[m * nch + c], acc[m]));
  }
#pragma unroll
  for (int m = 0; m < MM; ++m) {
    if (m < M) {
      const float t = warp_sum(acc[m]);
      if (lane == 0) y[(size_t)m * N + n] = t;
    }
  }
}

namespace {

template <int BITS>
cudaError_t launch_affine_fast_bits(const uint32_t* wq, const uint16_t* sc, const uint16_t* bi, const uint16_t* x,
                                    float* y, int M, int N, int K, int lg, cudaStream_t stream, bool pdl) {
  const dim3 grid((N + 7) / 8), block(256);
  const size_t smem = sizeof(float) * (size_t)M * (K / 32);
  if (M <= 1)
    return launch_kernel(affine_fast_kernel<BITS, 1>, grid, block, smem, stream, pdl, wq, sc, bi, x, y, M, N, K, lg);
  return launch_kernel(affine_fast_kernel<BITS, 4>, grid, block, smem, stream, pdl, wq, sc, bi, x, y, M, N, K, lg);
}

}  // namespace

// 2 / 3 / 4 / 5 / 6 / 8-bit codes, groups 32 / 64 / 128, 1 <= M <= 4, K a
// multiple of 32 and of the group, the chunk sums of x within 48 KB of shared
// memory; 16-byte aligned pointers
bool affine_fast_ok(int bits, int M, int K, int group) {
  return (bits == 2 || bits == 3 || bits == 4 || bits == 5 || bits == 6 || bits == 8) && M >= 1 && M <= 4 &&
         (group == 32 || group == 64 || group == 128) && K >= 32 && K % 32 == 0 && K % group == 0 &&
         sizeof(float) * (size_t)M * (K / 32) <= 48 * 1024;
}

cudaError_t launch_affine_fast(const uint32_t* wq, int bits, const uint16_t* sc, const uint16_t* bi,
                               const uint16_t* x, float* y, int M, int N, int K, int group, cudaStream_t stream,
                               bool pdl) {
  if (!affine_fast_ok(bits, M, K, group) || N < 1) return cudaErrorInvalidValue;
  const int lg = group == 32 ? 5 : (group == 64 ? 6 : 7);
  switch (bits) {
    case 2: return launch_affine_fast_bits<2>(wq, sc, bi, x, y, M, N, K, lg, stream, pdl);
    case 3: return launch_affine_fast_bits<3>(wq, sc, bi, x, y, M, N, K, lg, stream, pdl);
    case 4: return launch_affine_fast_bits<4>(wq, sc, bi, x, y, M, N, K, lg, stream, pdl);
    case 5: return launch_affine_fast_bits<5>(wq, sc, bi, x, y, M, N, K, lg, stream, pdl);
    case 6: return launch_affine_fast_bits<6>(wq, sc, bi, x, y, M, N, K, lg, stream, pdl);
    default: return launch_affine_fast_bits<8>(wq, sc, bi, x, y, M, N, K, lg, stream, pdl);
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
