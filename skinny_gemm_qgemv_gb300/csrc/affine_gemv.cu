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
// Up to 4 activation rows take the chunked kernels instead: lane l of a warp
// takes whole 32-code chunks (BITS consecutive words: exactly 32 codes, so a
// chunk never shares a word with the next one, and a warp reads 32 BITS words
// contiguously), four at a time with their loads issued first, and folds the
// affine group per chunk as s * sum(q x) + b * sum(x). At 2, 4 and 8 bits
// (affine_f16_kernel) codes become fp16 1024 + q 2^(j BITS) two at a time and
// meet fp16 activations prepared once per CTA; at 3, 5 and 6 bits
// (affine_fast_kernel) each code is extracted with constant shifts (a funnel
// shift where it spans two words) and converted to fp32.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

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

// One warp per output row at a time, 8 rows per CTA and pass; MM >= M
// activation rows.
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
  const int groups = K >> lg_group, gpc = lg_group - 5;  // chunks per group: 2^gpc
  for (int n = blockIdx.x * 8 + warp; n < N; n += gridDim.x * 8) {
    const uint32_t* row = wq + (size_t)n * nch * BITS;
    float acc[MM];
#pragma unroll
    for (int m = 0; m < MM; ++m) acc[m] = 0.f;
    // kU chunks a lane at a time, their weight words and factors loaded first
    constexpr int kU = 4;
    for (int c0 = lane; c0 < nch; c0 += 32 * kU) {
      uint32_t wv[kU][BITS + 1];
      uint16_t sv[kU], bv[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int c = c0 + 32 * u;
        if (c < nch) {
          load_chunk<BITS>(row + (size_t)BITS * c, wv[u]);
          sv[u] = __ldg(scales + (size_t)n * groups + (c >> gpc));
          bv[u] = __ldg(biases + (size_t)n * groups + (c >> gpc));
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int c = c0 + 32 * u;
        if (c >= nch) break;
        uint32_t xv[MM][16];
#pragma unroll
        for (int m = 0; m < MM; ++m) {
          const uint4* xp = reinterpret_cast<const uint4*>(x + (size_t)(m < M ? m : 0) * K + 32 * c);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint4 q4 = __ldg(xp + v);
            xv[m][4 * v] = q4.x, xv[m][4 * v + 1] = q4.y, xv[m][4 * v + 2] = q4.z, xv[m][4 * v + 3] = q4.w;
          }
        }
        float dot[MM];
#pragma unroll
        for (int m = 0; m < MM; ++m) dot[m] = 0.f;
        ChunkDot<BITS, MM, 0>::run(wv[u], xv, dot);
        const float sc = f16_bits_to_f32(sv[u]), bi = f16_bits_to_f32(bv[u]);
#pragma unroll
        for (int m = 0; m < MM; ++m)
          if (m < M) acc[m] = fmaf(sc, dot[m], fmaf(bi, sxs[m * nch + c], acc[m]));
      }
    }
#pragma unroll
    for (int m = 0; m < MM; ++m) {
      if (m < M) {
        const float t = warp_sum(acc[m]);
        if (lane == 0) y[(size_t)m * N + n] = t;
      }
    }
  }
}

// 2, 4 and 8 bits: the codes of a byte are classes j = 0 .. 8 / BITS - 1 (bits
// j BITS .. j BITS + BITS - 1); one lop3 per class turns bytes 0 and 2 of a
// word (then, on w >> 8, bytes 1 and 3) into two fp16 values 1024 + q 2^(j BITS)
// (exact: below 2048), so a word costs a shift and 2 (8 / BITS) lop3s for its
// 32 / BITS codes, and each code one mixed-precision FMA with its activation in
// fp16. Per chunk and activation row the CTA prepares once, in shared memory,
// the activations x 2^-(sigma + j BITS) in fp16 (sigma: the chunk's largest |x|
// just below 2^15; exact for bf16 x) in the order of those registers, and
// (2^sigma, 1024 times the sum of those fp16 values, sum x); the chunk then
// adds s 2^sigma (acc - offset) + b sum x. Products exact, fp32 sums.
template <int BITS>
__device__ __forceinline__ void chunk_regs(const uint32_t (&w)[BITS + 1], uint32_t (&r)[16]) {
  constexpr int J = 8 / BITS;  // classes per byte
  constexpr uint32_t kMagic = 0x64006400u;
#pragma unroll
  for (int i = 0; i < BITS; ++i) {
    const uint32_t t = w[i] >> 8;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      constexpr uint32_t m8 = (1u << BITS) - 1u;
      const uint32_t mask = (m8 << (j * BITS)) * 0x00010001u;
      asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r[(2 * i) * J + j]) : "r"(w[i]), "r"(mask), "r"(kMagic));
      asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r[(2 * i + 1) * J + j]) : "r"(t), "r"(mask), "r"(kMagic));
    }
  }
}

// code of chunk position k (0..31) in register r = (2 i + s) J + j: word i,
// byte s (low half) or s + 2 (high half), class j
template <int BITS>
__device__ __forceinline__ int reg_code(int r, int hi) {
  constexpr int J = 8 / BITS;
  const int i = r / (2 * J), s = (r / J) & 1, j = r % J;
  return i * (32 / BITS) + (s + 2 * hi) * J + j;
}

template <int BITS, int MM>
__global__ void __launch_bounds__(256) affine_f16_kernel(const uint32_t* __restrict__ wq,
                                                         const uint16_t* __restrict__ scales,
                                                         const uint16_t* __restrict__ biases,
                                                         const uint16_t* __restrict__ x, float* __restrict__ y,
                                                         int M, int N, int K, int lg_group) {
  // shared: activations [M][4][nch][4 words] (16-byte slices v of each chunk's
  // 16 registers, lanes reading consecutive chunks hit consecutive 16 bytes),
  // then per (row, chunk) {2^sigma, offset, sum x, 0}
  extern __shared__ __align__(16) uint32_t xs[];
  pdl_wait();
  const int nch = K >> 5;
  float4* po = reinterpret_cast<float4*>(xs + (size_t)M * nch * 16);
  for (int it = threadIdx.x; it < M * nch; it += blockDim.x) {
    const int m = it / nch, c = it - m * nch;
    const uint4* xp = reinterpret_cast<const uint4*>(x + (size_t)m * K + 32 * c);
    float v[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = __ldg(xp + q);
      const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        v[8 * q + 2 * h] = __uint_as_float(uu[h] << 16);
        v[8 * q + 2 * h + 1] = __uint_as_float(uu[h] & 0xFFFF0000u);
      }
    }
    float amax = 0.f, sx = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      amax = fmaxf(amax, fabsf(v[k]));
      sx += v[k];
    }
    const int sig = fp16_prescale_exp(amax);
    float off = 0.f;
    uint32_t reg[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const float sc = pow2f(-sig - (r % (8 / BITS)) * BITS);
      const __half2 h2 = __floats2half2_rn(v[reg_code<BITS>(r, 0)] * sc, v[reg_code<BITS>(r, 1)] * sc);
      reg[r] = *reinterpret_cast<const uint32_t*>(&h2);
      const float2 back = __half22float2(h2);
      off += back.x + back.y;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
      reinterpret_cast<uint4*>(xs)[((size_t)m * 4 + q) * nch + c] =
          make_uint4(reg[4 * q], reg[4 * q + 1], reg[4 * q + 2], reg[4 * q + 3]);
    po[it] = make_float4(pow2f(sig), 1024.f * off, sx, 0.f);
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int groups = K >> lg_group, gpc = lg_group - 5;
  for (int n = blockIdx.x * 8 + warp; n < N; n += gridDim.x * 8) {
    const uint32_t* row = wq + (size_t)n * nch * BITS;
    float acc[MM];
#pragma unroll
    for (int m = 0; m < MM; ++m) acc[m] = 0.f;
    // kU chunks a lane at a time, every load issued first: more weight bytes in
    // flight per warp (one chunk at a time left the loads latency-bound)
    constexpr int kU = 4;
    for (int c0 = lane; c0 < nch; c0 += 32 * kU) {
      uint32_t wv[kU][BITS + 1];
      uint16_t sv[kU], bv[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int c = c0 + 32 * u;
        if (c < nch) {
          load_chunk<BITS>(row + (size_t)BITS * c, wv[u]);
          sv[u] = __ldg(scales + (size_t)n * groups + (c >> gpc));
          bv[u] = __ldg(biases + (size_t)n * groups + (c >> gpc));
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int c = c0 + 32 * u;
        if (c >= nch) break;
        uint32_t r[16];
        chunk_regs<BITS>(wv[u], r);
        const float sc = f16_bits_to_f32(sv[u]);
        const float bi = f16_bits_to_f32(bv[u]);
#pragma unroll
        for (int m = 0; m < MM; ++m) {
          if (m < M) {
            uint32_t xv[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 u4 = reinterpret_cast<const uint4*>(xs)[((size_t)m * 4 + q) * nch + c];
              xv[4 * q] = u4.x, xv[4 * q + 1] = u4.y, xv[4 * q + 2] = u4.z, xv[4 * q + 3] = u4.w;
            }
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              a0 = fma_f16_lo_lo(r[k], xv[k], a0);
              a1 = fma_f16_hi_hi(r[k], xv[k], a1);
            }
            const float4 p = po[m * nch + c];
            acc[m] = fmaf(sc * p.x, (a0 + a1) - p.y, fmaf(bi, p.z, acc[m]));
          }
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MM; ++m) {
      if (m < M) {
        const float t = warp_sum(acc[m]);
        if (lane == 0) y[(size_t)m * N + n] = t;
      }
    }
  }
}

namespace {

// shared memory a CTA of the chunked kernels needs
size_t affine_fast_smem(int bits, int M, int K) {
  const size_t per = (bits == 2 || bits == 4 || bits == 8) ? 64 + 16 : 4;
  return per * (size_t)M * (K / 32);
}

template <int BITS>
cudaError_t launch_affine_fast_bits(const uint32_t* wq, const uint16_t* sc, const uint16_t* bi, const uint16_t* x,
                                    float* y, int M, int N, int K, int lg, cudaStream_t stream, bool pdl) {
  // persistent rows (at most 8 CTAs per SM): the activations are prepared
  // once per CTA
  const dim3 block(256);
  const size_t smem = affine_fast_smem(BITS, M, K);
  if constexpr (BITS == 2 || BITS == 4 || BITS == 8) {
    const dim3 grid((unsigned)std::min<long long>((N + 7) / 8, 8LL * device_sm_count()));
    if (M <= 1)
      return launch_kernel(affine_f16_kernel<BITS, 1>, grid, block, smem, stream, pdl, wq, sc, bi, x, y, M, N, K, lg);
    return launch_kernel(affine_f16_kernel<BITS, 4>, grid, block, smem, stream, pdl, wq, sc, bi, x, y, M, N, K, lg);
  } else {
    const dim3 grid((unsigned)std::min<long long>((N + 7) / 8, 8LL * device_sm_count()));
    if (M <= 1)
      return launch_kernel(affine_fast_kernel<BITS, 1>, grid, block, smem, stream, pdl, wq, sc, bi, x, y, M, N, K,
                           lg);
    return launch_kernel(affine_fast_kernel<BITS, 4>, grid, block, smem, stream, pdl, wq, sc, bi, x, y, M, N, K, lg);
  }
}

}  // namespace

// 2 / 3 / 4 / 5 / 6 / 8-bit codes, groups 32 / 64 / 128, 1 <= M <= 4, K a
// multiple of 32 and of the group, the chunk sums of x within 48 KB of shared
// memory; 16-byte aligned pointers
bool affine_fast_ok(int bits, int M, int K, int group) {
  return (bits == 2 || bits == 3 || bits == 4 || bits == 5 || bits == 6 || bits == 8) && M >= 1 && M <= 4 &&
         (group == 32 || group == 64 || group == 128) && K >= 32 && K % 32 == 0 && K % group == 0 &&
         affine_fast_smem(bits, M, K) <= 48 * 1024;
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
