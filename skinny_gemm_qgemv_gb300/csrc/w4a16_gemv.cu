// W4A16 affine-group GEMV (M = 1, 2) and the generic skinny kernel.
//
// Computes y[m][n] = sum_k (s[n][g] q[n][k] + b[n][g]) x[m][k], g = k / 64, the
// affine 4-bit format of "MLX Runner: An Inference Engine You Can Read",
// section "Architecture: one command buffer per token" (weight = scale x code +
// bias, multiplied against the packed codes with no dequantized copy).
//
// Fast kernel (GB300 design):
//  * Persistent grid, two CTAs per SM. One producer warp streams tiles of R
//    full rows (codes, scales, biases: three contiguous ranges) into a ring of
//    shared-memory stages with cp.async.bulk, completing on mbarriers. The
//    weights are read from HBM exactly once.
//  * Consumer warps own a fixed K-slice: lane l of slice s covers KPL
//    consecutive k, so its activations stay in registers (as bf16 pairs) for
//    the whole kernel. Each stage is consumed with 128-bit shared loads.
//  * Dequant in registers: (word >> 4j) & 0x000F000F | 0x43004300 gives two
//    bf16 values 128 + q (exact); a mixed-precision fma.rn.f32.bf16 multiplies
//    them by the bf16 activations into fp32. Per group of 64 codes the sum is
//    folded as s * (sum (128+q) x - 128 sum x) + b * sum x, the group-factored
//    form of the affine dot product.
//  * Lane partials are reduced with a transposed butterfly; slices of one row
//    are summed in a fixed order through shared memory (deterministic).
#include <cuda_runtime.h>

#include <algorithm>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

// ---------------------------------------------------------------------------
// Fast path
// ---------------------------------------------------------------------------
struct GemvArgs {
  const uint32_t* wq;
  const uint16_t* scales;
  const uint16_t* biases;
  const uint16_t* x;
  float* y;
  int N, K;
  int S;        // K-slices
  int RG;       // row groups (warps per slice)
  int R;        // rows per tile = RG * RPW
  int ST;       // pipeline stages
  int ntiles;
  uint32_t stage_bytes;  // bytes of one stage (codes + scales + biases), 16-aligned
  uint32_t* err;
};

constexpr int kRPW = 2;  // rows per consumer warp per tile

template <int M, int KPL>
__global__ void __launch_bounds__(288, 2) w4a16_gemv_kernel(const GemvArgs a) {
  constexpr int WPL = KPL / 8;  // 32-bit code words per lane per row
  extern __shared__ __align__(128) uint8_t smem[];
  const int NC = a.S * a.RG;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = a.K, N = a.N;
  const uint32_t row_code_bytes = K / 2, row_sb_bytes = K / 32;

  // shared layout: [ST stages][stage_bytes] | red [ST][S][R*M] f32 | barriers
  uint8_t* stages = smem;
  float* red = reinterpret_cast<float*>(smem + (size_t)a.ST * a.stage_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(red + (size_t)a.ST * a.S * a.R * M);
  uint64_t* full = bars;
  uint64_t* empty = bars + a.ST;
  uint64_t* redfull = bars + 2 * a.ST;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NC);
      mbar_init(&redfull[i], NC - a.RG > 0 ? NC - a.RG : 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == NC) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < a.ntiles && ok; tile += gridDim.x, ++it) {
        const int st = it % a.ST;
        if (it >= a.ST) ok = mbar_wait(&empty[st], ((it / a.ST) & 1) ^ 1, a.err, kErrGemvEmptyWait);
        if (!ok) break;
        const int r0 = tile * a.R;
        const int rows = min(a.R, N - r0);
        uint8_t* dst = stages + (size_t)st * a.stage_bytes;
        const uint32_t cb = rows * row_code_bytes, sb = rows * row_sb_bytes;
        mbar_arrive_expect_tx(&full[st], cb + 2 * sb);
        bulk_g2s_evict_first(dst, reinterpret_cast<const uint8_t*>(a.wq) + (size_t)r0 * row_code_bytes, cb,
                             &full[st], pol);
        bulk_g2s(dst + (size_t)a.R * row_code_bytes,
                 reinterpret_cast<const uint8_t*>(a.scales) + (size_t)r0 * row_sb_bytes, sb, &full[st]);
        bulk_g2s(dst + (size_t)a.R * (row_code_bytes + row_sb_bytes),
                 reinterpret_cast<const uint8_t*>(a.biases) + (size_t)r0 * row_sb_bytes, sb, &full[st]);
      }
      // drain: every issued copy must land before this CTA may exit
      const int issued = it;
      for (int j = max(0, issued - a.ST); j < issued; ++j)
        mbar_wait(&full[j % a.ST], (j / a.ST) & 1, a.err, kErrGemvDrain);
    }
    pdl_launch_dependents();
    return;
  }

  // -------------------------------------------------------------- consumers
  const int s = warp % a.S;           // K-slice of this warp
  const int rg = warp / a.S;          // row group
  const int k0 = s * 32 * KPL + lane * KPL;
  const bool active = k0 < K;

  // activations: pairs (k+j, k+j+4) of every word as bf16x2, and sum x
  pdl_wait();
  uint32_t xr[M][WPL][4];
  float sx[M];
#pragma unroll
  for (int m = 0; m < M; ++m) {
    sx[m] = 0.f;
#pragma unroll
    for (int i = 0; i < WPL; ++i) {
      uint4 v = make_uint4(0, 0, 0, 0);
      if (active) v = *reinterpret_cast<const uint4*>(a.x + (size_t)m * K + k0 + 8 * i);
      xr[m][i][0] = __byte_perm(v.x, v.z, 0x5410);
      xr[m][i][1] = __byte_perm(v.x, v.z, 0x7632);
      xr[m][i][2] = __byte_perm(v.y, v.w, 0x5410);
      xr[m][i][3] = __byte_perm(v.y, v.w, 0x7632);
      const uint32_t e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) sx[m] += bf16_bits_to_f32(e[j] & 0xFFFFu) + bf16_bits_to_f32(e[j] >> 16);
    }
  }
  const int g_lane = k0 / 64;  // this lane's group (KPL <= 64 never straddles)

  const uint32_t sbase = smem_u32(stages);
  int it = 0;
  for (int tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x, ++it) {
    const int st = it % a.ST;
    const uint32_t par = (it / a.ST) & 1;
    if (!mbar_wait(&full[st], par, a.err, kErrGemvFullWait)) break;
    const int r0 = tile * a.R;
    const int rows = min(a.R, N - r0);
    const uint32_t stg = sbase + st * a.stage_bytes;

    float part[kRPW][M];
#pragma unroll
    for (int i = 0; i < kRPW; ++i) {
      const int r = rg * kRPW + i;
#pragma unroll
      for (int m = 0; m < M; ++m) part[i][m] = 0.f;
      if (r < rows && active) {
        uint32_t w[WPL];
        const uint32_t caddr = stg + r * row_code_bytes + k0 / 2;
#pragma unroll
        for (int v4 = 0; v4 < WPL / 4; ++v4) {
          uint4 c = lds128(caddr + 16 * v4);
          w[4 * v4 + 0] = c.x;
          w[4 * v4 + 1] = c.y;
          w[4 * v4 + 2] = c.z;
          w[4 * v4 + 3] = c.w;
        }
        const float sc = f16_bits_to_f32(lds16(stg + a.R * row_code_bytes + r * row_sb_bytes + 2 * g_lane));
        const float bi =
            f16_bits_to_f32(lds16(stg + a.R * (row_code_bytes + row_sb_bytes) + r * row_sb_bytes + 2 * g_lane));
        float acc[M][4];
#pragma unroll
        for (int m = 0; m < M; ++m) {
          acc[m][0] = -128.f * sx[m];
          acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
        }
#pragma unroll
        for (int i2 = 0; i2 < WPL; ++i2) {
          uint32_t q[4];
          nib8_to_bf16x2_biased(w[i2], q);
#pragma unroll
          for (int m = 0; m < M; ++m) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              acc[m][j] = fma_bf16_lo_lo(q[j], xr[m][i2][j], acc[m][j]);
              acc[m][j] = fma_bf16_hi_hi(q[j], xr[m][i2][j], acc[m][j]);
            }
          }
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const float t = (acc[m][0] + acc[m][1]) + (acc[m][2] + acc[m][3]);
          part[i][m] = fmaf(sc, t, bi * sx[m]);
        }
      }
    }
    __syncwarp();
    // transposed butterfly over 32 lanes: lanes [16h, 16h+16) end with row h
    float v[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const bool hi = lane & 16;
      float keep = hi ? part[1][m] : part[0][m];
      float send = hi ? part[0][m] : part[1][m];
      keep += __shfl_xor_sync(0xffffffffu, send, 16);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
      v[m] = keep;
    }
    const int myrow = rg * kRPW + (lane >> 4);
    if (a.S == 1) {
      if ((lane & 15) == 0 && myrow < rows) {
#pragma unroll
        for (int m = 0; m < M; ++m) a.y[(size_t)m * N + r0 + myrow] = v[m];
      }
      if (lane == 0) mbar_arrive(&empty[st]);
    } else {
      float* rb = red + (size_t)st * a.S * a.R * M;
      if (s != 0) {
        if ((lane & 15) == 0) {
#pragma unroll
          for (int m = 0; m < M; ++m) rb[(s * a.R + myrow) * M + m] = v[m];
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&redfull[st]);
          mbar_arrive(&empty[st]);
        }
      } else {
        if (!mbar_wait(&redfull[st], par, a.err, kErrGemvFullWait)) break;
        if ((lane & 15) == 0 && myrow < rows) {
#pragma unroll
          for (int m = 0; m < M; ++m) {
            float tot = v[m];
            for (int s2 = 1; s2 < a.S; ++s2) tot += rb[(s2 * a.R + myrow) * M + m];
            a.y[(size_t)m * N + r0 + myrow] = tot;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
    }
  }
  pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// Generic kernel: any M <= 32, any K multiple of 64. One warp per output row;
// plain global loads. Used where the fast path's shape rules do not hold.
// ---------------------------------------------------------------------------
template <int MMAX>
__global__ void __launch_bounds__(256) w4a16_generic_kernel(const uint32_t* __restrict__ wq,
                                                            const uint16_t* __restrict__ scales,
                                                            const uint16_t* __restrict__ biases,
                                                            const uint16_t* __restrict__ x, float* __restrict__ y,
                                                            int M, int N, int K) {
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + warp;
  if (n >= N) return;
  const int words = K / 8, groups = K / 64;
  float acc[MMAX];
#pragma unroll
  for (int m = 0; m < MMAX; ++m) acc[m] = 0.f;
  for (int j = lane; j < words; j += 32) {
    const uint32_t w = wq[(size_t)n * words + j];
    const int g = j / 8;
    const float s = f16_bits_to_f32(scales[(size_t)n * groups + g]);
    const float b = f16_bits_to_f32(biases[(size_t)n * groups + g]);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float wt = fmaf(s, (float)((w >> (4 * i)) & 15u), b);
#pragma unroll
      for (int m = 0; m < MMAX; ++m)
        if (m < M) acc[m] = fmaf(wt, bf16_bits_to_f32(x[(size_t)m * K + 8 * j + i]), acc[m]);
    }
  }
#pragma unroll
  for (int m = 0; m < MMAX; ++m) {
    if (m < M) {
      const float t = warp_sum(acc[m]);
      if (lane == 0) y[(size_t)m * N + n] = t;
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
bool gemv_fast_path_ok(int M, int N, int K) {
  if (M < 1 || M > 2) return false;
  if (K % 1024 != 0) return false;
  const int KPL = (M == 1 && K % 2048 == 0) ? 64 : 32;
  const int S = K / (32 * KPL);
  return S >= 1 && S <= 8 && N >= 1;
}

template <int M, int KPL>
static cudaError_t launch_fast(const uint32_t* wq, const uint16_t* sc, const uint16_t* bi, const uint16_t* x,
                               float* y, int N, int K, uint32_t* err, cudaStream_t stream, bool pdl) {
  GemvArgs a;
  a.wq = wq;
  a.scales = sc;
  a.biases = bi;
  a.x = x;
  a.y = y;
  a.N = N;
  a.K = K;
  a.S = K / (32 * KPL);
  a.RG = std::max(1, 8 / a.S);
  a.R = a.RG * kRPW;
  a.ntiles = (N + a.R - 1) / a.R;
  const uint32_t row_bytes = K / 2 + K / 16;
  a.stage_bytes = (uint32_t)a.R * row_bytes;  // multiple of 16 since K % 512 == 0
  const int NC = a.S * a.RG;
  // two CTAs per SM: keep each CTA's shared memory under ~110 KB
  const size_t budget = 110 * 1024;
  int ST = (int)(budget / (a.stage_bytes + sizeof(float) * a.S * a.R * M + 24));
  ST = std::max(2, std::min(ST, 8));
  a.ST = ST;
  a.err = err;
  const size_t smem = (size_t)ST * a.stage_bytes + sizeof(float) * (size_t)ST * a.S * a.R * M + 3 * 8 * ST;
  static_assert(sizeof(GemvArgs) < 4096, "kernel params");

  auto kern = w4a16_gemv_kernel<M, KPL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = std::min(a.ntiles, 2 * sms);
  return launch_kernel(kern, dim3(grid), dim3((NC + 1) * 32), smem, stream, pdl, a);
}

cudaError_t launch_w4a16_fast(const uint32_t* wq, const uint16_t* sc, const uint16_t* bi, const uint16_t* x,
                              float* y, int M, int N, int K, uint32_t* err, cudaStream_t stream, bool pdl) {
  if (M == 1) {
    if (K % 2048 == 0) return launch_fast<1, 64>(wq, sc, bi, x, y, N, K, err, stream, pdl);
    return launch_fast<1, 32>(wq, sc, bi, x, y, N, K, err, stream, pdl);
  }
  return launch_fast<2, 32>(wq, sc, bi, x, y, N, K, err, stream, pdl);
}

cudaError_t launch_w4a16_generic(const uint32_t* wq, const uint16_t* sc, const uint16_t* bi, const uint16_t* x,
                                 float* y, int M, int N, int K, cudaStream_t stream, bool pdl) {
  dim3 grid((N + 7) / 8), block(256);
  if (M <= 1) return launch_kernel(w4a16_generic_kernel<1>, grid, block, 0, stream, pdl, wq, sc, bi, x, y, M, N, K);
  if (M <= 4) return launch_kernel(w4a16_generic_kernel<4>, grid, block, 0, stream, pdl, wq, sc, bi, x, y, M, N, K);
  if (M <= 8) return launch_kernel(w4a16_generic_kernel<8>, grid, block, 0, stream, pdl, wq, sc, bi, x, y, M, N, K);
  if (M <= 16)
    return launch_kernel(w4a16_generic_kernel<16>, grid, block, 0, stream, pdl, wq, sc, bi, x, y, M, N, K);
  return launch_kernel(w4a16_generic_kernel<32>, grid, block, 0, stream, pdl, wq, sc, bi, x, y, M, N, K);
}

}  // namespace qg
