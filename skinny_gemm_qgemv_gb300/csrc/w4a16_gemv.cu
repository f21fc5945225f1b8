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
#include <cuda_fp16.h>
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

template <int M, int KPL, int kRPW, int MINB>
__global__ void __launch_bounds__(288, MINB) w4a16_gemv_kernel(const GemvArgs a) {
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
  pdl_launch_dependents();

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
    return;
  }

  // -------------------------------------------------------------- consumers
  const int s = warp % a.S;           // K-slice of this warp
  const int rg = warp / a.S;          // row group
  const int k0 = s * 32 * KPL + lane * KPL;
  const bool active = k0 < K;

  // activations: fp16 pairs (k+j, k+j+4) of every word, scaled by 2^-sigma
  // (the lane's largest |x| just below 2^15; exact), the sum of x, and the
  // offset sums -1024 X_A, -1024 X_B of the scaled values of each code class
  pdl_wait();
  uint32_t xr[M][WPL][4];
  float sx[M], up[M], acc0a[M], acc0b[M];
#pragma unroll
  for (int m = 0; m < M; ++m) {
    sx[m] = 0.f;
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < WPL; ++i) {
      uint4 v = make_uint4(0, 0, 0, 0);
      if (active) v = *reinterpret_cast<const uint4*>(a.x + (size_t)m * K + k0 + 8 * i);
      xr[m][i][0] = v.x;
      xr[m][i][1] = v.y;
      xr[m][i][2] = v.z;
      xr[m][i][3] = v.w;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float lo = bf16_bits_to_f32(xr[m][i][j] & 0xFFFFu), hi = bf16_bits_to_f32(xr[m][i][j] >> 16);
        sx[m] += lo + hi;
        amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
      }
    }
    const int sig = fp16_prescale_exp(amax);
    const float down = pow2f(-sig);
    up[m] = pow2f(sig);
    float sxa = 0.f, sxb = 0.f;
#pragma unroll
    for (int i = 0; i < WPL; ++i) {
      float xv[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        xv[2 * j] = bf16_bits_to_f32(xr[m][i][j] & 0xFFFFu) * down;
        xv[2 * j + 1] = bf16_bits_to_f32(xr[m][i][j] >> 16) * down;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 h2 = __floats2half2_rn(xv[j], xv[j + 4]);
        xr[m][i][j] = *reinterpret_cast<const uint32_t*>(&h2);
        const float2 back = __half22float2(h2);
        if (j % 2 == 0) sxa += back.x + back.y; else sxb += back.x + back.y;
      }
    }
    acc0a[m] = -1024.f * sxa;
    acc0b[m] = -1024.f * sxb;
  }
  const int g_lane = k0 / 64;  // this lane's group (KPL <= 64 never straddles)

  const uint32_t sbase = smem_u32(stages);
  int st = 0;
  uint32_t par = 0;
  for (int tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
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
        // acc[m][0], [1]: the (1024 + q) class, [2], [3]: the (1024 + 16 q) class
        float acc[M][4];
#pragma unroll
        for (int m = 0; m < M; ++m) {
          acc[m][0] = acc0a[m];
          acc[m][2] = acc0b[m];
          acc[m][1] = acc[m][3] = 0.f;
        }
#pragma unroll
        for (int i2 = 0; i2 < WPL; ++i2) {
          uint32_t q[4];
          nib8_to_f16x2_offset(w[i2], q);
#pragma unroll
          for (int m = 0; m < M; ++m) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int c = (j & 1) * 2;
              acc[m][c] = fma_f16_lo_lo(q[j], xr[m][i2][j], acc[m][c]);
              acc[m][c + 1] = fma_f16_hi_hi(q[j], xr[m][i2][j], acc[m][c + 1]);
            }
          }
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const float t = (acc[m][0] + acc[m][1]) + 0.0625f * (acc[m][2] + acc[m][3]);
          part[i][m] = fmaf(sc * up[m], t, bi * sx[m]);
        }
      }
    }
    __syncwarp();
    float v[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float col[kRPW];
#pragma unroll
      for (int i = 0; i < kRPW; ++i) col[i] = part[i][m];
      v[m] = transposed_warp_sum<kRPW>(col, lane);
    }
    constexpr int kLanesPerRow = 32 / kRPW;
    const bool writer = (lane & (kLanesPerRow - 1)) == 0;
    const int myrow = rg * kRPW + transposed_row<kRPW>(lane);
    if (a.S == 1) {
      if (writer && myrow < rows) {
#pragma unroll
        for (int m = 0; m < M; ++m) a.y[(size_t)m * N + r0 + myrow] = v[m];
      }
      if (lane == 0) mbar_arrive(&empty[st]);
    } else {
      float* rb = red + (size_t)st * a.S * a.R * M;
      if (s != 0) {
        if (writer) {
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
        if (writer && myrow < rows) {
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
    if (++st == a.ST) {
      st = 0;
      par ^= 1u;
    }
  }
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
                                                            int M, int N, int K, int lg_group) {
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + warp;
  if (n >= N) return;
  const int words = K / 8, groups = K >> lg_group;  // group = 2^lg_group codes (32, 64 or 128)
  float acc[MMAX];
#pragma unroll
  for (int m = 0; m < MMAX; ++m) acc[m] = 0.f;
  for (int j = lane; j < words; j += 32) {
    const uint32_t w = wq[(size_t)n * words + j];
    const int g = (8 * j) >> lg_group;
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
  if (M < 1 || M > 2 || N < 1 || K % 1024 != 0) return false;
  // at most eight consumer warps cover one row (S <= 8)
  const int slices = (M == 1 && K % 2048 == 0) ? K / 2048 : K / 1024;
  return slices <= 8;
}

// Shape -> launch configuration of the fast kernel. Lanes cover KPL
// consecutive k, so one warp covers a K-slice of 32 * KPL and S = K / (32 KPL)
// warps cover a row; RG row groups of RPW rows each make a tile of R = RG * RPW
// rows. More rows per warp amortize the lane reduction and give independent
// FMA chains; small N trade rows per warp for enough tiles to fill the SMs.
GemvConfig gemv_pick_config(int M, int N, int K, int sms) {
  // Chosen from a sweep on GB300 (152 SMs) over the decode shapes: two CTAs of
  // at most nine warps per SM; 64 k per lane and 4 rows per warp for very
  // tall matrices and for K = 12288 (fewer K-slices per row), otherwise 32 k
  // per lane and up to 8 rows per warp, reduced until every CTA slot has a tile.
  GemvConfig c;
  const bool tall = N >= 65536;
  c.kpl = (M == 1 && K % 2048 == 0 && (tall || K / 1024 > 8)) ? 64 : 32;
  const int S = K / (32 * c.kpl);
  c.rg = S >= 8 ? 1 : 8 / S;
  c.ctas_per_sm = 2;
  c.smem_budget = 74 * 1024;
  c.rpw = (M == 1 && c.kpl == 32) ? 8 : 4;
  while (c.rpw > 2 && (N + c.rg * c.rpw - 1) / (c.rg * c.rpw) < c.ctas_per_sm * sms) c.rpw /= 2;
  while (c.rg > 1 && (N + c.rg * c.rpw - 1) / (c.rg * c.rpw) < c.ctas_per_sm * sms) c.rg /= 2;
  return c;
}

template <int M, int KPL, int RPW, int MINB>
static cudaError_t launch_fast(const uint32_t* wq, const uint16_t* sc, const uint16_t* bi, const uint16_t* x,
                               float* y, int N, int K, const GemvConfig& cfg, uint32_t* err, cudaStream_t stream,
                               bool pdl) {
  GemvArgs a;
  a.wq = wq;
  a.scales = sc;
  a.biases = bi;
  a.x = x;
  a.y = y;
  a.N = N;
  a.K = K;
  a.S = K / (32 * KPL);
  a.RG = cfg.rg;
  a.R = a.RG * RPW;
  a.ntiles = (N + a.R - 1) / a.R;
  const uint32_t row_bytes = K / 2 + K / 16;
  a.stage_bytes = (uint32_t)a.R * row_bytes;  // multiple of 16 since K % 512 == 0
  const int NC = a.S * a.RG;
  if ((NC + 1) * 32 > 288) return cudaErrorInvalidConfiguration;
  int ST = (int)(cfg.smem_budget / (a.stage_bytes + sizeof(float) * a.S * a.R * M + 24));
  ST = std::max(2, std::min(ST, 8));
  a.ST = ST;
  a.err = err;
  const size_t smem = (size_t)ST * a.stage_bytes + sizeof(float) * (size_t)ST * a.S * a.R * M + 3 * 8 * ST;
  auto kern = w4a16_gemv_kernel<M, KPL, RPW, MINB>;
  cudaError_t e = allow_max_smem(kern);
  if (e != cudaSuccess) return e;
  const int grid = std::min(a.ntiles, cfg.ctas_per_sm * device_sm_count());
  return launch_kernel(kern, dim3(grid), dim3((NC + 1) * 32), smem, stream, pdl, a);
}

template <int M, int KPL>
static cudaError_t launch_rpw(const uint32_t* wq, const uint16_t* sc, const uint16_t* bi, const uint16_t* x,
                              float* y, int N, int K, const GemvConfig& cfg, uint32_t* err, cudaStream_t stream,
                              bool pdl) {
  // MINB (CTAs per SM the register allocation is sized for) follows ctas_per_sm
#define QG_RPW_CASE(R)                                                                              \
  case R:                                                                                           \
    if (cfg.ctas_per_sm >= 4) return launch_fast<M, KPL, R, 4>(wq, sc, bi, x, y, N, K, cfg, err, stream, pdl); \
    if (cfg.ctas_per_sm == 3) return launch_fast<M, KPL, R, 3>(wq, sc, bi, x, y, N, K, cfg, err, stream, pdl); \
    return launch_fast<M, KPL, R, 2>(wq, sc, bi, x, y, N, K, cfg, err, stream, pdl);
  switch (cfg.rpw) {
    QG_RPW_CASE(2)
    QG_RPW_CASE(4)
    QG_RPW_CASE(8)
    default: return cudaErrorInvalidValue;
  }
#undef QG_RPW_CASE
}

cudaError_t launch_w4a16_fast_cfg(const uint32_t* wq, const uint16_t* sc, const uint16_t* bi, const uint16_t* x,
                                  float* y, int M, int N, int K, const GemvConfig& cfg, uint32_t* err,
                                  cudaStream_t stream, bool pdl) {
  if (K % (32 * cfg.kpl) != 0) return cudaErrorInvalidValue;
  if (M == 1) {
    if (cfg.kpl == 64) return launch_rpw<1, 64>(wq, sc, bi, x, y, N, K, cfg, err, stream, pdl);
    return launch_rpw<1, 32>(wq, sc, bi, x, y, N, K, cfg, err, stream, pdl);
  }
  if (cfg.kpl != 32) return cudaErrorInvalidValue;
  return launch_rpw<2, 32>(wq, sc, bi, x, y, N, K, cfg, err, stream, pdl);
}

cudaError_t launch_w4a16_fast(const uint32_t* wq, const uint16_t* sc, const uint16_t* bi, const uint16_t* x,
                              float* y, int M, int N, int K, uint32_t* err, cudaStream_t stream, bool pdl) {
  const GemvConfig cfg = gemv_pick_config(M, N, K, device_sm_count());
  return launch_w4a16_fast_cfg(wq, sc, bi, x, y, M, N, K, cfg, err, stream, pdl);
}

cudaError_t launch_w4a16_generic(const uint32_t* wq, const uint16_t* sc, const uint16_t* bi, const uint16_t* x,
                                 float* y, int M, int N, int K, int group, cudaStream_t stream, bool pdl) {
  if (group != 32 && group != 64 && group != 128) return cudaErrorInvalidValue;
  const int lg = group == 32 ? 5 : (group == 64 ? 6 : 7);
  dim3 grid((N + 7) / 8), block(256);
  if (M <= 1)
    return launch_kernel(w4a16_generic_kernel<1>, grid, block, 0, stream, pdl, wq, sc, bi, x, y, M, N, K, lg);
  if (M <= 4)
    return launch_kernel(w4a16_generic_kernel<4>, grid, block, 0, stream, pdl, wq, sc, bi, x, y, M, N, K, lg);
  if (M <= 8)
    return launch_kernel(w4a16_generic_kernel<8>, grid, block, 0, stream, pdl, wq, sc, bi, x, y, M, N, K, lg);
  if (M <= 16)
    return launch_kernel(w4a16_generic_kernel<16>, grid, block, 0, stream, pdl, wq, sc, bi, x, y, M, N, K, lg);
  return launch_kernel(w4a16_generic_kernel<32>, grid, block, 0, stream, pdl, wq, sc, bi, x, y, M, N, K, lg);
}

}  // namespace qg
