// Grouped W4A16 GEMV: many independent projections in one persistent launch.
//
// Each projection is y = W x with the affine 4-bit groups of "MLX Runner: An
// Inference Engine You Can Read", section "Architecture: one command buffer
// per token" (weight = scale x code + bias). That section issues the work of a
// whole token as one command buffer; on GB300 the same idea becomes one
// persistent kernel that walks the projections' row tiles back to back, so
// the HBM stream never drains between projections (no per-launch ramp-up or
// tail).
//
// Design (same per-tile arithmetic as the M = 1 kernel in w4a16_gemv.cu):
//  * The row tiles of all projections form one list; the host splits it into
//    one contiguous range per CTA with equal cost (two CTAs per SM; a tile's
//    cost is its bytes over the fraction of consumer warps it keeps busy). A CTA's
//    producer warp streams its range (codes, scales, biases of R whole rows,
//    three contiguous byte ranges) with cp.async.bulk into a ring of shared
//    memory stages; the HBM addresses of a CTA are sequential.
//  * Twelve consumer warps: lane l of K-slice s covers 64 consecutive k, so a
//    projection with K = 2048 S uses S slices and 12 / S row groups of 4 rows
//    (every tile then holds 96 K-rows' worth of codes, 55 KB).
//    When the range crosses into the next projection the consumers reload
//    their activations (x is small and stays in L2).
//  * Dequant and fold: a lane keeps its 64 activations in fp16, scaled by a
//    power of two 2^-sigma that puts the lane's largest |x| just below 2^15
//    (exact: bf16 has 8 significant bits, fp16 11). Each code word gives four
//    fp16x2 registers with one shift and four lop3s: (w & 0x000F000F) |
//    0x64006400 is (1024 + q) for the codes in bits 0-3 of each half and
//    (w & 0x00F000F0) | 0x64006400 is (1024 + 16 q) for bits 4-7, the same on
//    w >> 8 for the other two; fma.rn.f32.f16 multiplies them (exact products)
//    into fp32 sums A (1024 + q terms) and B (1024 + 16 q terms), and per lane
//    s * 2^sigma * ((A - 1024 X_A) + (B - 1024 X_B) / 16) + b * sum x folds the
//    affine group, X_A, X_B being the sums of the scaled activations of each
//    class.
//  * Slices of one row are summed in slice order through shared memory.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

namespace {

constexpr int kGrpKPL = 64;               // k per lane
constexpr int kGrpRPW = 4;                // rows per warp
// 12 consumer warps: K = 2048 S with S = 1, 2, 3, 4, 6 slices keeps every
// warp busy (S = 6 is the K = 12288 down projection); two CTAs per SM.
constexpr int kGrpWarps = 12;             // consumer warps
constexpr int kGrpCtasPerSm = 2;
constexpr size_t kGrpSmemBudget = 111 * 1024;
constexpr int kGrpMaxSlices = 8;          // K <= 16384
constexpr int kGrpThreads = 32 * (kGrpWarps + 1);
constexpr int kGrpWPL = kGrpKPL / 8;      // code words per lane per row
constexpr int kGrpRed = kGrpWarps * kGrpRPW;  // red floats per stage: S * R <= warps * RPW

struct GroupArgs {
  const GroupGemv* gemvs;
  const int* cta_tile0;  // [grid + 1] first tile of each CTA
  int ngemv;
  int ST;
  uint32_t stage_bytes;
  uint32_t* err;
};

}  // namespace

__global__ void __launch_bounds__(kGrpThreads, kGrpCtasPerSm) w4a16_group_kernel(const GroupArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // shared layout: [ST stages][stage_bytes] | red [ST][kGrpRed] f32 | barriers
  uint8_t* stages = smem;
  float* red = reinterpret_cast<float*>(smem + (size_t)a.ST * a.stage_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(red + (size_t)a.ST * kGrpRed);
  uint64_t* full = bars;
  uint64_t* empty = bars + a.ST;
  uint64_t* redfull = bars + 2 * a.ST;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kGrpWarps);
      mbar_init(&redfull[i], kGrpWarps);  // every consumer warp arrives once per tile
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  const int t0 = a.cta_tile0[blockIdx.x], t1 = a.cta_tile0[blockIdx.x + 1];

  if (warp == kGrpWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int g = 0;
      while (g + 1 < a.ngemv && a.gemvs[g].tile_end <= t0) ++g;
      GroupGemv d = a.gemvs[g];
      int it = 0;
      bool ok = true;
      for (int tile = t0; tile < t1 && ok; ++tile, ++it) {
        while (tile >= d.tile_end) d = a.gemvs[++g];
        const int st = it % a.ST;
        if (it >= a.ST) ok = mbar_wait(&empty[st], ((it / a.ST) & 1) ^ 1, a.err, kErrGemvEmptyWait);
        if (!ok) break;
        const uint32_t rcb = d.K / 2, rsb = d.K / 32;
        const int r0 = (tile - d.tile0) * d.R;
        const int rows = min(d.R, d.N - r0);
        uint8_t* dst = stages + (size_t)st * a.stage_bytes;
        const uint32_t cb = rows * rcb, sb = rows * rsb;
        mbar_arrive_expect_tx(&full[st], cb + 2 * sb);
        bulk_g2s_evict_first(dst, reinterpret_cast<const uint8_t*>(d.wq) + (size_t)r0 * rcb, cb, &full[st], pol);
        bulk_g2s(dst + (size_t)d.R * rcb, reinterpret_cast<const uint8_t*>(d.scales) + (size_t)r0 * rsb, sb,
                 &full[st]);
        bulk_g2s(dst + (size_t)d.R * (rcb + rsb), reinterpret_cast<const uint8_t*>(d.biases) + (size_t)r0 * rsb, sb,
                 &full[st]);
      }
      // drain: every issued copy must land before this CTA may exit
      const int issued = it;
      for (int j = max(0, issued - a.ST); j < issued; ++j)
        mbar_wait(&full[j % a.ST], (j / a.ST) & 1, a.err, kErrGemvDrain);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  pdl_wait();  // the activations may come from the previous kernel
  const uint32_t sbase = smem_u32(stages);
  int g = -1;
  GroupGemv d;
  int s = 0, rg = 0, k0 = 0, g_lane = 0;
  bool busy = false, active = false;
  uint32_t xr[kGrpWPL][4];  // fp16x2: (x0, x4), (x1, x5), (x2, x6), (x3, x7) of each word, scaled
  float sx = 0.f, up = 1.f, acc0a = 0.f, acc0b = 0.f;
  int it = 0, st = 0;
  uint32_t par = 0;
  for (int tile = t0; tile < t1; ++tile, ++it) {
    if (g < 0 || tile >= d.tile_end) {
      // next projection of the range: its slice layout and activations
      if (g < 0) {
        g = 0;
        while (g + 1 < a.ngemv && a.gemvs[g].tile_end <= t0) ++g;
      } else {
        ++g;
      }
      d = a.gemvs[g];
      while (tile >= d.tile_end) d = a.gemvs[++g];
      s = warp % d.S;
      rg = warp / d.S;
      busy = rg < d.RG;
      k0 = s * 32 * kGrpKPL + lane * kGrpKPL;
      active = busy && k0 < d.K;
      g_lane = k0 / 64;
      sx = 0.f;
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < kGrpWPL; ++i) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (active) v = *reinterpret_cast<const uint4*>(d.x + k0 + 8 * i);
        xr[i][0] = v.x;
        xr[i][1] = v.y;
        xr[i][2] = v.z;
        xr[i][3] = v.w;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float lo = bf16_bits_to_f32(xr[i][j] & 0xFFFFu), hi = bf16_bits_to_f32(xr[i][j] >> 16);
          sx += lo + hi;
          amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
        }
      }
      const int sig = fp16_prescale_exp(amax);
      const float down = pow2f(-sig);
      up = pow2f(sig);
      float sxa = 0.f, sxb = 0.f;
#pragma unroll
      for (int i = 0; i < kGrpWPL; ++i) {
        float xv[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          xv[2 * j] = bf16_bits_to_f32(xr[i][j] & 0xFFFFu) * down;
          xv[2 * j + 1] = bf16_bits_to_f32(xr[i][j] >> 16) * down;
        }
        // pair k and k + 4 of the word: the decode puts codes j and j + 4 in one register
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const __half2 h2 = __floats2half2_rn(xv[j], xv[j + 4]);
          xr[i][j] = *reinterpret_cast<const uint32_t*>(&h2);
          const float2 back = __half22float2(h2);
          if (j % 2 == 0) sxa += back.x + back.y; else sxb += back.x + back.y;
        }
      }
      acc0a = -1024.f * sxa;
      acc0b = -1024.f * sxb;
    }
    if (!mbar_wait(&full[st], par, a.err, kErrGemvFullWait)) break;
    const uint32_t rcb = d.K / 2, rsb = d.K / 32;
    const int r0 = (tile - d.tile0) * d.R;
    const int rows = min(d.R, d.N - r0);
    const uint32_t stg = sbase + st * a.stage_bytes;

    float part[kGrpRPW];
#pragma unroll
    for (int i = 0; i < kGrpRPW; ++i) {
      const int r = rg * kGrpRPW + i;
      part[i] = 0.f;
      if (active && r < rows) {
        uint32_t w[kGrpWPL];
        const uint32_t caddr = stg + r * rcb + k0 / 2;
#pragma unroll
        for (int v4 = 0; v4 < kGrpWPL / 4; ++v4) {
          const uint4 c = lds128(caddr + 16 * v4);
          w[4 * v4 + 0] = c.x;
          w[4 * v4 + 1] = c.y;
          w[4 * v4 + 2] = c.z;
          w[4 * v4 + 3] = c.w;
        }
        const float sc = f16_bits_to_f32(lds16(stg + d.R * rcb + r * rsb + 2 * g_lane));
        const float bi = f16_bits_to_f32(lds16(stg + d.R * (rcb + rsb) + r * rsb + 2 * g_lane));
        float aa = acc0a, ab = 0.f, ba = acc0b, bb = 0.f;
#pragma unroll
        for (int i2 = 0; i2 < kGrpWPL; ++i2) {
          uint32_t q[4];
          nib8_to_f16x2_offset(w[i2], q);
          aa = fma_f16_lo_lo(q[0], xr[i2][0], aa);
          ab = fma_f16_hi_hi(q[0], xr[i2][0], ab);
          ba = fma_f16_lo_lo(q[1], xr[i2][1], ba);
          bb = fma_f16_hi_hi(q[1], xr[i2][1], bb);
          aa = fma_f16_lo_lo(q[2], xr[i2][2], aa);
          ab = fma_f16_hi_hi(q[2], xr[i2][2], ab);
          ba = fma_f16_lo_lo(q[3], xr[i2][3], ba);
          bb = fma_f16_hi_hi(q[3], xr[i2][3], bb);
        }
        const float t = (aa + ab) + 0.0625f * (ba + bb);
        part[i] = fmaf(sc * up, t, bi * sx);
      }
    }
    const float v = transposed_warp_sum<kGrpRPW>(part, lane);
    constexpr int kLanesPerRow = 32 / kGrpRPW;
    const bool writer = (lane & (kLanesPerRow - 1)) == 0;
    const int myrow = rg * kGrpRPW + transposed_row<kGrpRPW>(lane);
    float* rb = red + (size_t)st * kGrpRed;
    if (busy && s != 0 && writer) rb[(s - 1) * d.R + myrow] = v;
    __syncwarp();
    if (lane == 0) mbar_arrive(&redfull[st]);
    if (busy && s == 0) {
      if (!mbar_wait(&redfull[st], par, a.err, kErrGemvFullWait)) break;
      if (writer && myrow < rows) {
        float tot = v;
        for (int s2 = 1; s2 < d.S; ++s2) tot += rb[(s2 - 1) * d.R + myrow];
        d.y[r0 + myrow] = tot;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    if (++st == a.ST) {
      st = 0;
      par ^= 1u;
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
bool group_gemv_ok(int N, int K) { return N >= 1 && K >= 2048 && K % 2048 == 0 && K / 2048 <= kGrpMaxSlices; }

cudaError_t group_plan_build(const GroupGemv* list, int n, int sms, GroupPlan* out) {
  GroupPlan p{};
  std::vector<GroupGemv> g(list, list + n);
  std::vector<long long> tile_bytes_end;  // cumulative bytes at the end of each projection's tiles
  long long tiles = 0;
  uint32_t stage_bytes = 0;
  for (auto& d : g) {
    d.S = d.K / 2048;
    d.RG = kGrpWarps / d.S;
    d.R = d.RG * kGrpRPW;
    d.tile0 = (int)tiles;
    tiles += (d.N + d.R - 1) / d.R;
    if (tiles >= (1LL << 31)) return cudaErrorInvalidValue;
    d.tile_end = (int)tiles;
    stage_bytes = std::max(stage_bytes, (uint32_t)d.R * (uint32_t)(d.K / 2 + d.K / 16));
  }
  // one contiguous tile range per CTA, equal cost per range:
  // a tile costs its bytes, scaled up when fewer than all consumer warps work
  // on it (K / 2048 slices that do not divide the eight warps)
  const int grid = (int)std::max<long long>(1, std::min<long long>((long long)kGrpCtasPerSm * sms, tiles));
  std::vector<long long> cum(tiles + 1, 0);
  for (const auto& d : g) {
    const long long row_cost = (long long)(d.K / 2 + d.K / 16) * kGrpWarps / (d.S * d.RG);
    for (int t = d.tile0; t < d.tile_end; ++t) {
      const int rows = std::min(d.R, d.N - (t - d.tile0) * d.R);
      cum[t + 1] = cum[t] + rows * row_cost;
    }
  }
  std::vector<int> cta(grid + 1);
  cta[0] = 0;
  for (int c = 1; c < grid; ++c) {
    const long long target = cum[tiles] * c / grid;
    cta[c] = (int)(std::lower_bound(cum.begin(), cum.end(), target) - cum.begin());
    cta[c] = std::max(cta[c], cta[c - 1]);
  }
  cta[grid] = (int)tiles;
  p.ngemv = n;
  p.grid = grid;
  p.stage_bytes = stage_bytes;  // a multiple of 16: K % 2048 == 0
  const size_t budget = kGrpSmemBudget;
  p.ST = (int)std::max<size_t>(2, std::min<size_t>(8, budget / (stage_bytes + sizeof(float) * kGrpRed + 24)));
  p.smem = (size_t)p.ST * stage_bytes + sizeof(float) * (size_t)p.ST * kGrpRed + 3 * 8 * (size_t)p.ST;
  cudaError_t e = cudaMalloc(&p.d_gemvs, sizeof(GroupGemv) * n);
  if (e != cudaSuccess) return e;
  e = cudaMalloc(&p.d_cta, sizeof(int) * (grid + 1));
  if (e != cudaSuccess) {
    cudaFree(p.d_gemvs);
    return e;
  }
  e = cudaMemcpy(p.d_gemvs, g.data(), sizeof(GroupGemv) * n, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(p.d_cta, cta.data(), sizeof(int) * (grid + 1), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(p.d_gemvs);
    cudaFree(p.d_cta);
    return e;
  }
  *out = p;
  return cudaSuccess;
}

void group_plan_free(GroupPlan* p) {
  if (p->d_gemvs) cudaFree(p->d_gemvs);
  if (p->d_cta) cudaFree(p->d_cta);
  p->d_gemvs = nullptr;
  p->d_cta = nullptr;
}

cudaError_t group_launch(const GroupPlan& p, uint32_t* err, cudaStream_t stream, bool pdl) {
  GroupArgs a;
  a.gemvs = p.d_gemvs;
  a.cta_tile0 = p.d_cta;
  a.ngemv = p.ngemv;
  a.ST = p.ST;
  a.stage_bytes = p.stage_bytes;
  a.err = err;
  cudaError_t e = allow_max_smem(w4a16_group_kernel);
  if (e != cudaSuccess) return e;
  return launch_kernel(w4a16_group_kernel, dim3(p.grid), dim3(kGrpThreads), p.smem, stream, pdl, a);
}

}  // namespace qg
