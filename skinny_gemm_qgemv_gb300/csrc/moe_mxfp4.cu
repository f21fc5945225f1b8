// MXFP4 routed-expert MoE forward.
//
// "Running Kimi K3 (2.8T) on one Apple Silicon Mac" (Deltafin): section "How
// it works" -- the router picks 16 experts per token and only the selected
// experts' weights are read; section "Technical approach / compute" -- the
// expert GEMV decodes MXFP4 (E2M1 codes through a 16-entry table, E8M0 scale
// applied to the fp32 exponent) in one pass with the multiply. Position-major
// batching of several tokens per expert is the "K3_METAL_POSITION_BATCH" row
// of its configuration table.
//
// GB300 mapping:
//  1. router: one CTA per token -- fp32 softmax and an exact top-k by logit
//     (ties to the lower expert index); also writes the token's activations as
//     fp16 scaled by a power of two 2^-sigma (sigma from the row maximum) so
//     they fit fp16's range exactly.
//  2. grouping: one CTA -- per-expert counts, offsets, a stable pair order and
//     the ascending list of active experts.
//  3. gate/up: one warp per (active expert, row of I); lanes stream 16-byte
//     chunks of 32 E2M1 codes (one E8M0 block) of both matrices. Decode is the
//     hardware cvt.rn.f16x2.e2m1x2; products use fma.rn.f32.f16 into fp32. The
//     block scale and 2^sigma are applied in fp32. h = silu(g) * u in fp32.
//  4. h prescale: per pair, h -> fp16 scaled by 2^-sigma_h (exact scaling).
//  5. down: one warp per output row of H; it walks the active experts in
//     ascending order, computes o = Wd[e] h for each of the expert's pairs and
//     stores p * o in shared memory; the token outputs are summed in slot order.
// Every selected expert's weights are read once; no floating-point atomics.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

constexpr int kMoeMaxTopK = 32;
constexpr int kMoeMaxE = 1024;
constexpr int kMoePairChunk = 4;     // pairs of one expert held in registers at once

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

MoeLayout moe_layout(int T, int H, int I, int E, int top_k) {
  MoeLayout L;
  size_t off = 0;
  const size_t P = (size_t)T * top_k;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.pair_expert = take(sizeof(int32_t) * P);
  L.pair_weight = take(sizeof(float) * P);
  L.counts = take(sizeof(int32_t) * E);
  L.offsets = take(sizeof(int32_t) * (E + 1));
  L.active = take(sizeof(int32_t) * E);
  L.order = take(sizeof(int32_t) * P);
  L.nactive = take(sizeof(int32_t) * 4);
  L.xh = take(sizeof(uint16_t) * (size_t)T * H);
  L.xexp = take(sizeof(int32_t) * T);
  L.h = take(sizeof(float) * P * I);
  L.hh = take(sizeof(uint16_t) * (P + 1) * I);  // + a zero row (the MMA path's down B)
  L.hexp = take(sizeof(int32_t) * P);
  L.hmax = take(sizeof(uint32_t) * P);
  L.partial = take(0);
  L.has_tc = !moe_mx_mma_ok(T, H, I, E, top_k) && moe_mx_tc_ok(T, H, I, E, top_k);
  if (L.has_tc) {
    L.tc = moe_tc_layout(T, H, I, E, top_k, off);
    off = L.tc.end;
  }
  L.total = off;
  return L;
}

// ---------------------------------------------------------------------------
// 1. router + activation prescale (one CTA of 256 threads per token)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) moe_router_kernel(const float* __restrict__ logits,
                                                         const uint16_t* __restrict__ x, int H, int E, int top_k,
                                                         int32_t* __restrict__ idx, float* __restrict__ wts,
                                                         uint16_t* __restrict__ xh, int32_t* __restrict__ xexp) {
  __shared__ float lg[kMoeMaxE];
  __shared__ float red[8];
  __shared__ int redi[8];
  __shared__ int chosen[kMoeMaxTopK];
  pdl_wait();
  const int t = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float* l = logits + (size_t)t * E;
  float mx = -INFINITY;
  for (int e = tid; e < E; e += 256) {
    lg[e] = l[e];
    mx = fmaxf(mx, lg[e]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  mx = red[0];
  for (int w = 1; w < 8; ++w) mx = fmaxf(mx, red[w]);
  __syncthreads();
  float sum = 0.f;
  for (int e = tid; e < E; e += 256) sum += expf(lg[e] - mx);
  sum = warp_sum(sum);
  if (lane == 0) red[warp] = sum;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < 8; ++w) tot += red[w];
  __syncthreads();
  // top-k: k rounds of argmax (largest logit, ties to the lowest index)
  for (int r = 0; r < top_k; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int e = tid; e < E; e += 256) {
      bool taken = false;
      for (int j = 0; j < r; ++j) taken |= (chosen[j] == e);
      if (taken) continue;
      const float v = lg[e];
      if (v > bv || (v == bv && e < bi)) {
        bv = v;
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0) {
      red[warp] = bv;
      redi[warp] = bi;
    }
    __syncthreads();
    if (tid == 0) {
      float b2 = red[0];
      int i2 = redi[0];
      for (int w = 1; w < 8; ++w)
        if (red[w] > b2 || (red[w] == b2 && redi[w] < i2)) {
          b2 = red[w];
          i2 = redi[w];
        }
      chosen[r] = i2;
      idx[(size_t)t * top_k + r] = i2;
      wts[(size_t)t * top_k + r] = expf(lg[i2] - mx) / tot;
    }
    __syncthreads();
  }
  // activations -> fp16 * 2^-sigma
  float amax = 0.f;
  for (int k = tid; k < H; k += 256) amax = fmaxf(amax, fabsf(bf16_bits_to_f32(x[(size_t)t * H + k])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  amax = red[0];
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
  const int sg = fp16_prescale_exp(amax);
  if (tid == 0) xexp[t] = sg;
  for (int k = tid; k < H; k += 256) {
    const float v = ldexpf(bf16_bits_to_f32(x[(size_t)t * H + k]), -sg);
    xh[(size_t)t * H + k] = __half_as_ushort(__float2half_rn(v));
  }
}

// ---------------------------------------------------------------------------
// 2. grouping (one CTA of up to 1024 threads; thread e owns expert e)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) moe_group_kernel(const int32_t* __restrict__ idx, int P, int E,
                                                         int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ active, int32_t* __restrict__ order,
                                                         int32_t* __restrict__ nactive) {
  __shared__ int cnt[kMoeMaxE];
  __shared__ int off[kMoeMaxE + 1];
  __shared__ int act[kMoeMaxE + 1];
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += blockDim.x) {
    int c = 0;
    for (int p = 0; p < P; ++p) c += (idx[p] == e);
    cnt[e] = c;
  }
  __syncthreads();
  if (tid == 0) {
    int o = 0, a = 0;
    for (int e = 0; e < E; ++e) {
      off[e] = o;
      act[e] = a;
      o += cnt[e];
      a += cnt[e] > 0;
    }
    off[E] = o;
    act[E] = a;
    nactive[0] = a;
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    counts[e] = cnt[e];
    offsets[e] = off[e];
    if (cnt[e] > 0) active[act[e]] = e;
    int o = off[e];
    for (int p = 0; p < P; ++p)
      if (idx[p] == e) order[o++] = p;
  }
  if (tid == 0) offsets[E] = off[E];
}

// ---------------------------------------------------------------------------
// 3. gate/up + SwiGLU: block = 8 warps = 8 rows of one active expert
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mx_chunk_dot(const uint4 c, const uint4 (&xv)[4], float& acc) {
  // 32 codes (bytes c.x..c.w, 4 per word, 2 per byte) against 32 fp16 activations
  const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
  const uint32_t xw[16] = {xv[0].x, xv[0].y, xv[0].z, xv[0].w, xv[1].x, xv[1].y, xv[1].z, xv[1].w,
                           xv[2].x, xv[2].y, xv[2].z, xv[2].w, xv[3].x, xv[3].y, xv[3].z, xv[3].w};
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t h0 = e2m1x2_to_f16x2<0>(cw[i]);
    const uint32_t h1 = e2m1x2_to_f16x2<1>(cw[i]);
    const uint32_t h2 = e2m1x2_to_f16x2<2>(cw[i]);
    const uint32_t h3 = e2m1x2_to_f16x2<3>(cw[i]);
    a0 = fma_f16_lo_lo(h0, xw[4 * i + 0], a0);
    a1 = fma_f16_hi_hi(h0, xw[4 * i + 0], a1);
    a0 = fma_f16_lo_lo(h1, xw[4 * i + 1], a0);
    a1 = fma_f16_hi_hi(h1, xw[4 * i + 1], a1);
    a0 = fma_f16_lo_lo(h2, xw[4 * i + 2], a0);
    a1 = fma_f16_hi_hi(h2, xw[4 * i + 2], a1);
    a0 = fma_f16_lo_lo(h3, xw[4 * i + 3], a0);
    a1 = fma_f16_hi_hi(h3, xw[4 * i + 3], a1);
  }
  acc = a0 + a1;
}

__global__ void __launch_bounds__(256) moe_gateup_kernel(
    const uint8_t* __restrict__ gq, const uint8_t* __restrict__ gs, const uint8_t* __restrict__ uq,
    const uint8_t* __restrict__ us, const uint16_t* __restrict__ xh, const int32_t* __restrict__ xexp,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ active, const int32_t* __restrict__ order,
    const int32_t* __restrict__ nactive, int H, int I, int top_k, float* __restrict__ hout) {
  pdl_wait();
  const int rows_per_block = 8;
  const int blocks_per_expert = (I + rows_per_block - 1) / rows_per_block;
  const int a = blockIdx.x / blocks_per_expert;
  if (a >= nactive[0]) return;
  const int e = active[a];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = (blockIdx.x % blocks_per_expert) * rows_per_block + warp;
  if (i >= I) return;
  const int p0 = offsets[e], np = offsets[e + 1] - p0;
  const size_t row = (size_t)e * I + i;
  const uint8_t* grow = gq + row * (H / 2);
  const uint8_t* urow = uq + row * (H / 2);
  const uint8_t* gsr = gs + row * (H / 32);
  const uint8_t* usr = us + row * (H / 32);
  const int nchunks = H / 32;
  for (int pc = 0; pc < np; pc += kMoePairChunk) {
    const int npc = min(kMoePairChunk, np - pc);
    int tok[kMoePairChunk];
#pragma unroll
    for (int j = 0; j < kMoePairChunk; ++j) tok[j] = j < npc ? order[p0 + pc + j] / top_k : 0;
    float ag[kMoePairChunk], au[kMoePairChunk];
#pragma unroll
    for (int j = 0; j < kMoePairChunk; ++j) ag[j] = au[j] = 0.f;
    for (int c = lane; c < nchunks; c += 32) {
      const uint4 cg = ldg_stream128(grow + 16 * c);
      const uint4 cu = ldg_stream128(urow + 16 * c);
      const float sgv = e8m0_to_f32(gsr[c]);
      const float suv = e8m0_to_f32(usr[c]);
#pragma unroll
      for (int j = 0; j < kMoePairChunk; ++j) {
        if (j < npc) {
          const uint4* xp = reinterpret_cast<const uint4*>(xh + (size_t)tok[j] * H + 32 * c);
          const uint4 xv[4] = {__ldg(xp), __ldg(xp + 1), __ldg(xp + 2), __ldg(xp + 3)};
          float dg, du;
          mx_chunk_dot(cg, xv, dg);
          mx_chunk_dot(cu, xv, du);
          ag[j] = fmaf(dg, sgv, ag[j]);
          au[j] = fmaf(du, suv, au[j]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kMoePairChunk; ++j) {
      if (j < npc) {
        const float g = ldexpf(warp_sum(ag[j]), xexp[tok[j]]);
        const float u = ldexpf(warp_sum(au[j]), xexp[tok[j]]);
        if (lane == 0) {
          const float hv = g / (1.f + expf(-g)) * u;
          hout[(size_t)order[p0 + pc + j] * I + i] = hv;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// 4. h -> fp16 * 2^-sigma (one CTA per pair)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) moe_hprep_kernel(const float* __restrict__ h, int I,
                                                        uint16_t* __restrict__ hh, int32_t* __restrict__ hexp) {
  __shared__ float red[8];
  pdl_wait();
  const int p = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float amax = 0.f;
  for (int k = tid; k < I; k += 256) amax = fmaxf(amax, fabsf(h[(size_t)p * I + k]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  amax = red[0];
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
  const int sg = fp16_prescale_exp(amax);
  if (tid == 0) hexp[p] = sg;
  for (int k = tid; k < I; k += 256)
    hh[(size_t)p * I + k] = __half_as_ushort(__float2half_rn(ldexpf(h[(size_t)p * I + k], -sg)));
}

// ---------------------------------------------------------------------------
// 5. down GEMV + routing-weighted combine: block = 8 warps = 8 rows of H
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) moe_down_kernel(
    const uint8_t* __restrict__ dq, const uint8_t* __restrict__ ds, const uint16_t* __restrict__ hh,
    const int32_t* __restrict__ hexp, const float* __restrict__ wts, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ active, const int32_t* __restrict__ order, const int32_t* __restrict__ nactive,
    int T, int H, int I, int top_k, float* __restrict__ y) {
  extern __shared__ float pbuf[];  // [P][8]
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + warp;
  const int P = T * top_k;
  const int na = nactive[0];
  const int nchunks = I / 32;
  if (n < H) {
    for (int a = 0; a < na; ++a) {
      const int e = active[a];
      const int p0 = offsets[e], np = offsets[e + 1] - p0;
      const size_t row = (size_t)e * H + n;
      const uint8_t* drow = dq + row * (I / 2);
      const uint8_t* dsr = ds + row * (I / 32);
      for (int pc = 0; pc < np; pc += kMoePairChunk) {
        const int npc = min(kMoePairChunk, np - pc);
        int pr[kMoePairChunk];
#pragma unroll
        for (int j = 0; j < kMoePairChunk; ++j) pr[j] = j < npc ? order[p0 + pc + j] : 0;
        float ao[kMoePairChunk];
#pragma unroll
        for (int j = 0; j < kMoePairChunk; ++j) ao[j] = 0.f;
        for (int c = lane; c < nchunks; c += 32) {
          const uint4 cd = ldg_stream128(drow + 16 * c);
          const float sv = e8m0_to_f32(dsr[c]);
#pragma unroll
          for (int j = 0; j < kMoePairChunk; ++j) {
            if (j < npc) {
              const uint4* hp = reinterpret_cast<const uint4*>(hh + (size_t)pr[j] * I + 32 * c);
              const uint4 hv[4] = {__ldg(hp), __ldg(hp + 1), __ldg(hp + 2), __ldg(hp + 3)};
              float d;
              mx_chunk_dot(cd, hv, d);
              ao[j] = fmaf(d, sv, ao[j]);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < kMoePairChunk; ++j) {
          if (j < npc) {
            const float o = ldexpf(warp_sum(ao[j]), hexp[pr[j]]);
            if (lane == 0) pbuf[(size_t)pr[j] * 8 + warp] = wts[pr[j]] * o;
          }
        }
      }
    }
  }
  __syncwarp();
  if (n < H) {
    for (int t = lane; t < T; t += 32) {
      float acc = 0.f;
      for (int j = 0; j < top_k; ++j) acc += pbuf[(size_t)(t * top_k + j) * 8 + warp];
      y[(size_t)t * H + n] = acc;
    }
  }
  (void)P;
}

cudaError_t launch_moe_mxfp4(const uint16_t* x, const float* logits, const uint8_t* gq, const uint8_t* gs,
                             const uint8_t* uq, const uint8_t* us, const uint8_t* dq, const uint8_t* ds, int T,
                             int H, int I, int E, int top_k, float* y, int32_t* idx, float* wts, void* ws,
                             uint32_t* err, cudaStream_t stream, bool pdl) {
  const MoeLayout L = moe_layout(T, H, I, E, top_k);
  uint8_t* base = static_cast<uint8_t*>(ws);
  auto I32 = [&](size_t off) { return reinterpret_cast<int32_t*>(base + off); };
  const int P = T * top_k;
  cudaError_t e;
  const bool aligned = ((reinterpret_cast<uintptr_t>(gq) | reinterpret_cast<uintptr_t>(gs) |
                         reinterpret_cast<uintptr_t>(uq) | reinterpret_cast<uintptr_t>(us) |
                         reinterpret_cast<uintptr_t>(dq) | reinterpret_cast<uintptr_t>(ds) |
                         reinterpret_cast<uintptr_t>(x)) & 15u) == 0;
  const bool aligned32 = ((reinterpret_cast<uintptr_t>(gq) | reinterpret_cast<uintptr_t>(uq) |
                           reinterpret_cast<uintptr_t>(dq)) & 31u) == 0;
  if (aligned && moe_mx_mma_ok(T, H, I, E, top_k)) {
    // main path (T <= 32): routing (one CTA per token), then gate/up and down on warp-level MMA
    return launch_moe_mx_mma(x, logits, gq, gs, uq, us, dq, ds, T, H, I, E, top_k, y, idx, wts, I32(L.xexp),
                             reinterpret_cast<uint16_t*>(base + L.xh),
                             reinterpret_cast<uint32_t*>(base + L.hmax), reinterpret_cast<float*>(base + L.h),
                             reinterpret_cast<uint16_t*>(base + L.hh), err, stream, pdl);
  }
  if (aligned && aligned32 && L.has_tc) {
    // larger batches (33..64 tokens): block-scaled tcgen05 MMAs on the stored E2M1 codes and E8M0 scales
    return launch_moe_mx_tc(x, logits, gq, gs, uq, us, dq, ds, T, H, I, E, top_k, y, idx, wts, base, L.tc,
                            reinterpret_cast<float*>(base + L.h), err, stream, pdl);
  }
  // shapes outside the main path's tiling: one warp per row
  e = launch_kernel(moe_router_kernel, dim3(T), dim3(256), 0, stream, pdl, logits, x, H, E, top_k, idx, wts,
                    reinterpret_cast<uint16_t*>(base + L.xh), I32(L.xexp));
  if (e != cudaSuccess) return e;
  e = launch_kernel(moe_group_kernel, dim3(1), dim3(E < 1024 ? ((E + 31) / 32) * 32 : 1024), 0, stream, pdl,
                    (const int32_t*)idx, P, E, I32(L.counts), I32(L.offsets), I32(L.active), I32(L.order),
                    I32(L.nactive));
  if (e != cudaSuccess) return e;
  // every active expert gets its row blocks; at most min(E, P) experts are active
  const int maxact = P < E ? P : E;
  const int gu_blocks = maxact * ((I + 7) / 8);
  e = launch_kernel(moe_gateup_kernel, dim3(gu_blocks), dim3(256), 0, stream, pdl, gq, gs, uq, us,
                    (const uint16_t*)(base + L.xh), (const int32_t*)I32(L.xexp), (const int32_t*)I32(L.offsets),
                    (const int32_t*)I32(L.active), (const int32_t*)I32(L.order), (const int32_t*)I32(L.nactive), H,
                    I, top_k, reinterpret_cast<float*>(base + L.h));
  if (e != cudaSuccess) return e;
  e = launch_kernel(moe_hprep_kernel, dim3(P), dim3(256), 0, stream, pdl, (const float*)(base + L.h), I,
                    reinterpret_cast<uint16_t*>(base + L.hh), I32(L.hexp));
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(float) * (size_t)P * 8;
  e = allow_max_smem(moe_down_kernel);
  if (e != cudaSuccess) return e;
  e = launch_kernel(moe_down_kernel, dim3((H + 7) / 8), dim3(256), smem, stream, pdl, dq, ds,
                    (const uint16_t*)(base + L.hh), (const int32_t*)I32(L.hexp), (const float*)wts,
                    (const int32_t*)I32(L.offsets), (const int32_t*)I32(L.active), (const int32_t*)I32(L.order),
                    (const int32_t*)I32(L.nactive), T, H, I, top_k, y);
  return e;
}

}  // namespace qg
