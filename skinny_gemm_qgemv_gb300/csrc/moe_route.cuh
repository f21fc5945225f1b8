// Router building blocks shared by the MoE kernels: order-preserving keys of
// the fp32 logits, a CTA-wide exclusive scan, and the exact top-k of one
// token on one warp (radix select on the keys, ties to the lower expert index,
// softmax probabilities of the selected experts).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace qg {
namespace {

constexpr unsigned kRouteFull = 0xFFFFFFFFu;

// 32-bit key with the order of the logits: larger logit, larger key; -0 = +0
__device__ __forceinline__ uint32_t logit_key(float v) {
  uint32_t b = __float_as_uint(v);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// exclusive prefix sum of one value per thread of the CTA (blockDim a multiple
// of 32); every thread calls it
__device__ __forceinline__ int cta_exclusive_scan(int v, int* wsum, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kRouteFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < (int)(blockDim.x >> 5) ? wsum[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kRouteFull, wi, o);
      if (lane >= o) wi += t;
    }
    wsum[lane] = wi - w;
    if (lane == 31) wsum[32] = wi;
  }
  __syncthreads();
  const int r = wsum[warp] + incl - v;
  total = wsum[32];
  __syncthreads();
  return r;
}

// One token's router on one warp. Lane l holds the keys of experts l + 32 i.
// The top_k-th largest key is found bit by bit from the top (a radix select
// that stops as soon as the keys matching the prefix are exactly the ones
// still needed); equal keys at the threshold are taken in expert order. The
// selected experts are ranked among themselves (larger logit first, ties to
// the lower index) and written with their softmax probabilities. PER: logits
// per lane (E <= 32 PER).
template <int PER>
__device__ __forceinline__ void route_token(const float* __restrict__ lg, int E, int top_k, int lane,
                                            uint32_t* sel_k, int* sel_e, int32_t* __restrict__ idx,
                                            float* __restrict__ wts, int* pe) {
  const int ne = (E + 31) >> 5;
  uint32_t key[PER];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    key[i] = 0u;
    const int e = 32 * i + lane;
    if (i < ne && e < E) {
      const float v = __ldg(lg + e);
      key[i] = logit_key(v);
      mx = fmaxf(mx, v);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kRouteFull, mx, o));
  float sm = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (i < ne && 32 * i + lane < E) sm += expf(key_logit(key[i]) - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(kRouteFull, sm, o);

  uint32_t prefix = 0u, mask = 0u;
  int need = top_k, match = E;  // keys still needed among those matching the prefix; how many match
  for (int b = 31; b >= 0 && match != need; --b) {
    const uint32_t bit = 1u << b, m2 = mask | bit, want = prefix | bit;
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if (i < ne && 32 * i + lane < E) cnt += (key[i] & m2) == want;
    cnt = (int)__reduce_add_sync(kRouteFull, (unsigned)cnt);
    if (cnt >= need) {
      prefix = want;
      match = cnt;
    } else {
      need -= cnt;
      match -= cnt;
    }
    mask = m2;
  }
  // every key above the prefix range, and `need` of the keys in it in expert order
  const unsigned below = (1u << lane) - 1u;
  int base = 0, eq_seen = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    if (i < ne) {
      const bool valid = 32 * i + lane < E;
      const uint32_t km = key[i] & mask;
      const bool eq = valid && km == prefix;
      const unsigned eqb = __ballot_sync(kRouteFull, eq);
      const bool take = (valid && km > prefix) || (eq && eq_seen + __popc(eqb & below) < need);
      eq_seen += __popc(eqb);
      const unsigned tb = __ballot_sync(kRouteFull, take);
      const int pos = base + __popc(tb & below);
      if (take && pos < 32) {
        sel_k[pos] = key[i];
        sel_e[pos] = 32 * i + lane;
      }
      base += __popc(tb);
    }
  }
  __syncwarp();
  if (lane < top_k) {
    const uint32_t kj = sel_k[lane];
    const int ej = sel_e[lane];
    int rank = 0;
    for (int l = 0; l < top_k; ++l) {
      const uint32_t kl = sel_k[l];
      rank += (kl > kj) || (kl == kj && sel_e[l] < ej);
    }
    idx[rank] = ej;
    wts[rank] = expf(key_logit(kj) - mx) / sm;
    pe[rank] = ej;
  }
  __syncwarp();
}

}  // namespace
}  // namespace qg
