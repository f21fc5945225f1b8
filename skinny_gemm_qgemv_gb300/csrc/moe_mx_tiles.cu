// MXFP4 routed-expert GEMVs, streamed through shared memory (the main path).
//
// "Running Kimi K3 (2.8T) on one Apple Silicon Mac" (Deltafin), section "How it
// works": only the router's selected experts are read; section "Technical
// approach / compute": the expert GEMV decodes the E2M1 codes and applies the
// E8M0 block scale in the same pass as the multiply. The layer is
// g = Wg[e] x, u = Wu[e] x, h = silu(g) u, y = sum_j p_j (Wd[e_j] h_j).
//
// GB300 design, shared by both kernels:
//  * The pairs (token, slot) routed to one expert are cut into "virtual
//    experts" of at most kMxTC pairs (built by the grouping kernel); a
//    consumer holds the activations of one virtual expert in registers.
//  * Persistent grid, one CTA per SM: one producer warp streams row tiles of
//    the selected experts' matrices (E2M1 codes and E8M0 scales are contiguous
//    per row range) into a ring of shared-memory stages with cp.async.bulk,
//    completing on mbarriers. Every selected expert's weights are read from
//    HBM once per virtual expert (once per expert unless more than kMxTC of
//    the batch's pairs chose it).
//  * Consumer warps own a fixed K slice: lane l covers one 32-element E8M0
//    block of every row. Codes go through the hardware cvt.rn.f16x2.e2m1x2 and
//    multiply fp16 activations prescaled by an exact power of two with
//    fma.rn.f32.f16 into fp32; the block scale is applied once per block.
//  * Lane partials are reduced with the transposed butterfly; K slices of one
//    row are summed in slice order through shared memory (deterministic).
//
// gate/up (one tile = R rows of I for both matrices of one virtual expert;
// contiguous tile ranges per CTA, so the activations are reloaded only when
// the virtual expert changes) writes h in fp32 and the per-pair max |h|.
// down (one CTA walks a range of R rows of H over every virtual expert; the
// producer also copies the fp32 h rows of the virtual expert's pairs) keeps
// p_j (Wd h_j) per pair and row in shared memory and finally sums each
// token's slots in slot order.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr size_t kSmemBudget = 224 * 1024;
// Consumer warps and rows per warp. With one pair per virtual expert (T = 1)
// the activations take 16 registers, so more warps fit the register file.
constexpr int gu_warps(int tc) { return tc == 1 ? 21 : 14; }
constexpr int dn_warps(int tc) { return tc == 1 ? 12 : 12; }
constexpr int gu_rpw(int) { return 4; }
constexpr int dn_rpw(int tc) { return tc == 1 ? 8 : 4; }
constexpr int kMaxSlices = 12;  // K / 1024 of either matrix (one 32-k block per lane)

struct MxGateUpArgs {
  const uint8_t* gq;
  const uint8_t* gs;
  const uint8_t* uq;
  const uint8_t* us;
  const uint16_t* x;
  const int32_t* xexp;
  const int32_t* vexp;   // [nv][kMxVexpInts]: expert, pair count, kMxTC pair indices (-1 padded)
  const int32_t* nvirt;
  float* h;
  uint32_t* hmax;
  int H, I, top_k;
  int S, RG, R, ST, tpe;
  uint32_t stage_bytes;
  uint32_t* err;
};

struct MxDownArgs {
  const uint8_t* dq;
  const uint8_t* ds;
  const float* h;
  const uint32_t* hmax;
  const float* wts;
  const int32_t* vexp;
  const int32_t* nvirt;
  float* y;
  int T, H, I, top_k;
  int S, RG, R, ST, nranges, nvmax;
  uint32_t stage_bytes;
  uint32_t* err;
};

// 32 E2M1 codes (16 bytes) -> 16 f16x2 registers, register q = codes 2q, 2q+1
__device__ __forceinline__ void e2m1x32_to_f16x2(const uint4 c, uint32_t (&o)[16]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[4 * i + 0] = e2m1x2_to_f16x2<0>(w[i]);
    o[4 * i + 1] = e2m1x2_to_f16x2<1>(w[i]);
    o[4 * i + 2] = e2m1x2_to_f16x2<2>(w[i]);
    o[4 * i + 3] = e2m1x2_to_f16x2<3>(w[i]);
  }
}

// sum of 32 products (f16 x f16, exact) in fp32
__device__ __forceinline__ float dot32_f16(const uint32_t (&wv)[16], const uint32_t (&xv)[16]) {
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    a0 = fma_f16_lo_lo(wv[q], xv[q], a0);
    a1 = fma_f16_hi_hi(wv[q], xv[q], a1);
  }
  return a0 + a1;
}

__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace

// ---------------------------------------------------------------------------
// routing and grouping in one CTA of 1024 threads
// ---------------------------------------------------------------------------
// Block-wide exclusive scan of one value per thread (blockDim.x == 1024).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane], wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFull, wi, o);
      if (lane >= o) wi += t;
    }
    warp_tot[lane] = wi - w;  // exclusive prefix of the warp totals
    if (lane == 31) warp_tot[32] = wi;
  }
  __syncthreads();
  const int r = warp_tot[warp] + incl - v;
  total = warp_tot[32];
  __syncthreads();
  return r;
}

// Per token: softmax over the E logits in fp32, the top_k experts by logit
// (descending, ties to the lower index; "How it works": the router picks 16
// experts per token) and the fp16 prescale of the token's activations. Tokens
// are handled in chunks of Tg; a group of 1024 / Tg threads serves one token and
// ranks each expert by counting the experts ahead of it, so the selection is
// exact and order-independent. Then the grouping: per-expert counts, the stable
// pair order and the virtual experts (runs of at most kMxTC pairs of one expert).
constexpr int kRouteLogits = 6144;  // logits of one token chunk in shared memory

__global__ void __launch_bounds__(1024) moe_mx_route_kernel(const float* __restrict__ logits,
                                                            const uint16_t* __restrict__ x, int T, int H, int E,
                                                            int top_k, int Tg, int32_t* __restrict__ idx,
                                                            float* __restrict__ wts, int32_t* __restrict__ xexp,
                                                            int32_t* __restrict__ order, int32_t* __restrict__ vexp,
                                                            int32_t* __restrict__ nvirt, uint32_t* __restrict__ hmax) {
  __shared__ float slog[kRouteLogits];
  __shared__ float red[32];
  __shared__ int cnt[1024];
  __shared__ int warp_tot[33];
  __shared__ int sidx[1024];
  __shared__ int sorder[1024];
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = T * top_k;
  const int G = 1024 / Tg, WG = G / 32;  // threads and warps per token
  const int grp = tid / G, g = tid % G;
  for (int t0 = 0; t0 < T; t0 += Tg) {
    const int nt = min(Tg, T - t0);
    for (int q = tid; q < nt * E; q += 1024) slog[q] = logits[(size_t)t0 * E + q];
    __syncthreads();
    const bool act = grp < nt;
    const int t = t0 + grp;
    const float* lg = slog + grp * E;
    float m = -INFINITY;
    if (act)
      for (int e = g; e < E; e += G) m = fmaxf(m, lg[e]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    float mx = red[grp * WG];
    for (int w = 1; w < WG; ++w) mx = fmaxf(mx, red[grp * WG + w]);
    __syncthreads();
    float sm = 0.f;
    if (act)
      for (int e = g; e < E; e += G) sm += expf(lg[e] - mx);
    sm = warp_sum(sm);
    if (lane == 0) red[warp] = sm;
    __syncthreads();
    float sum = 0.f;
    for (int w = 0; w < WG; ++w) sum += red[grp * WG + w];
    __syncthreads();
    if (act) {
      // TPE adjacent threads per expert (a power of two, TPE * E <= G) each
      // count the experts ahead of it in a strided share of the logits; their
      // counts add up over the TPE lanes (the whole warp runs every round)
      int tpe = 1;
      while (tpe < 32 && tpe * 2 * E <= G) tpe *= 2;
      const int per_round = G / tpe, rounds = (E + per_round - 1) / per_round;
      const int part = g % tpe;
      for (int r = 0; r < rounds; ++r) {
        const int e = r * per_round + g / tpe;
        const bool valid = e < E;
        const float v = valid ? lg[e] : 0.f;
        int rank = 0;
        if (valid) {
#pragma unroll 8
          for (int f = part; f < E; f += tpe) {
            const float vf = lg[f];
            rank += (vf > v) || (vf == v && f < e);
          }
        }
        for (int o = 1; o < tpe; o <<= 1) rank += __shfl_xor_sync(kFull, rank, o);
        if (valid && part == 0 && rank < top_k) {
          idx[(size_t)t * top_k + rank] = e;
          wts[(size_t)t * top_k + rank] = expf(v - mx) / sum;
          sidx[t * top_k + rank] = e;
        }
      }
    }
    // activations -> fp16 * 2^-sigma: sigma from max |x| of the token
    float amax = 0.f;
    if (act) {
      const uint4* xp = reinterpret_cast<const uint4*>(x + (size_t)t * H);
      for (int c = g; c < H / 8; c += G) {
        const uint4 w = __ldg(xp + c);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_f32(ww[q] & 0xFFFFu)), fabsf(bf16_bits_to_f32(ww[q] >> 16))));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    if (act && g == 0) {
      float am = red[grp * WG];
      for (int w = 1; w < WG; ++w) am = fmaxf(am, red[grp * WG + w]);
      xexp[t] = fp16_prescale_exp(am);
    }
    __syncthreads();
  }
  for (int e = tid; e < 1024; e += 1024) cnt[e] = 0;
  __syncthreads();
  // per-expert counts and each pair's rank among the earlier pairs of its expert
  for (int p = tid; p < P; p += 1024) atomicAdd(&cnt[sidx[p]], 1);
  __syncthreads();
  int total_pairs;
  const int off = block_exclusive_scan(tid < E ? cnt[tid] : 0, warp_tot, total_pairs);
  const int nv_e = tid < E ? (cnt[tid] + kMxTC - 1) / kMxTC : 0;
  int total_v;
  const int voff = block_exclusive_scan(nv_e, warp_tot, total_v);
  __syncthreads();
  // offsets replace the counts' slots (thread e owns expert e)
  if (tid < E) cnt[tid] = off;
  __syncthreads();
  for (int p = tid; p < P; p += 1024) {
    const int e = sidx[p];
    int rank = 0;
    for (int q = 0; q < p; ++q) rank += (sidx[q] == e);
    sorder[cnt[e] + rank] = p;
    order[cnt[e] + rank] = p;
    hmax[p] = 0u;
  }
  __syncthreads();
  if (tid < E) {
    const int n_e = (tid + 1 < E ? cnt[tid + 1] : total_pairs) - off;
    for (int c = 0; c < nv_e; ++c) {
      int32_t* ent = vexp + (size_t)(voff + c) * kMxVexpInts;
      const int n = min(kMxTC, n_e - c * kMxTC);
      ent[0] = tid;
      ent[1] = n;
      for (int j = 0; j < kMxTC; ++j) ent[2 + j] = j < n ? sorder[off + c * kMxTC + j] : -1;
    }
  }
  if (tid == 0) nvirt[0] = total_v;
}

// ---------------------------------------------------------------------------
// gate/up + SwiGLU
// ---------------------------------------------------------------------------
// TC: pairs per virtual expert held in registers (1 when every virtual expert
// has one pair, else kMxTC); the tile is RG x RPW rows
template <int TC>
__global__ void __launch_bounds__(32 * (gu_warps(TC) + 1), 1) moe_mx_gateup_kernel(const MxGateUpArgs a) {
  constexpr int kGuWarps = gu_warps(TC);
  constexpr int RPW = gu_rpw(TC);
  constexpr int V = RPW * TC * 2;  // values per lane: rows x pairs x {gate, up}
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H, I = a.I;
  const uint32_t rcb = H / 2, rsb = H / 32;  // code and scale bytes of one row
  const uint32_t o_gs = a.R * rcb, o_uq = o_gs + a.R * rsb, o_us = o_uq + a.R * rcb;
  // shared layout: stages | red [ST][S][RG][32] f32 | outv [RG][32] f32 | barriers
  uint8_t* stages = smem;
  float* red = reinterpret_cast<float*>(smem + (size_t)a.ST * a.stage_bytes);
  float* outv = red + (size_t)a.ST * a.S * a.RG * 32;
  uint64_t* bars = reinterpret_cast<uint64_t*>(outv + a.RG * 32);
  uint64_t* full = bars;
  uint64_t* empty = bars + a.ST;
  uint64_t* redfull = bars + 2 * a.ST;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kGuWarps);
      mbar_init(&redfull[i], a.S > 1 ? (a.S - 1) * a.RG : 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();  // the routing and the activations come from the previous kernels
  pdl_launch_dependents();
  const int nv = *a.nvirt;
  const int total = nv * a.tpe;
  const int per = (total + (int)gridDim.x - 1) / (int)gridDim.x;
  const int t0 = blockIdx.x * per, t1 = min(total, t0 + per);

  if (warp == kGuWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int it = 0;
      bool ok = true;
      for (int tile = t0; tile < t1 && ok; ++tile, ++it) {
        const int st = it % a.ST;
        if (it >= a.ST) ok = mbar_wait(&empty[st], ((it / a.ST) & 1) ^ 1, a.err, kErrMoeWait);
        if (!ok) break;
        const int v = tile / a.tpe, r0 = (tile % a.tpe) * a.R;
        const int rows = min(a.R, I - r0);
        const size_t row0 = (size_t)a.vexp[v * kMxVexpInts] * I + r0;
        uint8_t* dst = stages + (size_t)st * a.stage_bytes;
        const uint32_t cb = rows * rcb, sb = rows * rsb;
        mbar_arrive_expect_tx(&full[st], 2 * (cb + sb));
        bulk_g2s_evict_first(dst, a.gq + row0 * rcb, cb, &full[st], pol);
        bulk_g2s(dst + o_gs, a.gs + row0 * rsb, sb, &full[st]);
        bulk_g2s_evict_first(dst + o_uq, a.uq + row0 * rcb, cb, &full[st], pol);
        bulk_g2s(dst + o_us, a.us + row0 * rsb, sb, &full[st]);
      }
      const int issued = it;
      for (int j = max(0, issued - a.ST); j < issued; ++j)
        mbar_wait(&full[j % a.ST], (j / a.ST) & 1, a.err, kErrMoeWait);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int s = warp % a.S, rg = warp / a.S;
  const bool busy = rg < a.RG;
  const int kb = s * 32 + lane;  // the E8M0 block of this lane in every row
  const bool on = busy && kb < H / 32;
  uint32_t xr[TC][16];
  int cur_v = -1, np = 0;
  int my_pair = -1, my_sig = 0;  // lane j < TC: pair j of the virtual expert and its prescale
  int st = 0;
  uint32_t par = 0;
  for (int tile = t0; tile < t1; ++tile) {
    const int v = tile / a.tpe, r0 = (tile % a.tpe) * a.R;
    if (v != cur_v) {
      cur_v = v;
      np = a.vexp[v * kMxVexpInts + 1];
      my_pair = lane < np ? a.vexp[v * kMxVexpInts + 2 + lane] : -1;
      my_sig = my_pair >= 0 ? a.xexp[my_pair / a.top_k] : 0;
#pragma unroll
      for (int j = 0; j < TC; ++j) {
        const int pj = __shfl_sync(kFull, my_pair, j);
        const int sj = __shfl_sync(kFull, my_sig, j);
        if (on && pj >= 0) {
          // x * 2^-sigma rounded to fp16: the exact power-of-two prescale of the router
          const uint4* xp = reinterpret_cast<const uint4*>(a.x + (size_t)(pj / a.top_k) * H + 32 * kb);
          const float sc = pow2f(-sj);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 w = __ldg(xp + c);
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int q = 0; q < 4; ++q)
              xr[j][4 * c + q] = f32x2_to_f16x2(bf16_bits_to_f32(ww[q] & 0xFFFFu) * sc,
                                                bf16_bits_to_f32(ww[q] >> 16) * sc);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 16; ++q) xr[j][q] = 0u;
        }
      }
    }
    const int jl = lane % TC;
    const int pj_l = __shfl_sync(kFull, my_pair, jl);
    const int sj_l = __shfl_sync(kFull, my_sig, jl);
    if (!mbar_wait(&full[st], par, a.err, kErrMoeWait)) break;
    const uint8_t* sbase = stages + (size_t)st * a.stage_bytes;
    float acc[V];
#pragma unroll
    for (int q = 0; q < V; ++q) acc[q] = 0.f;
    if (on) {
#pragma unroll
      for (int rr = 0; rr < RPW; ++rr) {
        const int row = rg * RPW + rr;
        if (r0 + row < I) {
          uint32_t wv[16];
          e2m1x32_to_f16x2(lds128(smem_u32(sbase + row * rcb + 16 * kb)), wv);
          const float sg = e8m0_to_f32(sbase[o_gs + row * rsb + kb]);
#pragma unroll
          for (int j = 0; j < TC; ++j)
            if (j < np) acc[(rr * TC + j) * 2 + 0] = sg * dot32_f16(wv, xr[j]);
          e2m1x32_to_f16x2(lds128(smem_u32(sbase + o_uq + row * rcb + 16 * kb)), wv);
          const float su = e8m0_to_f32(sbase[o_us + row * rsb + kb]);
#pragma unroll
          for (int j = 0; j < TC; ++j)
            if (j < np) acc[(rr * TC + j) * 2 + 1] = su * dot32_f16(wv, xr[j]);
        }
      }
    }
    float tot = transposed_warp_sum<V>(acc, lane);
    if (s > 0) {
      if (busy) red[((st * a.S + s) * a.RG + rg) * 32 + lane] = tot;
      __syncwarp();
      if (lane == 0) {
        if (busy) mbar_arrive(&redfull[st]);
        mbar_arrive(&empty[st]);
      }
      if (++st == a.ST) {
        st = 0;
        par ^= 1u;
      }
      continue;
    }
    if (busy) {
      if (a.S > 1 && !mbar_wait(&redfull[st], par, a.err, kErrMoeWait)) break;
      for (int s2 = 1; s2 < a.S; ++s2) tot += red[((st * a.S + s2) * a.RG + rg) * 32 + lane];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);  // the stage and red[st] are no longer read
    if (busy) {
      outv[rg * 32 + transposed_row<V>(lane)] = tot;  // lanes holding the same total write the same value
      __syncwarp();
      if (lane < RPW * TC) {
        const int rr = lane / TC, j = lane % TC;
        const int row = r0 + rg * RPW + rr;
        if (j < np && row < I) {
          const float g = outv[rg * 32 + 2 * lane] * pow2f(sj_l);
          const float u = outv[rg * 32 + 2 * lane + 1] * pow2f(sj_l);
          const float hv = g / (1.f + expf(-g)) * u;
          a.h[(size_t)pj_l * I + row] = hv;
          atomicMax(&a.hmax[pj_l], __float_as_uint(fabsf(hv)));
        }
      }
      __syncwarp();
    }
    if (++st == a.ST) {
      st = 0;
      par ^= 1u;
    }
  }
}

// ---------------------------------------------------------------------------
// down + routing-weighted combine
// ---------------------------------------------------------------------------
template <int TC>
__global__ void __launch_bounds__(32 * (dn_warps(TC) + 2), 1)
    moe_mx_down_kernel(const __grid_constant__ CUtensorMap tm_h, const MxDownArgs a) {
  constexpr int kDnWarps = dn_warps(TC);
  constexpr int RPW = dn_rpw(TC);
  constexpr int V = RPW * TC;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H, I = a.I, P = a.T * a.top_k;
  const uint32_t rcb = I / 2, rsb = I / 32;
  // h rows land 128B-swizzled (16-byte unit u of block b at u ^ (b & 7)): 1024-byte aligned;
  // the converter warp writes them as fp16 * 2^-sigma at o_hf: block b's four
  // 16-byte units at b * 64 + ((c ^ ((b >> 1) & 3)) << 4), conflict-free for
  // the consumers' 128-bit loads
  const uint32_t o_s = a.R * rcb, o_h = (o_s + a.R * rsb + 1023u) & ~1023u, o_hf = o_h + TC * I * 4;
  pdl_wait();  // the routing table and h come from the previous kernels
  const int nv = *a.nvirt;
  // shared layout (from a 1024-byte aligned base): stages | red [ST][S][RG][32] |
  //                outv [RG][32] | pbl [P][R] | vtab [nv][kMxVexpInts] | sigp [P] | barriers
  uint8_t* stages = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);
  float* red = reinterpret_cast<float*>(stages + (size_t)a.ST * a.stage_bytes);
  float* outv = red + (size_t)a.ST * a.S * a.RG * 32;
  float* pbl = outv + a.RG * 32;
  int32_t* vtab = reinterpret_cast<int32_t*>(pbl + (size_t)P * a.R);
  int32_t* sigp = vtab + (size_t)a.nvmax * kMxVexpInts;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sigp + ((P + 1) & ~1));
  uint64_t* full = bars;
  uint64_t* empty = bars + a.ST;
  uint64_t* redfull = bars + 2 * a.ST;
  uint64_t* hready = bars + 3 * a.ST;  // the stage's h is in fp16

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kDnWarps + 1);  // consumers + the h converter
      mbar_init(&redfull[i], a.S > 1 ? (a.S - 1) * a.RG : 1);
      mbar_init(&hready[i], 1);
    }
    fence_mbar_init();
  }
  // the virtual-expert table and every pair's fp16 prescale, once per CTA
  for (int q = threadIdx.x; q < nv * kMxVexpInts; q += blockDim.x) vtab[q] = a.vexp[q];
  for (int q = threadIdx.x; q < P; q += blockDim.x) sigp[q] = fp16_prescale_exp(__uint_as_float(a.hmax[q]));
  __syncthreads();
  pdl_launch_dependents();
  // CTAs walk the virtual experts from different starting points, so that at
  // any time they read different h rows (no L2 hot spot on one pair's h)
  const int vstart = nv > 0 ? (int)(((long long)blockIdx.x * nv) / gridDim.x) % nv : 0;
  if (warp == kDnWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int it = 0;
      bool ok = true;
      for (int ri = blockIdx.x; ri < a.nranges && ok; ri += gridDim.x) {
        const int n0 = ri * a.R, rows = min(a.R, H - n0);
        for (int i = 0; i < nv && ok; ++i, ++it) {
          const int v = (vstart + i) % nv;
          const int st = it % a.ST;
          if (it >= a.ST) ok = mbar_wait(&empty[st], ((it / a.ST) & 1) ^ 1, a.err, kErrMoeWait);
          if (!ok) break;
          const int np = vtab[v * kMxVexpInts + 1];
          const size_t row0 = (size_t)vtab[v * kMxVexpInts] * H + n0;
          uint8_t* dst = stages + (size_t)st * a.stage_bytes;
          const uint32_t cb = rows * rcb, sb = rows * rsb, hb = I * 4;
          mbar_arrive_expect_tx(&full[st], cb + sb + np * hb);
          bulk_g2s_evict_first(dst, a.dq + row0 * rcb, cb, &full[st], pol);
          bulk_g2s(dst + o_s, a.ds + row0 * rsb, sb, &full[st]);
          for (int j = 0; j < np; ++j)
            tma_load_2d(smem_u32(dst + o_h + j * hb), &tm_h, 0, vtab[v * kMxVexpInts + 2 + j] * (I / 32),
                        &full[st]);
        }
      }
      const int issued = it;
      for (int j = max(0, issued - a.ST); j < issued; ++j)
        mbar_wait(&full[j % a.ST], (j / a.ST) & 1, a.err, kErrMoeWait);
    }
    return;
  }

  if (warp == kDnWarps + 1) {
    // ------------------------------------------------------- h converter
    // once per stage for the whole CTA: fp32 h of the virtual expert's pairs
    // -> fp16 * 2^-sigma (sigma from the pair's max |h|: in fp16's range)
    int st = 0;
    uint32_t par = 0;
    bool ok = true;
    for (int ri = blockIdx.x; ri < a.nranges && ok; ri += gridDim.x) {
      for (int i = 0, v = vstart; i < nv; ++i, v = (v + 1 == nv ? 0 : v + 1)) {
        const int np = vtab[v * kMxVexpInts + 1];
        if (ok) ok = mbar_wait(&full[st], par, a.err, kErrMoeWait);
        if (ok) {
          uint8_t* sbase = stages + (size_t)st * a.stage_bytes;
          for (int j = 0; j < np; ++j) {
            const float sc = pow2f(-sigp[vtab[v * kMxVexpInts + 2 + j]]);
            for (int b = lane; b < I / 32; b += 32) {
              const uint32_t hp = smem_u32(sbase + o_h + j * (I * 4) + b * 128);
              const uint32_t hq = smem_u32(sbase + o_hf + j * (I * 2) + b * 64);
              const uint32_t sw = (uint32_t)b & 7u, sw2 = ((uint32_t)b >> 1) & 3u;
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const uint4 w0 = lds128(hp + (((uint32_t)(2 * c) ^ sw) << 4));
                const uint4 w1 = lds128(hp + (((uint32_t)(2 * c + 1) ^ sw) << 4));
                uint4 o;
                o.x = f32x2_to_f16x2(__uint_as_float(w0.x) * sc, __uint_as_float(w0.y) * sc);
                o.y = f32x2_to_f16x2(__uint_as_float(w0.z) * sc, __uint_as_float(w0.w) * sc);
                o.z = f32x2_to_f16x2(__uint_as_float(w1.x) * sc, __uint_as_float(w1.y) * sc);
                o.w = f32x2_to_f16x2(__uint_as_float(w1.z) * sc, __uint_as_float(w1.w) * sc);
                sts128(hq + (((uint32_t)c ^ sw2) << 4), o);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&hready[st]);
          mbar_arrive(&empty[st]);
        }
        if (++st == a.ST) {
          st = 0;
          par ^= 1u;
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int s = warp % a.S, rg = warp / a.S;
  const bool busy = rg < a.RG;
  const int kb = s * 32 + lane;
  const bool on = busy && kb < I / 32;
  int st = 0;
  uint32_t par = 0;
  bool ok = true;
  for (int ri = blockIdx.x; ri < a.nranges; ri += gridDim.x) {
    const int n0 = ri * a.R, rows = min(a.R, H - n0);
    for (int i = 0, v = vstart; i < nv; ++i, v = (v + 1 == nv ? 0 : v + 1)) {
      const int cst = st;
      const uint32_t cpar = par;
      if (++st == a.ST) {
        st = 0;
        par ^= 1u;
      }
      const int np = vtab[v * kMxVexpInts + 1];
      const int jl = lane % TC;
      const int pj_l = vtab[v * kMxVexpInts + 2 + jl];
      const int sj_l = pj_l >= 0 ? sigp[pj_l] : 0;
      if (ok) ok = mbar_wait(&hready[cst], cpar, a.err, kErrMoeWait);
      const uint8_t* sbase = stages + (size_t)cst * a.stage_bytes;
      float acc[V];
#pragma unroll
      for (int q = 0; q < V; ++q) acc[q] = 0.f;
      if (on && ok) {
        // this lane's 32 values of h per pair, fp16 * 2^-sigma from the converter warp
        uint32_t xr[TC][16];
#pragma unroll
        for (int j = 0; j < TC; ++j) {
          if (j < np) {
            const uint32_t hq = smem_u32(sbase + o_hf + j * (I * 2) + kb * 64);
            const uint32_t sw2 = ((uint32_t)kb >> 1) & 3u;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint4 w = lds128(hq + (((uint32_t)c ^ sw2) << 4));
              xr[j][4 * c] = w.x;
              xr[j][4 * c + 1] = w.y;
              xr[j][4 * c + 2] = w.z;
              xr[j][4 * c + 3] = w.w;
            }
          } else {
#pragma unroll
            for (int q = 0; q < 16; ++q) xr[j][q] = 0u;
          }
        }
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
          const int row = rg * RPW + rr;
          if (row < rows) {
            uint32_t wv[16];
            e2m1x32_to_f16x2(lds128(smem_u32(sbase + row * rcb + 16 * kb)), wv);
            const float sd = e8m0_to_f32(sbase[o_s + row * rsb + kb]);
#pragma unroll
            for (int j = 0; j < TC; ++j)
              if (j < np) acc[rr * TC + j] = sd * dot32_f16(wv, xr[j]);
          }
        }
      }
      float tot = transposed_warp_sum<V>(acc, lane);
      if (s > 0) {
        if (busy) red[((cst * a.S + s) * a.RG + rg) * 32 + lane] = tot;
        __syncwarp();
        if (lane == 0) {
          if (busy) mbar_arrive(&redfull[cst]);
          mbar_arrive(&empty[cst]);
        }
        continue;
      }
      if (busy) {
        if (a.S > 1 && ok) ok = mbar_wait(&redfull[cst], cpar, a.err, kErrMoeWait);
        for (int s2 = 1; s2 < a.S; ++s2) tot += red[((cst * a.S + s2) * a.RG + rg) * 32 + lane];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[cst]);
      if (busy) {
        outv[rg * 32 + transposed_row<V>(lane)] = tot;
        __syncwarp();
        if (lane < RPW * TC) {
          const int rr = lane / TC, j = lane % TC;
          const int row = rg * RPW + rr;
          if (j < np && row < rows)
            pbl[(size_t)pj_l * a.R + row] = a.wts[pj_l] * (outv[rg * 32 + lane] * pow2f(sj_l));
        }
        __syncwarp();
      }
    }
    // every pair's row range is in pbl: the tokens' sums in slot order
    named_bar(1, 32 * kDnWarps);
    for (int q = threadIdx.x; q < a.T * rows; q += 32 * kDnWarps) {
      const int t = q / rows, r = q % rows;
      float acc = 0.f;
      for (int j = 0; j < a.top_k; ++j) acc += pbl[(size_t)(t * a.top_k + j) * a.R + r];
      a.y[(size_t)t * H + n0 + r] = acc;
    }
    named_bar(1, 32 * kDnWarps);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {

struct MxPlan {
  int S, RG, R, ST, nvmax;
  uint32_t stage_bytes;
  size_t smem;
  int count;  // tiles per virtual expert (gate/up) or row ranges (down)
};

MxPlan plan_gateup(int H, int I, int tc) {
  MxPlan p{};
  p.S = (H / 32 + 31) / 32;
  p.RG = gu_warps(tc) / p.S;
  p.R = p.RG * gu_rpw(tc);
  p.stage_bytes = (uint32_t)(2 * p.R * (H / 2 + H / 32));
  const size_t fixed = sizeof(float) * ((size_t)4 * p.S * p.RG * 32 + p.RG * 32) + 3 * 4 * 8 + 64;
  p.ST = (int)std::min<size_t>(6, (kSmemBudget - fixed) / (p.stage_bytes + sizeof(float) * p.S * p.RG * 32));
  p.smem = (size_t)p.ST * p.stage_bytes + sizeof(float) * ((size_t)p.ST * p.S * p.RG * 32 + p.RG * 32) +
           3 * (size_t)p.ST * 8 + 64;
  p.count = (I + p.R - 1) / p.R;
  return p;
}

MxPlan plan_down(int T, int H, int I, int E, int top_k, int tc) {
  MxPlan p{};
  p.S = (I / 32 + 31) / 32;
  p.RG = dn_warps(tc) / p.S;
  p.R = p.RG * dn_rpw(tc);
  const uint32_t o_h = (uint32_t)((p.R * (I / 2 + I / 32) + 1023) & ~1023);
  p.stage_bytes = (uint32_t)((o_h + tc * I * 6 + 1023) & ~1023);  // + fp32 h and its fp16 copy
  const size_t P = (size_t)T * top_k;
  p.nvmax = moe_nvirt_max(T, E, top_k);
  const size_t fixed = sizeof(float) * (p.RG * 32 + P * p.R) +
                       sizeof(int32_t) * ((size_t)p.nvmax * kMxVexpInts + ((P + 1) & ~(size_t)1)) + 64 + 1024;
  const size_t per_stage = p.stage_bytes + sizeof(float) * p.S * p.RG * 32 + 4 * 8;
  p.ST = fixed < kSmemBudget ? (int)std::min<size_t>(4, (kSmemBudget - fixed) / per_stage) : 0;
  p.smem = fixed + (size_t)p.ST * per_stage;
  p.count = (H + p.R - 1) / p.R;
  return p;
}

}  // namespace

bool moe_mx_tiles_ok(int T, int H, int I, int E, int top_k) {
  if (H % 512 || I % 512) return false;       // 16-byte aligned rows of E8M0 scales
  if (E > kRouteLogits || T * top_k > 1024) return false;  // routing in one CTA
  if (H / 1024 > kMaxSlices || I / 1024 > kMaxSlices) return false;
  if (I / 32 > 256) return false;  // one TMA box of h per pair
  const int tc = T == 1 ? 1 : kMxTC;
  if (plan_gateup(H, I, tc).ST < 2) return false;
  return plan_down(T, H, I, E, top_k, tc).ST >= 2;
}

cudaError_t launch_moe_mx_route(const float* logits, const uint16_t* x, int T, int H, int E, int top_k, int32_t* idx,
                                float* wts, int32_t* xexp, int32_t* order, int32_t* vexp, int32_t* nvirt,
                                uint32_t* hmax, cudaStream_t stream, bool pdl) {
  // tokens per chunk: a power of two, at most 32 (a warp per token), logits fit
  int Tg = 1;
  while (Tg * 2 <= 32 && Tg * 2 <= T && (Tg * 2) * E <= kRouteLogits) Tg *= 2;
  if (Tg * E > kRouteLogits) return cudaErrorInvalidValue;
  return launch_kernel(moe_mx_route_kernel, dim3(1), dim3(1024), 0, stream, pdl, logits, x, T, H, E, top_k, Tg, idx,
                       wts, xexp, order, vexp, nvirt, hmax);
}

template <int TC>
static cudaError_t launch_mx_tc(const uint8_t* gq, const uint8_t* gs, const uint8_t* uq, const uint8_t* us,
                                const uint8_t* dq, const uint8_t* ds, const uint16_t* x, const int32_t* xexp,
                                const int32_t* vexp, const int32_t* nvirt, const float* wts, float* h,
                                uint32_t* hmax, float* y, int T, int H, int I, int E, int top_k, uint32_t* err,
                                cudaStream_t stream, bool pdl) {
  const int sms = device_sm_count();
  const MxPlan pg = plan_gateup(H, I, TC);
  MxGateUpArgs ga{gq, gs, uq, us, x, xexp, vexp, nvirt, h, hmax, H, I, top_k,
                  pg.S, pg.RG, pg.R, pg.ST, pg.count, pg.stage_bytes, err};
  cudaError_t e = allow_max_smem(moe_mx_gateup_kernel<TC>);
  if (e != cudaSuccess) return e;
  e = launch_kernel(moe_mx_gateup_kernel<TC>, dim3(sms), dim3(32 * (gu_warps(TC) + 1)), pg.smem, stream, pdl, ga);
  if (e != cudaSuccess) return e;
  const MxPlan pd = plan_down(T, H, I, E, top_k, TC);
  MxDownArgs da{dq, ds, h, hmax, wts, vexp, nvirt, y, T, H, I, top_k,
                pd.S, pd.RG, pd.R, pd.ST, pd.count, pd.nvmax, pd.stage_bytes, err};
  // h [P][I] fp32 viewed as rows of one 32-element block (128 bytes), swizzled
  CUtensorMap tm_h;
  if (!tmap_2d(&tm_h, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, h, 32, (uint64_t)T * top_k * (I / 32), 128, 32,
               (uint32_t)(I / 32), CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  e = allow_max_smem(moe_mx_down_kernel<TC>);
  if (e != cudaSuccess) return e;
  return launch_kernel(moe_mx_down_kernel<TC>, dim3(std::min(sms, pd.count)), dim3(32 * (dn_warps(TC) + 2)), pd.smem,
                       stream, pdl, tm_h, da);
}

cudaError_t launch_moe_mx_tiles(const uint8_t* gq, const uint8_t* gs, const uint8_t* uq, const uint8_t* us,
                                const uint8_t* dq, const uint8_t* ds, const uint16_t* x, const int32_t* xexp,
                                const int32_t* vexp, const int32_t* nvirt, const float* wts, float* h,
                                uint32_t* hmax, float* y, int T, int H, int I, int E, int top_k, uint32_t* err,
                                cudaStream_t stream, bool pdl) {
  // with one token every expert holds one pair: single-pair kernels
  if (T == 1) return launch_mx_tc<1>(gq, gs, uq, us, dq, ds, x, xexp, vexp, nvirt, wts, h, hmax, y, T, H, I, E, top_k,
                                     err, stream, pdl);
  return launch_mx_tc<kMxTC>(gq, gs, uq, us, dq, ds, x, xexp, vexp, nvirt, wts, h, hmax, y, T, H, I, E, top_k, err,
                             stream, pdl);
}

}  // namespace qg
