// MXFP4 routed-expert MoE layer on the tensor cores (warp-level MMA): the main path.
//
// "Running Kimi K3 (2.8T) on one Apple Silicon Mac" (Deltafin), section "How it
// works": the router picks 16 experts per token and only the selected experts'
// weights are read; section "Technical approach / compute": the expert GEMV
// decodes the E2M1 codes and applies the E8M0 block scale in the same pass as
// the multiply. The layer is g = Wg[e] x, u = Wu[e] x, h = silu(g) u,
// y = sum_j p_j (Wd[e_j] h_j).
//
// Four launches:
//  * route (one CTA of 1024 threads per token): the exact top-k by a radix
//    select on order-preserving 32-bit keys of the logits with block-wide
//    counts (ties to the lower expert index), softmax weights, and the token's
//    x * 2^-sigma in fp16 (sigma an exact power of two that puts max |x| in
//    [2^14, 2^15)). The per-expert grouping into "virtual experts" (runs of at
//    most kMxTC = 8 pairs (token, slot) of one expert, the N = 8 columns of one
//    MMA) is built from the routing table by every CTA of the next kernels
//    (mx_group), so no CTA waits for another.
//  * gate/up: persistent, 16 warps; a tile is (virtual expert, 32 rows of I)
//    with both matrices, CTAs take contiguous tile ranges. A stage is 1024 k
//    (512 if H is not a multiple of 1024) of the tile's 32 gate and 32 up rows:
//    E2M1 codes by TMA (128B-swizzled) and E8M0 scales, in a ring of 4. Every
//    warp owns two 32-k blocks of every stage; one mma.sync.m16n8k16 row block
//    holds 8 gate rows (MMA rows 0..7) and the same 8 up rows (rows 8..15), so
//    g and u of a row meet in one accumulator fragment. B is the fp16 x of the
//    tile's pairs, loaded from L2 one stage ahead. Per block: 2 MMAs from
//    zero, then acc += result * 2^(scale - 127) per row (the block scale is a
//    row factor of the MMA result). No warp is set aside for the copies: the
//    last warp to release a slot issues the stage that goes into it. At the end
//    of a tile the warps' partial sums are added in warp order through shared
//    memory by one half of the warps (alternating per tile) and h = silu(g) u
//    is written in fp32 with the pair's max |h|.
//  * B rows of the down product (moe_mx_hprep_kernel): p h 2^-sigma_t in fp16
//    once per pair (sigma_t per token from max_j p_j max|h_j|), and a zero row.
//  * down: one CTA of 16 warps per range of R = 16 * MT rows of H, over every
//    virtual expert, 2048-k stages of its R rows as far as I allows. Up to 8
//    tokens the MMA columns are the batch's tokens, so one accumulator per
//    (row, token) collects all of a token's experts and one cross-warp sum
//    ends the kernel; with more tokens the columns are the pairs of the
//    current virtual expert (one n tile) and each virtual expert's columns are
//    added into per-warp token sums in shared memory. y = sum * 2^sigma_t.
// E2M1 codes go through the hardware cvt.rn.f16x2.e2m1x2 (exact); products are
// f16 x f16 with fp32 accumulation. Lane (g, c) of an MMA takes the 4 code
// bytes 4c..4c+3 of a block (codes 8c..8c+7): bytes 0, 1 are the k slots
// (2c, 2c+1) and (2c+8, 2c+9) of the first MMA, bytes 2, 3 those of the
// second; B is loaded in the same order (8 consecutive fp16 values), so the k
// permutation is the same on both sides and the dot product is unchanged.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qg_common.cuh"
#include "qg_internal.h"
#include "moe_route.cuh"

namespace qg {

namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kMxWarps = 16;                       // BPW 32-k blocks of every stage each
constexpr int kMxThreads = 32 * kMxWarps;
constexpr size_t kMxSmem = 227 * 1024;
// gate/up stage (up to 1024 k): codes [4 chunks][32 rows][128 B] per matrix, scales [32][32] per matrix
constexpr uint32_t kGuCodes = 4 * 32 * 128;
constexpr uint32_t kGuScales = 32 * 32;
constexpr uint32_t kGuStage = 2 * kGuCodes + 2 * kGuScales;
constexpr uint32_t kGuRed = 2u * kMxWarps * 4 * 32 * 16;  // two buffers of the warps' partial tiles

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = A B (zero accumulator)
__device__ __forceinline__ void mma_f16_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// E8M0 byte -> 2^(e - 127) by an integer multiply (the exponent field); e = 0
// (2^-127, below the normal range) gives 0
__device__ __forceinline__ float e8m0_mul(uint32_t e) { return __uint_as_float(e * 8388608u); }

__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}


__device__ __forceinline__ void bar_consumers() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kMxWarps) : "memory"); }

// split barrier over all warps of the CTA: the epilogue warps wait, the others
// only arrive (ids 2, 3)
__device__ __forceinline__ void bar_arrive_all(int id) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "n"(32 * kMxWarps) : "memory");
}
__device__ __forceinline__ void bar_sync_all(int id) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(32 * kMxWarps) : "memory");
}

// Stage release: every warp adds one to the slot's counter after its last read
// of the slot (acquire-release, so the last adder sees all the other warps'
// reads done); the last one re-arms the slot and issues the copies of the
// stage ST ahead into it. No warp is set aside for the copies.
__device__ __forceinline__ bool release_is_last(uint32_t* cnt, uint32_t warps) {
  uint32_t old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;" : "=r"(old) : "r"(smem_u32(cnt)) : "memory");
  if (old + 1u != warps) return false;
  *cnt = 0u;  // nobody touches the counter again before the new copies land
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic reads before the async-proxy writes
  return true;
}
// E8M0 scales land with the TMA swizzle that matches their row length S
// (S = 32: 32-byte swizzle, 16-byte unit ^= row bit 2; S = 64: 64-byte swizzle,
// unit ^= row bits 1..2; S = 16: none), so the 8 rows a warp reads at once sit
// in different banks. For the rows the kernels read (8 m + g, 16 m + g,
// 16 m + g + 8) the unit flip depends on g only.
template <uint32_t S>
__device__ __forceinline__ uint32_t scale_byte(uint32_t g, uint32_t b) {
  if (S == 32) return b ^ (((g >> 2) & 1u) << 4);
  if (S == 64) return b ^ (((g >> 1) & 3u) << 4);
  return b;
}
constexpr CUtensorMapSwizzle scale_swizzle(uint32_t S) {
  return S == 32 ? CU_TENSOR_MAP_SWIZZLE_32B : (S == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

// TMA 3D load with an L2 eviction-priority hint (streamed weights: evict first)
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const void* tm, int x, int y, int z, uint64_t* bar,
                                                 uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

}  // namespace

// ---------------------------------------------------------------------------
// route: top-k and softmax weights of one token per CTA, its fp16 activations
// ---------------------------------------------------------------------------
constexpr int kRouteThreads = 1024;  // one logit per thread (E <= 1024)

// CTA t routes token t: thread e holds logit e; the top_k-th largest key is
// found bit by bit from the top with block-wide counts (__syncthreads_count),
// stopping as soon as the keys matching the prefix are exactly the ones still
// needed; equal keys at the threshold are taken in expert order. The selected
// experts are ranked (larger logit first, ties to the lower index) and written
// with their softmax probabilities. In the same CTA: max |x| of the token and
// x * 2^-sigma in fp16 (sigma an exact power of two that puts max |x| in
// [2^14, 2^15)). The grouping into virtual experts is left to the kernels that
// use it (each CTA builds it from idx), so no CTA waits for another.
__global__ void __launch_bounds__(kRouteThreads) moe_mx_route_mma_kernel(
    const float* __restrict__ logits, const uint16_t* __restrict__ x, int H, int E, int top_k,
    int32_t* __restrict__ idx, float* __restrict__ wts, int32_t* __restrict__ xexp, uint16_t* __restrict__ xh,
    uint32_t* __restrict__ hmax) {
  __shared__ float s_mx[32], s_sum[32];
  __shared__ uint32_t s_xm[32];
  __shared__ int s_eq[32];
  __shared__ uint32_t sel_k[32];
  __shared__ int sel_e[32];
  __shared__ int s_n;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.x;
  const int cpt = H >> 3;  // 16-byte chunks of x per token
  const bool valid = tid < E;
  if (tid == 0) s_n = 0;
  pdl_wait();  // the logits and x may come from the previous kernel
  // every load first: logit tid of the token and the thread's chunks of x
  constexpr int kXr = 2;  // chunks a thread keeps in registers (H <= 16384); the rest is read twice
  const uint4* x4 = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  const float l = valid ? __ldg(logits + (size_t)t * E + tid) : 0.f;
  uint4 xv[kXr];
#pragma unroll
  for (int i = 0; i < kXr; ++i) {
    const int q = tid + i * kRouteThreads;
    xv[i] = q < cpt ? __ldg(x4 + q) : make_uint4(0u, 0u, 0u, 0u);
  }
  auto absmax8 = [](const uint4& w) {
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      m = fmaxf(m, fmaxf(fabsf(bf16_bits_to_f32(ww[j] & 0xFFFFu)), fabsf(bf16_bits_to_f32(ww[j] >> 16))));
    return m;
  };
  float xm = 0.f;
#pragma unroll
  for (int i = 0; i < kXr; ++i) xm = fmaxf(xm, absmax8(xv[i]));
  for (int q = tid + kXr * kRouteThreads; q < cpt; q += kRouteThreads) xm = fmaxf(xm, absmax8(__ldg(x4 + q)));
  // block maxima of the logits and of |x|
  float lm = valid ? l : -INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lm = fmaxf(lm, __shfl_xor_sync(kFull, lm, o));
    xm = fmaxf(xm, __shfl_xor_sync(kFull, xm, o));
  }
  if (lane == 0) {
    s_mx[warp] = lm;
    s_xm[warp] = __float_as_uint(xm);
  }
  __syncthreads();
  float mx = s_mx[lane];
  uint32_t xmb = s_xm[lane];  // non-negative floats: integer order
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    xmb = max(xmb, __shfl_xor_sync(kFull, xmb, o));
  }
  pdl_launch_dependents();
  // x * 2^-sigma in fp16 (exact scaling)
  const int sig = fp16_prescale_exp(__uint_as_float(xmb));
  if (tid == 0) xexp[t] = sig;
  const float sc = pow2f(-sig);
  uint4* xo = reinterpret_cast<uint4*>(xh + (size_t)t * H);
  auto scale8 = [sc](const uint4& w) {
    uint4 o;
    o.x = f16x2_rn(bf16_bits_to_f32(w.x & 0xFFFFu) * sc, bf16_bits_to_f32(w.x >> 16) * sc);
    o.y = f16x2_rn(bf16_bits_to_f32(w.y & 0xFFFFu) * sc, bf16_bits_to_f32(w.y >> 16) * sc);
    o.z = f16x2_rn(bf16_bits_to_f32(w.z & 0xFFFFu) * sc, bf16_bits_to_f32(w.z >> 16) * sc);
    o.w = f16x2_rn(bf16_bits_to_f32(w.w & 0xFFFFu) * sc, bf16_bits_to_f32(w.w >> 16) * sc);
    return o;
  };
#pragma unroll
  for (int i = 0; i < kXr; ++i) {
    const int q = tid + i * kRouteThreads;
    if (q < cpt) xo[q] = scale8(xv[i]);
  }
  for (int q = tid + kXr * kRouteThreads; q < cpt; q += kRouteThreads) xo[q] = scale8(__ldg(x4 + q));
  // softmax denominator: warp sums now, the block sum after the select's barriers
  float ev = valid ? expf(l - mx) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ev += __shfl_xor_sync(kFull, ev, o);
  if (lane == 0) s_sum[warp] = ev;
  // radix select of the top_k-th largest key
  const uint32_t key = valid ? logit_key(l) : 0u;
  uint32_t prefix = 0u, mask = 0u;
  int need = top_k, match = E;  // keys still needed among those matching the prefix; how many match
  for (int b = 31; b >= 0 && match != need; --b) {
    const uint32_t bit = 1u << b, m2 = mask | bit, want = prefix | bit;
    const int cnt = __syncthreads_count(valid && (key & m2) == want);
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
  const uint32_t km = key & mask;
  const bool eq = valid && km == prefix;
  bool take = valid && km > prefix;
  if (match == need) {
    take = take || eq;
  } else {  // all bits fixed and more equal keys than needed: the lowest expert indices
    const unsigned eqb = __ballot_sync(kFull, eq);
    if (lane == 0) s_eq[warp] = __popc(eqb);
    __syncthreads();
    int before = __popc(eqb & ((1u << lane) - 1u));
    for (int w = 0; w < warp; ++w) before += s_eq[w];
    take = take || (eq && before < need);
  }
  if (take) {
    const int pos = atomicAdd(&s_n, 1);
    sel_k[pos] = key;
    sel_e[pos] = tid;
  }
  __syncthreads();
  float sm = s_sum[lane];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(kFull, sm, o);
  if (tid < top_k) {
    const uint32_t kj = sel_k[tid];
    const int ej = sel_e[tid];
    int rank = 0;
    for (int j = 0; j < top_k; ++j) {
      const uint32_t kl = sel_k[j];
      rank += (kl > kj) || (kl == kj && sel_e[j] < ej);
    }
    const int p = t * top_k + rank;
    idx[p] = ej;
    wts[p] = expf(key_logit(kj) - mx) / sm;
    hmax[p] = 0u;
  }
}

// Virtual experts of the batch from the routing table idx [T][top_k]
// (T <= 32): the pairs (token, slot) of every expert in token order, cut into
// runs of at most kMxTC pairs (the N = 8 columns of one MMA), experts in index
// order. Table entry v: {expert, pair count, kMxTC pairs (-1 padded)} as
// int16, a pair p of token t stored as t << 10 | p (T, top_k <= 32, so p <
// 1024 and t < 32). Every thread of the CTA calls it; returns the number of
// entries.
// Scratch: 3 E words of shared memory.
constexpr int kVt = 2 + kMxTC;  // int16 per table entry
__device__ int mx_group(const int32_t* __restrict__ idx, int T, int E, int top_k, int* cnt, uint32_t* msk,
                        int* voff, int16_t* vt) {
  __shared__ int wsum[33];
  const int P = T * top_k;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    cnt[e] = 0;
    msk[e] = 0u;
  }
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int e = __ldcg(idx + p);
    atomicAdd(&cnt[e], 1);
    atomicOr(&msk[e], 1u << (p / top_k));
  }
  __syncthreads();
  // exclusive scan of the entries per expert; thread i owns experts [i EPT, (i + 1) EPT)
  const int ept = (E + (int)blockDim.x - 1) / (int)blockDim.x;
  const int e0 = threadIdx.x * ept;
  int mine = 0;
  for (int e = e0; e < min(E, e0 + ept); ++e) mine += (cnt[e] + kMxTC - 1) / kMxTC;
  int nv;
  int run = cta_exclusive_scan(mine, wsum, nv);
  for (int e = e0; e < min(E, e0 + ept); ++e) {
    voff[e] = run;
    run += (cnt[e] + kMxTC - 1) / kMxTC;
  }
  for (int q = threadIdx.x; q < nv * kVt; q += blockDim.x) vt[q] = -1;
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int e = __ldcg(idx + p), t = p / top_k;
    const int r = __popc(msk[e] & ((1u << t) - 1u));  // earlier tokens with this expert
    int16_t* ent = vt + (voff[e] + r / kMxTC) * kVt;
    const int j = r % kMxTC;
    ent[2 + j] = (int16_t)(t << 10 | p);
    if (j == 0) {
      ent[0] = (int16_t)e;
      ent[1] = (int16_t)min(kMxTC, cnt[e] - r);
    }
  }
  __syncthreads();
  return nv;
}


// ---------------------------------------------------------------------------
// gate/up + SwiGLU
// ---------------------------------------------------------------------------
struct MxGuArgs {
  const uint16_t* xh;    // [T][H] fp16 x * 2^-sigma_t
  const int32_t* xexp;   // [T] sigma_t
  const int32_t* idx;    // [T][top_k] routed experts
  float* h;              // [P][I]
  uint32_t* hmax;        // [P] bits of max |h|
  int H, I, T, E, top_k, ST, BPW;  // BPW: 32-k blocks per warp and stage (stage = 512 BPW k)
  uint32_t* err;
};

// x row of pair g of the tile's virtual expert (shared-memory table); columns
// past the pair count take pair 0's row (their MMA results are never read)
__device__ __forceinline__ const uint16_t* gu_xrow(const MxGuArgs& a, const int16_t* vt, int tile, int tpv, int g) {
  const int16_t* ent = vt + (tile / tpv) * kVt;
  const int j = min(g, ent[1] - 1);
  return a.xh + (size_t)(ent[2 + j] >> 10) * a.H;
}

// BPW: 32-k blocks per warp and stage (a stage is 512 BPW k of the tile's rows)
template <int BPW>
__global__ void __launch_bounds__(kMxThreads, 1)
    moe_mx_gu_mma_kernel(const __grid_constant__ CUtensorMap tm_gq, const __grid_constant__ CUtensorMap tm_uq,
                         const __grid_constant__ CUtensorMap tm_gs, const __grid_constant__ CUtensorMap tm_us,
                         const MxGuArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  // shared layout: stages | red (two buffers; the grouping's scratch before the
  //                first tile) | full barriers | release counters | virtual-expert table
  float4* red = reinterpret_cast<float4*>(gbase + (size_t)a.ST * kGuStage);
  uint64_t* full = reinterpret_cast<uint64_t*>(gbase + (size_t)a.ST * kGuStage + kGuRed);
  uint32_t* rel = reinterpret_cast<uint32_t*>(full + a.ST);
  int16_t* vt = reinterpret_cast<int16_t*>(rel + a.ST);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.ST; ++i) {
      mbar_init(&full[i], 1);
      rel[i] = 0u;
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();  // the routing table and x come from the route kernel
  pdl_launch_dependents();
  const int H = a.H, I = a.I;
  constexpr int KS = 512 * BPW;
  constexpr uint32_t kSRow = 16u * BPW;    // scale bytes of one row in a stage
  const int nks = H / KS;                   // stages per tile
  const int tpv = I / 32;                   // tiles per virtual expert
  int* scratch = reinterpret_cast<int*>(red);  // free until the first tile ends
  const int nv = mx_group(a.idx, a.T, a.E, a.top_k, scratch, reinterpret_cast<uint32_t*>(scratch + a.E),
                          scratch + 2 * a.E, vt);
  const int total = nv * tpv;
  const int per = (total + (int)gridDim.x - 1) / (int)gridDim.x;
  const int t0 = min(total, (int)blockIdx.x * per), t1 = min(total, t0 + per);
  const int nstages = (t1 - t0) * nks;
  const uint64_t pol = policy_evict_first();
  // stage q of this CTA into its slot: codes and scales of 32 gate and 32 up rows, 512 BPW k
  auto issue = [&](int q) {
    const int tl = q / nks, ks = q - tl * nks;
    const int v = (t0 + tl) / tpv;
    const int row = vt[v * kVt] * I + (t0 + tl - v * tpv) * 32;
    const int st = q % a.ST;
    const uint32_t sb = base + st * kGuStage;
    mbar_arrive_expect_tx(&full[st], (2 * 4096u + 512u) * 2u * BPW);
    tma_load_3d_hint(sb, &tm_gq, 0, row, 2 * BPW * ks, &full[st], pol);
    tma_load_3d_hint(sb + kGuCodes, &tm_uq, 0, row, 2 * BPW * ks, &full[st], pol);
    tma_load_2d(sb + 2 * kGuCodes, &tm_gs, 16 * BPW * ks, row, &full[st]);
    tma_load_2d(sb + 2 * kGuCodes + kGuScales, &tm_us, 16 * BPW * ks, row, &full[st]);
  };
  if (threadIdx.x == 0)
    for (int q = 0; q < min(a.ST, nstages); ++q) issue(q);

  // lane (g, c): MMA rows g (gate) and g + 8 (up) of each 8-row block, pair g,
  // codes / x at k = 8c .. 8c + 7 of blocks BPW w + j of every stage
  const int g = lane >> 2, c = lane & 3;
  const int et = threadIdx.x;
  // byte offsets in a stage of this lane's code word of row g, block BPW w + j (128B swizzle:
  // 16-byte unit u of row r at u ^ (r & 7)), and of its E8M0 scale; + 1024 mt / + 8 kSRow mt for
  // the rows of 8-row block mt
  uint32_t coff[BPW], soff[BPW];
#pragma unroll
  for (int j = 0; j < BPW; ++j) {
    const uint32_t blk = BPW * warp + j;
    coff[j] = (blk >> 3) * 4096u + g * 128u + (((blk & 7u) ^ (uint32_t)g) << 4) + 4u * c;
    soff[j] = 2 * kGuCodes + g * kSRow + scale_byte<kSRow>(g, blk);
  }
  int st = 0, q = 0, buf = 0;
  uint32_t par = 0;
  bool ok = true;
  // x of the next stage, loaded one stage ahead (L2-resident)
  uint4 xn[BPW];
  const uint16_t* xrow = t0 < t1 ? gu_xrow(a, vt, t0, tpv, g) : a.xh;
  auto load_x = [&](const uint16_t* row, int ks) {
#pragma unroll
    for (int j = 0; j < BPW; ++j)
      xn[j] = __ldg(reinterpret_cast<const uint4*>(row + ks * KS + 32 * (BPW * warp + j) + 8 * c));
  };
  if (t0 < t1) load_x(xrow, 0);
  for (int tile = t0; tile < t1; ++tile) {
    const int v = tile / tpv, r0 = (tile - v * tpv) * 32;
    const int16_t* ent = vt + v * kVt;
    const int np = ent[1];
    const uint16_t* xnext = tile + 1 < t1 ? gu_xrow(a, vt, tile + 1, tpv, g) : xrow;
    // this thread's epilogue column (pair) and its 2^sigma, fetched early
    const int ecol = 2 * (et & 3) + ((et >> 5) & 1);
    const int eent = ecol < np ? ent[2 + ecol] : 0;
    const int epair = eent & 1023;
    const float esc = pow2f(__ldg(a.xexp + (eent >> 10)));
    float acc[4][4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[mt][i] = 0.f;
    for (int ks = 0; ks < nks; ++ks, ++q) {
      uint4 xb[BPW];
#pragma unroll
      for (int j = 0; j < BPW; ++j) xb[j] = xn[j];
      if (ks + 1 < nks)
        load_x(xrow, ks + 1);
      else if (tile + 1 < t1)
        load_x(xnext, 0);
      if (ok) ok = mbar_wait(&full[st], par, a.err, kErrMoeWait);
      if (ok) {
        const uint8_t* sp = gbase + (size_t)st * kGuStage;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
          for (int j = 0; j < BPW; ++j) {
            const uint32_t wg = *reinterpret_cast<const uint32_t*>(sp + coff[j] + 1024u * mt);
            const uint32_t wu = *reinterpret_cast<const uint32_t*>(sp + kGuCodes + coff[j] + 1024u * mt);
            const float fg = e8m0_mul(sp[soff[j] + 8u * kSRow * mt]);
            const float fu = e8m0_mul(sp[kGuScales + soff[j] + 8u * kSRow * mt]);
            float t[4];
            mma_f16_z(t, e2m1x2_to_f16x2<0>(wg), e2m1x2_to_f16x2<0>(wu), e2m1x2_to_f16x2<1>(wg),
                      e2m1x2_to_f16x2<1>(wu), xb[j].x, xb[j].y);
            mma_f16(t, e2m1x2_to_f16x2<2>(wg), e2m1x2_to_f16x2<2>(wu), e2m1x2_to_f16x2<3>(wg),
                    e2m1x2_to_f16x2<3>(wu), xb[j].z, xb[j].w);
            acc[mt][0] = fmaf(t[0], fg, acc[mt][0]);
            acc[mt][1] = fmaf(t[1], fg, acc[mt][1]);
            acc[mt][2] = fmaf(t[2], fu, acc[mt][2]);
            acc[mt][3] = fmaf(t[3], fu, acc[mt][3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0 && release_is_last(&rel[st], kMxWarps) && q + a.ST < nstages) issue(q + a.ST);
      if (++st == a.ST) {
        st = 0;
        par ^= 1u;
      }
    }
    xrow = xnext;
    // the warps' partial tiles, summed in warp order; h = silu(g) u. Buffer and
    // barrier b alternate per tile, and so does the half of the warps that sums
    // (the other half only arrives and goes on). A warp writes buffer b again
    // two tiles later, after it waited at the other barrier for every warp,
    // which each arrive there only after they finished reading buffer b.
    float4* rb = red + buf * (kMxWarps * 4 * 32);
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
      rb[(warp * 4 + mt) * 32 + lane] = make_float4(acc[mt][0], acc[mt][1], acc[mt][2], acc[mt][3]);
    if ((warp >> 3) != buf) {
      bar_arrive_all(2 + buf);
    } else {
      bar_sync_all(2 + buf);
      const int e2 = et & 255;
      const int mt = e2 >> 6, hs = (e2 >> 5) & 1, l = e2 & 31;
      const int col = 2 * (l & 3) + hs;  // the pair
      if (col < np) {
        float gs = 0.f, us = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kMxWarps; ++w2) {
          const float4 r4 = rb[(w2 * 4 + mt) * 32 + l];
          gs += hs ? r4.y : r4.x;
          us += hs ? r4.w : r4.z;
        }
        const int pair = epair;
        const float gv = gs * esc, uv = us * esc;
        const float hv = gv / (1.f + expf(-gv)) * uv;
        const int row = r0 + 8 * mt + (l >> 2);
        a.h[(size_t)pair * I + row] = hv;
        atomicMax(&a.hmax[pair], __float_as_uint(fabsf(hv)));
      }
    }
    buf ^= 1;
  }
}

// ---------------------------------------------------------------------------
// B of the down product, once: p h 2^-sigma_t of every pair in fp16
// ---------------------------------------------------------------------------
// sigma_t puts the largest p |h| of token t's pairs in [2^14, 2^15) (the same
// exact power of two the down kernel undoes at the end). Every CTA of the down
// kernel reads these rows instead of converting the fp32 h of each of its
// stages itself. Row P is all zeros (the B column of a token not in a virtual
// expert).
__global__ void __launch_bounds__(256) moe_mx_hprep_kernel(const float* __restrict__ h,
                                                           const uint32_t* __restrict__ hmax,
                                                           const float* __restrict__ wts, uint16_t* __restrict__ hh,
                                                           int T, int I, int top_k) {
  pdl_wait();  // h and its maxima come from gate/up
  pdl_launch_dependents();
  const int P = T * top_k;
  const int lane = threadIdx.x & 31;
  const long long n8 = (long long)(P + 1) * I / 8;
  // 2^-sigma_t of token tok (warp-uniform): its pairs' p |h| maxima, one load per lane
  auto token_scale = [&](int tok) {
    float m = 0.f;
    for (int j = lane; j < top_k; j += 32)
      m = fmaxf(m, __ldcg(wts + tok * top_k + j) * __uint_as_float(__ldcg(hmax + tok * top_k + j)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    return pow2f(-fp16_prescale_exp(m));
  };
  // the loop is uniform over the block: every lane of a warp takes part in the shuffles
  for (long long q0 = (long long)blockIdx.x * blockDim.x; q0 < n8; q0 += (long long)gridDim.x * blockDim.x) {
    const long long q = q0 + threadIdx.x;
    const int p = q < n8 ? (int)(q * 8 / I) : P;
    const int tok = p < P ? p / top_k : -1;
    float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
    if (tok >= 0) {  // h first, so its latency overlaps the scale's loads
      lo = __ldcg(reinterpret_cast<const float4*>(h + q * 8));
      hi = __ldcg(reinterpret_cast<const float4*>(h + q * 8 + 4));
    }
    // a warp's items cover one or two tokens (at least 32 items per token);
    // any other token falls back to its own loop
    const int ta = __shfl_sync(kFull, tok, 0), tb = __shfl_sync(kFull, tok, 31);
    const float fa = ta >= 0 ? token_scale(ta) : 0.f;
    const float fb = (tb >= 0 && tb != ta) ? token_scale(tb) : fa;
    float f = tok == ta ? fa : fb;
    if (tok >= 0 && tok != ta && tok != tb) {
      float m = 0.f;
      for (int j = 0; j < top_k; ++j)
        m = fmaxf(m, __ldcg(wts + tok * top_k + j) * __uint_as_float(__ldcg(hmax + tok * top_k + j)));
      f = pow2f(-fp16_prescale_exp(m));
    }
    f *= tok >= 0 ? __ldcg(wts + p) : 0.f;
    uint4 o;
    o.x = f16x2_rn(lo.x * f, lo.y * f);
    o.y = f16x2_rn(lo.z * f, lo.w * f);
    o.z = f16x2_rn(hi.x * f, hi.y * f);
    o.w = f16x2_rn(hi.z * f, hi.w * f);
    if (q < n8) reinterpret_cast<uint4*>(hh)[q] = o;
  }
}

// ---------------------------------------------------------------------------
// down + routing-weighted combine
// ---------------------------------------------------------------------------
struct MxDnArgs {
  const uint16_t* hh;     // [P + 1][I] fp16 p h 2^-sigma_t of every pair (moe_mx_hprep_kernel), then a zero row
  const uint32_t* hmax;   // [P]
  const float* wts;       // [P] routing weights
  const int32_t* idx;     // [T][top_k] routed experts
  float* y;               // [T][H]
  int T, H, I, E, top_k, R, ST, BPW, nvmax;
  uint32_t stage_bytes, o_s;  // stage size; offset of the scales in a stage
  uint32_t* err;
};

// A lane's B columns in one virtual expert. Token columns (PC false): the
// columns are the batch's tokens 8 nt + g, B the fp16 row of the token's pair
// in this virtual expert (a token not in it: the zero row, so its column of B
// is 0); act: n tiles with at least one of their tokens in it. Pair columns
// (PC true, one n tile): column j is pair j of the virtual expert (past its
// pair count: the zero row); tk0, tk1: the tokens of the lane's accumulator
// columns 2c, 2c + 1, or -1.
template <int NT>
struct DnLane {
  const uint16_t* hp[NT];
  uint32_t act;
  int tk0, tk1;
};

// from the shared table: token columns, [nvmax][8 NT] pair of (virtual
// expert, token) or -1; pair columns, [nvmax][8] pairs of the virtual expert
// with their tokens, token << 10 | pair (T, top_k <= 32), or -1
template <int NT, bool PC>
__device__ __forceinline__ void dn_lane(const MxDnArgs& a, int v, int g, int c, const int16_t* tab, DnLane<NT>& L) {
  L.act = 0u;
  const int P = a.T * a.top_k;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int e = tab[v * 8 * NT + 8 * nt + g];
    const int pair = PC ? e & 1023 : e;
    L.hp[nt] = a.hh + (size_t)(e >= 0 ? pair : P) * a.I;
    if (PC || __any_sync(kFull, e >= 0)) L.act |= 1u << nt;
  }
  if (PC) {  // -1 >> 10 is -1: no token
    L.tk0 = tab[v * 8 + 2 * c] >> 10;
    L.tk1 = tab[v * 8 + 2 * c + 1] >> 10;
  }
}

// NT: n tiles of 8 tokens (T <= 8 NT); MT: 16-row blocks per CTA (R = 16 MT);
// BPW: 32-k blocks per warp and stage (a stage is 512 BPW k); PC: pair
// columns (NT = 1) with per-warp token sums in shared memory, for T > 8
template <int NT, int MT, int BPW, bool PC>
__global__ void __launch_bounds__(kMxThreads, 1)
    moe_mx_dn_mma_kernel(const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_ds,
                         const MxDnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  constexpr int R = 16 * MT;
  constexpr int KS = 512 * BPW;
  constexpr uint32_t kOS = 256u * R * BPW;                          // scales after the codes
  constexpr uint32_t kStage = (272u * R * BPW + 1023u) & ~1023u;
  constexpr uint32_t kSRow = 16u * BPW;
  // shared layout: stages (the cross-warp sums reuse them at the end) | sigma per token |
  //                full barriers | release counters | first weight rows | pair table |
  //                (pair columns) per-warp token sums [warp][T][R + 8]
  int* sig = reinterpret_cast<int*>(gbase + (size_t)a.ST * kStage);
  uint64_t* full = reinterpret_cast<uint64_t*>(sig + 32);
  uint32_t* rel = reinterpret_cast<uint32_t*>(full + a.ST);
  int* vrow = reinterpret_cast<int*>(rel + a.ST);  // first weight row of each virtual expert's range
  int16_t* tab = reinterpret_cast<int16_t*>(vrow + a.nvmax);              // [nvmax][8 NT] pair or -1
  float* ys = reinterpret_cast<float*>(
      (reinterpret_cast<uintptr_t>(tab + (size_t)a.nvmax * 8 * NT) + 15) & ~(uintptr_t)15);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.ST; ++i) {
      mbar_init(&full[i], 1);
      rel[i] = 0u;
    }
    fence_mbar_init();
  }
  // With programmatic launch this kernel starts once every CTA of the
  // preparation kernel has passed its own dependency wait, i.e. after gate/up
  // (and before it the route kernel) completed: h's maxima, the routing
  // weights and the virtual-expert table are final, so the prologue and the
  // first weight copies run before this kernel's wait. Only the prepared B rows
  // (read in the loop below) need it.
  // sigma_t: max over the token's pairs of p |h| lands in [2^14, 2^15) after scaling
  if (threadIdx.x < 32) {
    const int t = threadIdx.x;
    float m = 0.f;
    if (t < a.T)
      for (int j = 0; j < a.top_k; ++j) {
        const int p = t * a.top_k + j;
        m = fmaxf(m, a.wts[p] * __uint_as_float(a.hmax[p]));
      }
    sig[t] = fp16_prescale_exp(m);
  }
  __syncthreads();
  pdl_launch_dependents();
  const int H = a.H, I = a.I;
  const int nks = I / KS;
  const int n0 = blockIdx.x * R;
  // the virtual experts, built in the (still empty) stage ring: scratch, then the table
  int* scratch = reinterpret_cast<int*>(gbase);
  int16_t* vt = reinterpret_cast<int16_t*>(scratch + 3 * a.E);
  const int nv = mx_group(a.idx, a.T, a.E, a.top_k, scratch, reinterpret_cast<uint32_t*>(scratch + a.E),
                          scratch + 2 * a.E, vt);
  // CTAs walk the virtual experts from different starting points (no L2 hot spot on one h row)
  const int vstart = nv > 0 ? (int)(((long long)blockIdx.x * nv) / gridDim.x) : 0;
  const int nstages = nv * nks;
  const uint64_t pol = policy_evict_first();
  for (int v2 = threadIdx.x; v2 < nv; v2 += blockDim.x) vrow[v2] = vt[v2 * kVt] * H + n0;
  for (int q = threadIdx.x; q < nv * 8 * NT; q += blockDim.x) tab[q] = -1;
  __syncthreads();
  for (int q = threadIdx.x; q < nv * kMxTC; q += blockDim.x) {
    const int v2 = q / kMxTC, j = q - v2 * kMxTC;
    if (j < vt[v2 * kVt + 1]) {
      const int16_t ent = vt[v2 * kVt + 2 + j];  // token << 10 | pair
      if (PC)
        tab[v2 * 8 + j] = ent;
      else
        tab[v2 * 8 * NT + (ent >> 10)] = (int16_t)(ent & 1023);
    }
  }
  if (PC)
    for (int q = threadIdx.x; q < kMxWarps * (R + 8) * a.T; q += blockDim.x) ys[q] = 0.f;
  // the ring's generic writes (scratch, table) before the copies that refill it
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  // stage q of this CTA into its slot: codes and scales of its R rows of one virtual expert, KS k
  auto issue = [&](int q) {
    const int i = q / nks, ks = q - i * nks;
    int v = vstart + i;
    if (v >= nv) v -= nv;
    const int row = vrow[v];
    const int st = q % a.ST;
    const uint32_t sb = base + st * kStage;
    mbar_arrive_expect_tx(&full[st], 272u * R * BPW);
    tma_load_3d_hint(sb, &tm_dq, 0, row, 2 * BPW * ks, &full[st], pol);
    tma_load_2d(sb + kOS, &tm_ds, 16 * BPW * ks, row, &full[st]);
  };
  if (threadIdx.x == 0)
    for (int q = 0; q < min(a.ST, nstages); ++q) issue(q);
  pdl_wait();  // the prepared B rows come from the preparation kernel

  // lane (g, c): rows g, g + 8 of each 16-row block, tokens 8 nt + g, k = 8c .. 8c + 7
  // of blocks BPW w + j of every stage
  const int g = lane >> 2, c = lane & 3;
  const int et = threadIdx.x;
  uint32_t coff[BPW], soff[BPW];
#pragma unroll
  for (int j = 0; j < BPW; ++j) {
    const uint32_t blk = BPW * warp + j;
    coff[j] = (blk >> 3) * (128u * R) + g * 128u + (((blk & 7u) ^ (uint32_t)g) << 4) + 4u * c;
    soff[j] = kOS + g * kSRow + scale_byte<kSRow>(g, blk);
  }
  float acc[MT][NT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.f;
  // the next stage's B (fp16 p h 2^-sigma_t, k = 8c .. 8c + 7 of each block),
  // loaded one stage ahead (L2-resident): [nt][block]
  uint4 hn[NT][BPW];
  auto load_h = [&](const DnLane<NT>& L, int ks) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      if ((L.act >> nt) & 1u)
#pragma unroll
        for (int j = 0; j < BPW; ++j)
          hn[nt][j] = __ldcg(reinterpret_cast<const uint4*>(L.hp[nt] + ks * KS + 32 * (BPW * warp + j) + 8 * c));
  };
  DnLane<NT> cur, nxt;
  int st = 0, v = vstart, ks = 0, i = 0;
  uint32_t par = 0;
  bool ok = true;
  if (nv > 0) {
    dn_lane<NT, PC>(a, v, g, c, tab, cur);
    load_h(cur, 0);
  }
  for (int q = 0; q < nstages; ++q) {
    // this stage's B: p h 2^-sigma_t in fp16, as prepared
    uint32_t b[NT][BPW][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < BPW; ++j) {
        b[nt][j][0] = hn[nt][j].x;
        b[nt][j][1] = hn[nt][j].y;
        b[nt][j][2] = hn[nt][j].z;
        b[nt][j][3] = hn[nt][j].w;
      }
    // the next stage's h
    bool newv = false;
    if (ks + 1 < nks) {
      load_h(cur, ks + 1);
    } else if (i + 1 < nv) {
      dn_lane<NT, PC>(a, v + 1 == nv ? 0 : v + 1, g, c, tab, nxt);
      load_h(nxt, 0);
      newv = true;
    }
    if (PC && ks == 0)  // pair columns: the accumulators hold one virtual expert at a time
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i2 = 0; i2 < 4; ++i2) acc[mt][0][i2] = 0.f;
    if (ok) ok = mbar_wait(&full[st], par, a.err, kErrMoeWait);
    if (ok) {
      const uint8_t* sp = gbase + (size_t)st * kStage;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int j = 0; j < BPW; ++j) {
          // rows 16 mt + g and 16 mt + g + 8 (both with row & 7 = g)
          const uint32_t w0 = *reinterpret_cast<const uint32_t*>(sp + coff[j] + 2048u * mt);
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(sp + coff[j] + 2048u * mt + 1024u);
          const float f0 = e8m0_mul(sp[soff[j] + 16u * kSRow * mt]);
          const float f1 = e8m0_mul(sp[soff[j] + 16u * kSRow * mt + 8u * kSRow]);
          const uint32_t a0 = e2m1x2_to_f16x2<0>(w0), a1 = e2m1x2_to_f16x2<0>(w1);
          const uint32_t a2 = e2m1x2_to_f16x2<1>(w0), a3 = e2m1x2_to_f16x2<1>(w1);
          const uint32_t a4 = e2m1x2_to_f16x2<2>(w0), a5 = e2m1x2_to_f16x2<2>(w1);
          const uint32_t a6 = e2m1x2_to_f16x2<3>(w0), a7 = e2m1x2_to_f16x2<3>(w1);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (!((cur.act >> nt) & 1u)) continue;  // none of the n tile's tokens is in this virtual expert
            float t[4];
            mma_f16_z(t, a0, a1, a2, a3, b[nt][j][0], b[nt][j][1]);
            mma_f16(t, a4, a5, a6, a7, b[nt][j][2], b[nt][j][3]);
            acc[mt][nt][0] = fmaf(t[0], f0, acc[mt][nt][0]);
            acc[mt][nt][1] = fmaf(t[1], f0, acc[mt][nt][1]);
            acc[mt][nt][2] = fmaf(t[2], f1, acc[mt][nt][2]);
            acc[mt][nt][3] = fmaf(t[3], f1, acc[mt][nt][3]);
          }
        }
      }
    }
    if (PC && ks == nks - 1) {
      // the virtual expert is complete: add its columns to their tokens' sums
      // (this warp's own region; the lanes' (row, token) cells are distinct;
      // a token's rows are contiguous and tokens R + 8 words apart, so the 8
      // rows of one column fall in 8 consecutive banks)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i2 = 0; i2 < 4; ++i2) {
          const int tok = (i2 & 1) ? cur.tk1 : cur.tk0;
          if (tok >= 0) ys[(warp * a.T + tok) * (R + 8) + 16 * mt + g + 8 * (i2 >> 1)] += acc[mt][0][i2];
        }
    }
    __syncwarp();
    if (lane == 0 && release_is_last(&rel[st], kMxWarps) && q + a.ST < nstages) issue(q + a.ST);
    if (++st == a.ST) {
      st = 0;
      par ^= 1u;
    }
    if (++ks == nks) {
      ks = 0;
      ++i;
      v = v + 1 == nv ? 0 : v + 1;
    }
    if (newv) cur = nxt;
  }
  // every stage is consumed (and every copy landed): the ring holds the warps' partial tiles
  bar_consumers();
  if (PC) {
    for (int q = et; q < R * a.T; q += 32 * kMxWarps) {
      const int t = q / R, row = q - t * R;
      if (n0 + row >= H) continue;
      float sum = 0.f;
#pragma unroll 4
      for (int w2 = 0; w2 < kMxWarps; ++w2) sum += ys[(w2 * a.T + t) * (R + 8) + row];
      a.y[(size_t)t * H + n0 + row] = sum * pow2f(sig[t]);
    }
    return;
  }
  float4* red = reinterpret_cast<float4*>(gbase);
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      red[((warp * MT + mt) * NT + nt) * 32 + lane] =
          make_float4(acc[mt][nt][0], acc[mt][nt][1], acc[mt][nt][2], acc[mt][nt][3]);
  bar_consumers();
  const float* redf = reinterpret_cast<const float*>(gbase);
  for (int q = et; q < R * a.T; q += 32 * kMxWarps) {
    const int row = q / a.T, t = q - row * a.T;
    if (n0 + row >= H) continue;
    const int mt = row >> 4, rr = row & 15, nt = t >> 3, tc = t & 7;
    const int l = (rr & 7) * 4 + (tc >> 1), comp = (rr >> 3) * 2 + (tc & 1);
    float sum = 0.f;
#pragma unroll 4
    for (int w2 = 0; w2 < kMxWarps; ++w2) sum += redf[(((w2 * MT + mt) * NT + nt) * 32 + l) * 4 + comp];
    a.y[(size_t)t * H + n0 + row] = sum * pow2f(sig[t]);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {

struct MxDnPlan {
  int R, MT, NT, ST, BPW, grid;
  bool PC;  // pair columns
  uint32_t stage_bytes, o_s;
  size_t smem;
};

MxDnPlan plan_down(int T, int H, int I, int top_k, int nvmax, int sms) {
  MxDnPlan p{};
  // rows per CTA: a multiple of 16 that gives about one range per SM
  p.MT = std::min(4, std::max(1, (H + 16 * sms - 1) / (16 * sms)));
  p.R = 16 * p.MT;
  p.grid = (H + p.R - 1) / p.R;
  // up to 8 tokens: the MMA columns are the tokens; more: the columns are the
  // pairs of one virtual expert, with per-warp token sums in shared memory
  p.PC = T > 8;
  p.NT = 1;
  const size_t fixed = 1024 + 4 * 32 + 4 * (size_t)nvmax + 2 * (size_t)nvmax * 8 * p.NT + 64 +
                       (p.PC ? 16 + 4 * (size_t)kMxWarps * (p.R + 8) * T : 0);
  // 2048 k stages as far as I allows (the per-stage work of a warp -- the next
  // B rows, the wait, the release -- is spread over more blocks; measured on
  // T = 16 and 32: 2048 k with 3 or 2 stages in flight beats 1024 k with 6 or
  // 4), shorter ones only while fewer than 2 fit
  for (p.BPW = I % 2048 == 0 ? 4 : (I % 1024 == 0 ? 2 : 1);; p.BPW /= 2) {
    p.o_s = 256u * p.R * p.BPW;  // codes: [2 BPW chunks][R rows][128 B], then scales [R][16 BPW]
    p.stage_bytes = (272u * p.R * p.BPW + 1023u) & ~1023u;
    p.ST = fixed >= kMxSmem ? 0 : (int)std::min<size_t>(8, (kMxSmem - fixed) / (p.stage_bytes + 16));
    if (p.ST >= 2 || p.BPW == 1) break;
  }
  p.smem = fixed + (size_t)p.ST * (p.stage_bytes + 16);
  return p;
}

int plan_gateup_stages(int nvmax) {
  return (int)std::min<size_t>(8, (kMxSmem - 1024 - kGuRed - 2 * kVt * (size_t)nvmax - 64) / (kGuStage + 16));
}

size_t gateup_smem(int ST, int nvmax) {
  return 1024 + (size_t)ST * (kGuStage + 16) + kGuRed + 2 * kVt * (size_t)nvmax + 64;
}

template <int MT, int BPW, bool PC>
cudaError_t launch_down(const CUtensorMap& tm_dq, const CUtensorMap& tm_ds, const MxDnArgs& da, const MxDnPlan& pd,
                        cudaStream_t stream, bool pdl) {
  cudaError_t e = allow_max_smem(moe_mx_dn_mma_kernel<1, MT, BPW, PC>);
  if (e != cudaSuccess) return e;
  return launch_kernel(moe_mx_dn_mma_kernel<1, MT, BPW, PC>, dim3(pd.grid), dim3(kMxThreads), pd.smem, stream, pdl,
                       tm_dq, tm_ds, da);
}

template <int BPW, bool PC>
cudaError_t launch_down_mt(const CUtensorMap& tm_dq, const CUtensorMap& tm_ds, const MxDnArgs& da,
                           const MxDnPlan& pd, cudaStream_t stream, bool pdl) {
  switch (pd.MT) {
    case 1: return launch_down<1, BPW, PC>(tm_dq, tm_ds, da, pd, stream, pdl);
    case 2: return launch_down<2, BPW, PC>(tm_dq, tm_ds, da, pd, stream, pdl);
    case 3: return launch_down<3, BPW, PC>(tm_dq, tm_ds, da, pd, stream, pdl);
    default: return launch_down<4, BPW, PC>(tm_dq, tm_ds, da, pd, stream, pdl);
  }
}

template <bool PC>
cudaError_t launch_down_bpw(const CUtensorMap& tm_dq, const CUtensorMap& tm_ds, const MxDnArgs& da,
                            const MxDnPlan& pd, cudaStream_t stream, bool pdl) {
  return pd.BPW == 4   ? launch_down_mt<4, PC>(tm_dq, tm_ds, da, pd, stream, pdl)
         : pd.BPW == 2 ? launch_down_mt<2, PC>(tm_dq, tm_ds, da, pd, stream, pdl)
                       : launch_down_mt<1, PC>(tm_dq, tm_ds, da, pd, stream, pdl);
}

template <int BPW>
cudaError_t launch_gateup(const CUtensorMap* tm, const MxGuArgs& ga, int grid, size_t smem, cudaStream_t stream,
                          bool pdl) {
  cudaError_t e = allow_max_smem(moe_mx_gu_mma_kernel<BPW>);
  if (e != cudaSuccess) return e;
  return launch_kernel(moe_mx_gu_mma_kernel<BPW>, dim3(grid), dim3(kMxThreads), smem, stream, pdl, tm[0], tm[1],
                       tm[2], tm[3], ga);
}

}  // namespace

bool moe_mx_mma_ok(int T, int H, int I, int E, int top_k) {
  if (T < 1 || T > 32 || E < 1 || E > 1024 || top_k < 1 || top_k > 32 || top_k > E) return false;
  if (H < 512 || I < 512 || H % 512 || I % 512) return false;
  const int nvmax = moe_nvirt_max(T, E, top_k);
  const MxDnPlan pd = plan_down(T, H, I, top_k, nvmax, device_sm_count());
  if (pd.ST < 2 || (size_t)kMxWarps * pd.MT * pd.NT * 512 > (size_t)pd.ST * pd.stage_bytes) return false;
  // the down kernel builds the virtual-expert table in its stage ring before the first copy
  if ((size_t)12 * E + 2 * kVt * (size_t)nvmax > (size_t)pd.ST * pd.stage_bytes) return false;
  return plan_gateup_stages(nvmax) >= 2;
}

cudaError_t launch_moe_mx_mma(const uint16_t* x, const float* logits, const uint8_t* gq, const uint8_t* gs,
                              const uint8_t* uq, const uint8_t* us, const uint8_t* dq, const uint8_t* ds, int T,
                              int H, int I, int E, int top_k, float* y, int32_t* idx, float* wts, int32_t* xexp,
                              uint16_t* xh, uint32_t* hmax, float* h, uint16_t* hh, uint32_t* err,
                              cudaStream_t stream, bool pdl) {
  const int sms = device_sm_count();
  const int nvmax = moe_nvirt_max(T, E, top_k);
  cudaError_t e = launch_kernel(moe_mx_route_mma_kernel, dim3(T), dim3(kRouteThreads), 0, stream, pdl, logits, x, H,
                                E, top_k, idx, wts, xexp, xh, hmax);
  if (e != cudaSuccess) return e;
  // E2M1 codes as [rows][128-byte chunks] with 128B swizzle; E8M0 scales as 16 BPW-byte boxes
  const int gbpw = H % 1024 == 0 ? 2 : 1;
  const MxDnPlan pd = plan_down(T, H, I, top_k, nvmax, sms);
  CUtensorMap tm_gq, tm_uq, tm_gs, tm_us, tm_dq, tm_ds;
  const uint64_t rows_gu = (uint64_t)E * I, rows_d = (uint64_t)E * H;
  const uint32_t gb = 2 * gbpw, db = 2 * pd.BPW;
  if (!tmap_3d(&tm_gq, CU_TENSOR_MAP_DATA_TYPE_UINT8, gq, 128, rows_gu, H / 256, H / 2, 128, 128, 32, gb) ||
      !tmap_3d(&tm_uq, CU_TENSOR_MAP_DATA_TYPE_UINT8, uq, 128, rows_gu, H / 256, H / 2, 128, 128, 32, gb) ||
      !tmap_2d(&tm_gs, CU_TENSOR_MAP_DATA_TYPE_UINT8, gs, H / 32, rows_gu, H / 32, 8 * gb, 32,
               scale_swizzle(8 * gb)) ||
      !tmap_2d(&tm_us, CU_TENSOR_MAP_DATA_TYPE_UINT8, us, H / 32, rows_gu, H / 32, 8 * gb, 32,
               scale_swizzle(8 * gb)) ||
      !tmap_3d(&tm_dq, CU_TENSOR_MAP_DATA_TYPE_UINT8, dq, 128, rows_d, I / 256, I / 2, 128, 128, pd.R, db) ||
      !tmap_2d(&tm_ds, CU_TENSOR_MAP_DATA_TYPE_UINT8, ds, I / 32, rows_d, I / 32, 8 * db, pd.R,
               scale_swizzle(8 * db)))
    return cudaErrorInvalidValue;
  const int gst = plan_gateup_stages(nvmax);
  const MxGuArgs ga{xh, xexp, idx, h, hmax, H, I, T, E, top_k, gst, gbpw, err};
  const int gu_grid = std::min(sms, nvmax * (I / 32));
  const CUtensorMap gmaps[4] = {tm_gq, tm_uq, tm_gs, tm_us};
  e = gbpw == 2 ? launch_gateup<2>(gmaps, ga, gu_grid, gateup_smem(gst, nvmax), stream, pdl)
                : launch_gateup<1>(gmaps, ga, gu_grid, gateup_smem(gst, nvmax), stream, pdl);
  if (e != cudaSuccess) return e;
  {
    const long long n8 = (long long)(T * top_k + 1) * I / 8;
    const int grid = (int)std::min<long long>(4LL * sms, (n8 + 255) / 256);
    e = launch_kernel(moe_mx_hprep_kernel, dim3(grid), dim3(256), 0, stream, pdl, (const float*)h,
                      (const uint32_t*)hmax, (const float*)wts, hh, T, I, top_k);
    if (e != cudaSuccess) return e;
  }
  const MxDnArgs da{hh, hmax, wts, idx, y, T, H, I, E, top_k, pd.R, pd.ST, pd.BPW, nvmax, pd.stage_bytes, pd.o_s, err};
  return pd.PC ? launch_down_bpw<true>(tm_dq, tm_ds, da, pd, stream, pdl)
               : launch_down_bpw<false>(tm_dq, tm_ds, da, pd, stream, pdl);
}

}  // namespace qg
