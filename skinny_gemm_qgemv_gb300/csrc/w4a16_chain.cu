// W4A16 GEMV chain: the M = 1 projections of a decode step in dependency order,
// as one persistent launch.
//
// Each projection is y = W x with the affine 4-bit groups of "MLX Runner: An
// Inference Engine You Can Read", section "Architecture: one command buffer
// per token" (weight = scale x code + bias, g = 64). That section issues a
// whole token as one command buffer; in a decoder most projections depend on
// the previous one (q/k/v -> o -> gate_up -> down -> next layer), so the
// projections carry a dependency level: every projection of level L may read
// the outputs of levels < L. One kernel walks all levels; a level's inputs are
// awaited with an in-kernel barrier (a per-level tile counter in global
// memory), while the weights -- which depend on nothing -- keep streaming
// through each CTA's shared-memory ring across the barrier, so HBM does not
// drain between projections.
//
// Weights are copied once, at create, into a fragment-major layout (same
// bytes as the stored format): for every 16-row block and 64-k group one
// 576-byte unit, 512 bytes of codes ordered so that lane (g, c) of a warp
// finds the four code words of its mma.sync A fragments (rows g and g + 8) in
// 16 consecutive bytes, then the 16 rows' (scale, bias) pairs, (s_g, b_g,
// s_g+8, b_g+8) at byte 8 g. A row block is K/64 consecutive units, so a CTA
// streams contiguous runs with plain bulk copies and every shared-memory read
// is conflict-free.
//
// Arithmetic per 16 x 64 unit (one warp): a code word gives four fp16x2
// registers with one shift and four lop3s -- (1024 + q) for the codes in bits
// 0-3 of each half, (1024 + 16 q) for bits 4-7 -- that are exactly the A
// fragments of four m16n8k16 MMAs (the packing puts the right codes there). B
// holds the activations of the group scaled by a power of two 2^-sigma into
// fp16 (the largest |x| just below 2^15), divided by 16 in the (1024 + 16 q)
// slots; every lane loads the same B for its column, so all eight output
// columns carry the row sums. The MMA sum is sum q x' + 1024 (X'_a + X'_b),
// X' the sums of the B values of the group, so with P = 2^sigma and
// Q = 1024 P (X'_a + X'_b) the group adds s (P d - Q) + b sum x to the row.
// Products are exact; only fp32 sums round.
//
// CTA: one per SM; warp 8 is the producer (bulk copies of 64-group chunks of
// row blocks into a ring of stages), warps 0..7 the consumers: warp w owns the
// groups w, w + 8, ... of every chunk, so each warp only ever needs the B
// fragments of its own groups (built when its CTA enters a projection) and no
// warp waits for another inside a stage. At the end of a row block the 8
// warps' partial rows are added in warp order through shared memory by one
// warp (rotating with the block), which writes y and, at the end of a run of
// blocks, publishes the blocks to the level counter with a release add.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <numeric>
#include <vector>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

namespace {

constexpr int kChWarps = 8;                          // consumer warps
constexpr int kChThreads = 32 * (kChWarps + 1);      // + producer warp
constexpr int kChStageGroups = 64;                   // 64-k groups per stage (4096 k)
constexpr uint32_t kChUnit = 576;                    // one 16-row x 64-k unit
constexpr uint32_t kChStageBytes = kChStageGroups * kChUnit;
constexpr uint32_t kChRedBytes = kChWarps * 16 * 4;  // partial rows of one block, all warps
constexpr unsigned long long kChLevelWaitNs = 1000000000ull;  // 1 s

struct ChainArgs {
  const ChainProj* proj;
  const ChainSeg* seg;
  const int* cta_seg;      // [grid + 1] first segment of each CTA
  const int* level_tiles;  // [nlevels] row blocks per level
  unsigned* cnt;           // [nlevels + 1] blocks finished per level, then CTAs finished
  int nlevels;
  int ST;
  uint32_t bfr_bytes;      // B-fragment area: (max K / 64) x 128 bytes
  uint32_t* err;
  unsigned long long* trace;  // null, or [grid][nlevels][4] globaltimer stamps (see chain_trace)
};

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float f16x2_sum(uint32_t v) {
  float lo, hi;
  asm("{.reg .f16 l, h; mov.b32 {l, h}, %2; cvt.f32.f16 %0, l; cvt.f32.f16 %1, h;}" : "=f"(lo), "=f"(hi) : "r"(v));
  return lo + hi;
}
__device__ __forceinline__ void f16x2_split(uint32_t v, float& lo, float& hi) {
  asm("{.reg .f16 l, h; mov.b32 {l, h}, %2; cvt.f32.f16 %0, l; cvt.f32.f16 %1, h;}" : "=f"(lo), "=f"(hi) : "r"(v));
}

// Loads of data other CTAs of the same launch may have written: L2, not L1
// (ldcg32 in the common header).
__device__ __forceinline__ float2 ldcg_f2(const float* p) {
  float2 v;
  asm volatile("ld.global.cg.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
  return v;
}
// Trace stamps of one (CTA, level), in globaltimer nanoseconds: 0 the first
// consumer warp reaches the level, 1 its wait for the level below ends, 2 its
// input fragments are built, 3 the CTA's last row block of the level is
// published. Only with a trace buffer (off by default).
__device__ __forceinline__ void stamp(unsigned long long* tr, int nlevels, int level, int field, bool latest);

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void stamp(unsigned long long* tr, int nlevels, int level, int field, bool latest) {
  if (!tr) return;
  unsigned long long* p = tr + ((size_t)blockIdx.x * nlevels + level) * 4 + field;
  const unsigned long long t = globaltimer();
  if (latest)
    atomicMax(p, t);
  else
    *p = t;
}

// bf16 rounding (nearest even) of an fp32 value, returned as fp32
__device__ __forceinline__ float round_bf16(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// Bounded mbarrier wait that also gives up when another warp of the CTA did.
__device__ __forceinline__ bool ch_wait(uint64_t* bar, uint32_t parity, uint32_t* err, uint32_t code,
                                        volatile int* abort_flag) {
  for (uint32_t i = 0; i < kMaxPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  report_error(err, code);
  *abort_flag = 1;
  return false;
}

// Wait (bounded in time) until `cnt` reaches `target`: acquire load, so the
// outputs published with the release adds are visible afterwards.
__device__ __forceinline__ bool wait_level(const unsigned* cnt, unsigned target, uint32_t* err,
                                           volatile int* abort_flag) {
  const uint64_t t0 = globaltimer();
  unsigned ns = 32;
  for (;;) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
    if (v >= target) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kChLevelWaitNs) {
      report_error(err, kErrChainLevelWait);
      *abort_flag = 1;
      return false;
    }
    __nanosleep(ns);
    if (ns < 64) ns <<= 1;
  }
}

// The 16 activations lane c of a group needs, in slot order: for MMA step s,
// k = 16 s + 2c, 16 s + 2c + 1 (slots a) and 16 s + 2c + 8, + 9 (slots b).
__device__ __forceinline__ void load_x16(const ChainProj& p, int k0, int c, float (&v)[16]) {
  if (p.op == kChainXBf16) {
    const uint16_t* x = static_cast<const uint16_t*>(p.xsrc);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t w = ldcg32(x + k0 + 16 * s + 2 * c + 8 * h);
        v[4 * s + 2 * h] = bf16_bits_to_f32(w & 0xFFFFu);
        v[4 * s + 2 * h + 1] = bf16_bits_to_f32(w >> 16);
      }
    }
  } else if (p.op == kChainXCopy) {
    const float* src = static_cast<const float*>(p.xsrc);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float2 f = ldcg_f2(src + k0 + 16 * s + 2 * c + 8 * h);
        v[4 * s + 2 * h] = round_bf16(p.alpha * f.x);
        v[4 * s + 2 * h + 1] = round_bf16(p.alpha * f.y);
      }
    }
  } else {  // SwiGLU of a fused gate/up output: gate at [0, K), up at [K, 2K)
    const float* src = static_cast<const float*>(p.xsrc);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int k = k0 + 16 * s + 2 * c + 8 * h;
        const float2 gt = ldcg_f2(src + k);
        const float2 up = ldcg_f2(src + p.K + k);
        v[4 * s + 2 * h] = round_bf16(gt.x / (1.0f + expf(-gt.x)) * up.x * p.alpha);
        v[4 * s + 2 * h + 1] = round_bf16(gt.y / (1.0f + expf(-gt.y)) * up.y * p.alpha);
      }
    }
  }
}

// B fragments and the fold constants (P, Q, sum x) of this warp's groups of a
// projection. In pass ps lane (j, c) = (lane / 4, lane % 4) handles group
// w + 8 (8 ps + j).
__device__ void build_x(const ChainProj& p, int w, int lane, uint32_t bfr_s, uint32_t kc_s) {
  constexpr int kPass = kChainMaxK / 64 / kChWarps / 8;  // passes of 8 groups a warp may need
  const int G = p.K >> 6;
  const int c = lane & 3;
  // every pass's loads first: one round trip to L2 for the whole input
  float v[kPass][16];
#pragma unroll
  for (int ps = 0; ps < kPass; ++ps) {
    const int gi = w + kChWarps * (8 * ps + (lane >> 2));
    if (gi < G) {
      load_x16(p, 64 * gi, c, v[ps]);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[ps][i] = 0.f;
    }
  }
#pragma unroll
  for (int ps = 0; ps < kPass; ++ps) {
    if (w + kChWarps * 8 * ps >= G) break;  // warp-uniform
    const int gi = w + kChWarps * (8 * ps + (lane >> 2));
    const bool act = gi < G;
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[ps][i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int sig = fp16_prescale_exp(amax);
    const float down = pow2f(-sig), P = pow2f(sig);
    uint32_t bq[8];
    float sa = 0.f, sb = 0.f, sx = 0.f;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      bq[2 * s] = f16x2_rn(v[ps][4 * s] * down, v[ps][4 * s + 1] * down);
      bq[2 * s + 1] = f16x2_rn(v[ps][4 * s + 2] * down * 0.0625f, v[ps][4 * s + 3] * down * 0.0625f);
      sa += f16x2_sum(bq[2 * s]);
      sb += f16x2_sum(bq[2 * s + 1]);
      sx += (v[ps][4 * s] + v[ps][4 * s + 1]) + (v[ps][4 * s + 2] + v[ps][4 * s + 3]);
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      sa += __shfl_xor_sync(0xffffffffu, sa, o);
      sb += __shfl_xor_sync(0xffffffffu, sb, o);
      sx += __shfl_xor_sync(0xffffffffu, sx, o);
    }
    if (act) {
      sts128(bfr_s + gi * 128 + c * 32, make_uint4(bq[0], bq[1], bq[2], bq[3]));
      sts128(bfr_s + gi * 128 + c * 32 + 16, make_uint4(bq[4], bq[5], bq[6], bq[7]));
      if (c == 0)
        sts128(kc_s + gi * 16, make_uint4(__float_as_uint(P), __float_as_uint(P * 1024.f * (sa + sb)),
                                          __float_as_uint(sx), 0u));
    }
  }
}

// Operands of one 16-row x 64-k unit for one lane.
struct UnitOps {
  uint4 wv;      // code words: row g steps 0-1, row g steps 2-3, row g+8 steps 0-1, row g+8 steps 2-3
  uint2 sb;      // (s, b) of rows g and g + 8
  uint4 bA, bB;  // B fragments of steps 0-1 and 2-3
  uint4 kq;      // P, Q, sum x of the group
};

__device__ __forceinline__ void unit_load(UnitOps& o, uint32_t u, uint32_t bfr, uint32_t kc, int lane, int g, int c) {
  o.wv = lds128(u + lane * 16);
  o.sb = lds64(u + 512 + 8 * g);
  o.bA = lds128(bfr + c * 32);
  o.bB = lds128(bfr + c * 32 + 16);
  o.kq = lds128(kc);
}

// Four MMAs in two independent chains (steps 0, 1 and 2, 3), then the group
// fold s (P d - Q) + b sum x into rows g and g + 8.
__device__ __forceinline__ void unit_fold(const UnitOps& o, float& y0, float& y1) {
  uint32_t r0[4], r1[4], r2[4], r3[4];
  nib8_to_f16x2_offset(o.wv.x, r0);
  nib8_to_f16x2_offset(o.wv.y, r1);
  nib8_to_f16x2_offset(o.wv.z, r2);
  nib8_to_f16x2_offset(o.wv.w, r3);
  float da[4] = {0.f, 0.f, 0.f, 0.f}, db[4] = {0.f, 0.f, 0.f, 0.f};
  mma_16816(da, r0[0], r2[0], r0[1], r2[1], o.bA.x, o.bA.y);
  mma_16816(db, r1[0], r3[0], r1[1], r3[1], o.bB.x, o.bB.y);
  mma_16816(da, r0[2], r2[2], r0[3], r2[3], o.bA.z, o.bA.w);
  mma_16816(db, r1[2], r3[2], r1[3], r3[3], o.bB.z, o.bB.w);
  float sg0, bg0, sg1, bg1;
  f16x2_split(o.sb.x, sg0, bg0);
  f16x2_split(o.sb.y, sg1, bg1);
  const float P = __uint_as_float(o.kq.x), Q = __uint_as_float(o.kq.y), X = __uint_as_float(o.kq.z);
  y0 = fmaf(sg0, fmaf(P, da[0] + db[0], -Q), fmaf(bg0, X, y0));
  y1 = fmaf(sg1, fmaf(P, da[2] + db[2], -Q), fmaf(bg1, X, y1));
}

}  // namespace

// 288 threads (9 warps, at most 3 on one SM sub-partition), one CTA per SM: up
// to 168 registers a thread
__global__ void __maxnreg__(168) w4a16_chain_kernel(const ChainArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // shared layout: ring [ST][36864] | B fragments | fold constants | red [ST][8 warps][16 rows] f32 | barriers
  uint8_t* ring = smem;
  uint8_t* bfr = smem + (size_t)a.ST * kChStageBytes;
  uint8_t* kconst = bfr + a.bfr_bytes;
  float* red = reinterpret_cast<float*>(kconst + a.bfr_bytes / 8);
  uint64_t* bars = reinterpret_cast<uint64_t*>(red + (size_t)a.ST * kChWarps * 16);
  uint64_t* full = bars;
  uint64_t* empty = bars + a.ST;
  uint64_t* redfull = bars + 2 * a.ST;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kChWarps);
      mbar_init(&redfull[i], kChWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abortp = &abort_flag;
  const int s0 = a.cta_seg[blockIdx.x], s1 = a.cta_seg[blockIdx.x + 1];

  if (warp == kChWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int it = 0;
      bool ok = true;
      for (int si = s0; si < s1 && ok; ++si) {
        const ChainSeg sg = a.seg[si];
        const ChainProj& p = a.proj[sg.proj];
        const int G = p.K >> 6;
        for (int b = sg.b0; b < sg.b1 && ok; ++b) {
          for (int g0 = 0; g0 < G; g0 += kChStageGroups, ++it) {
            const int st = it % a.ST;
            if (it >= a.ST && !ch_wait(&empty[st], ((it / a.ST) & 1) ^ 1, a.err, kErrChainEmptyWait, abortp)) {
              ok = false;
              break;
            }
            const uint32_t bytes = (uint32_t)min(kChStageGroups, G - g0) * kChUnit;
            mbar_arrive_expect_tx(&full[st], bytes);
            bulk_g2s_evict_first(ring + (size_t)st * kChStageBytes,
                                 p.packed + ((size_t)b * G + g0) * kChUnit, bytes, &full[st], pol);
          }
        }
      }
      // drain: every issued copy must land before this CTA may exit
      for (int j = max(0, it - a.ST); j < it; ++j) mbar_wait(&full[j % a.ST], (j / a.ST) & 1, a.err, kErrChainDrain);
    }
  } else {
    // -------------------------------------------------------------- consumers
    const int w = warp;
    const int g = lane >> 2, c = lane & 3;
    const uint32_t ring_s = smem_u32(ring), bfr_s = smem_u32(bfr), kc_s = smem_u32(kconst), red_s = smem_u32(red);
    pdl_wait();  // inputs may come from the previous kernel on the stream
    int cur_proj = -1, waited = -1, it = 0;
    const void* cur_x = nullptr;
    int cur_op = -1, cur_K = 0, cur_level = -1;
    float cur_alpha = 0.f;
    uint32_t redpar = 0;  // parity of the next completion of redfull[st], bit st
    int tiles = 0;        // row blocks finished by this CTA; block t is summed by warp t % 8
    bool ok = true;
    for (int si = s0; si < s1 && ok; ++si) {
      const ChainSeg sg = a.seg[si];
      const ChainProj p = a.proj[sg.proj];
      if (w == 0 && lane == 0 && sg.level != cur_level) stamp(a.trace, a.nlevels, sg.level, 0, false);
      if (sg.level > 0 && waited < sg.level - 1) {
        bool got = true;
        if (lane == 0) got = wait_level(&a.cnt[sg.level - 1], (unsigned)a.level_tiles[sg.level - 1], a.err, abortp);
        got = __shfl_sync(0xffffffffu, got, 0);
        __syncwarp();  // lane 0's acquire orders the whole warp's input loads
        if (!got) {
          ok = false;
          break;
        }
        waited = sg.level - 1;
        if (w == 0 && lane == 0) stamp(a.trace, a.nlevels, sg.level, 1, false);
      }
      if (sg.proj != cur_proj) {
        // a new projection: new B fragments unless it reads the same input
        // (q, k and v of one layer) that the current ones were built from
        const bool same = cur_proj >= 0 && p.xsrc == cur_x && p.op == cur_op && p.alpha == cur_alpha &&
                          p.K == cur_K && sg.level == cur_level;
        if (!same) {
          build_x(p, w, lane, bfr_s, kc_s);
          __syncwarp();
          if (w == 0 && lane == 0) stamp(a.trace, a.nlevels, sg.level, 2, false);
        }
        cur_proj = sg.proj;
        cur_x = p.xsrc;
        cur_op = p.op;
        cur_alpha = p.alpha;
        cur_K = p.K;
        cur_level = sg.level;
      }
      const int G = p.K >> 6;
      for (int b = sg.b0; b < sg.b1 && ok; ++b) {
        float y0 = 0.f, y1 = 0.f;  // rows 16 b + g and 16 b + g + 8 (every lane holds them)
        for (int g0 = 0; g0 < G; g0 += kChStageGroups, ++it) {
          const int st = it % a.ST;
          if (!ch_wait(&full[st], (it / a.ST) & 1, a.err, kErrChainFullWait, abortp)) {
            ok = false;
            break;
          }
          const int gch = min(kChStageGroups, G - g0);
          const uint32_t sbase = ring_s + st * kChStageBytes;
          if (gch == kChStageGroups) {
            // full stage: this warp's eight groups, two at a time
#pragma unroll
            for (int j = 0; j < kChStageGroups / kChWarps; j += 2) {
              const int gl = w + kChWarps * j;
              UnitOps o0, o1;
              unit_load(o0, sbase + gl * kChUnit, bfr_s + (g0 + gl) * 128, kc_s + (g0 + gl) * 16, lane, g, c);
              unit_load(o1, sbase + (gl + kChWarps) * kChUnit, bfr_s + (g0 + gl + kChWarps) * 128,
                        kc_s + (g0 + gl + kChWarps) * 16, lane, g, c);
              unit_fold(o0, y0, y1);
              unit_fold(o1, y0, y1);
            }
          } else {
            for (int gl = w; gl < gch; gl += kChWarps) {
              UnitOps o;
              unit_load(o, sbase + gl * kChUnit, bfr_s + (g0 + gl) * 128, kc_s + (g0 + gl) * 16, lane, g, c);
              unit_fold(o, y0, y1);
            }
          }
          if (g0 + kChStageGroups >= G) {
            // end of the row block: partial rows of every warp, summed in warp
            // order by warp (block count % 8)
            const uint32_t rb = red_s + st * kChRedBytes;
            if (c == 0) {
              asm volatile("st.shared.f32 [%0], %1;" ::"r"(rb + (w * 16 + g) * 4), "f"(y0) : "memory");
              asm volatile("st.shared.f32 [%0], %1;" ::"r"(rb + (w * 16 + g + 8) * 4), "f"(y1) : "memory");
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&redfull[st]);
            const uint32_t rp = (redpar >> st) & 1u;
            redpar ^= 1u << st;
            if (w == (tiles & (kChWarps - 1))) {
              if (!ch_wait(&redfull[st], rp, a.err, kErrChainFullWait, abortp)) {
                ok = false;
                break;
              }
              const int row = 16 * b + lane;
              if (lane < 16 && row < p.N) {
                float tot = 0.f;
#pragma unroll
                for (int ww = 0; ww < kChWarps; ++ww) {
                  float v;
                  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(rb + (ww * 16 + lane) * 4));
                  tot += v;
                }
                p.y[row] = tot;
              }
              __syncwarp();  // the lanes' stores precede lane 0's release below
              if (b == sg.b1 - 1 && lane == 0) {
                asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(&a.cnt[sg.level]),
                             "r"((unsigned)(sg.b1 - sg.b0))
                             : "memory");
                stamp(a.trace, a.nlevels, sg.level, 3, true);
              }
            }
            ++tiles;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[st]);
        }
      }
    }
    if (!ok) *abortp = 1;
  }
  __syncwarp();
  __syncthreads();
  // the last CTA to finish returns the counters to zero for the next run
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(&a.cnt[a.nlevels], 1u);
    if (prev == gridDim.x - 1) {
      for (int l = 0; l < a.nlevels; ++l) atomicExch(&a.cnt[l], 0u);
      __threadfence();
      atomicExch(&a.cnt[a.nlevels], 0u);
    }
  }
}

// Copy one projection into the fragment-major layout: one warp per 16-row x
// 64-k unit. Codes of rows past N and their scales and biases are zero.
__global__ void __launch_bounds__(256) w4a16_chain_repack_kernel(const uint32_t* wq, const uint16_t* sc,
                                                                 const uint16_t* bi, int N, int K, uint8_t* out) {
  const int G = K >> 6;
  const long long unit = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const long long units = (long long)((N + 15) / 16) * G;
  if (unit >= units) return;
  const int lane = threadIdx.x & 31;
  const int b = (int)(unit / G), gi = (int)(unit % G);
  const int g = lane >> 2, c = lane & 3;
  uint32_t wout[4];
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    const int r = 16 * b + g + 8 * (wi >> 1);  // words 0, 1: row g; 2, 3: row g + 8
    const int half = wi & 1;                   // MMA steps 2 half, 2 half + 1
    uint32_t word = 0;
    if (r < N) {
      const uint32_t* row = wq + (size_t)r * (K / 8);
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        // nibble n of the word: t = n & 3 picks the (step, slot pair): t = 0, 2 the
        // slots 2c, 2c + 1 of steps 2 half, 2 half + 1; t = 1, 3 the slots 2c + 8, + 9
        // (n >> 2 the second of the pair), read back by the decode as (1024 + q)
        // (t even) and (1024 + 16 q) (t odd)
        const int t = n & 3;
        const int k = 64 * gi + 32 * half + 16 * (t >> 1) + 8 * (t & 1) + 2 * c + (n >> 2);
        word |= ((row[k >> 3] >> (4 * (k & 7))) & 0xFu) << (4 * n);
      }
    }
    wout[wi] = word;
  }
  uint8_t* u = out + (size_t)unit * kChUnit;
  *reinterpret_cast<uint4*>(u + lane * 16) = make_uint4(wout[0], wout[1], wout[2], wout[3]);
  if (lane < 8) {
    const int r0 = 16 * b + lane, r1 = r0 + 8;
    const uint32_t s0 = r0 < N ? sc[(size_t)r0 * G + gi] : 0u, b0 = r0 < N ? bi[(size_t)r0 * G + gi] : 0u;
    const uint32_t s1 = r1 < N ? sc[(size_t)r1 * G + gi] : 0u, b1 = r1 < N ? bi[(size_t)r1 * G + gi] : 0u;
    *reinterpret_cast<uint2*>(u + 512 + 8 * lane) = make_uint2(s0 | (b0 << 16), s1 | (b1 << 16));
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
bool chain_proj_ok(int N, int K) { return N >= 1 && K >= 64 && K % 64 == 0 && K <= kChainMaxK; }

size_t chain_packed_bytes(int N, int K) { return (size_t)((N + 15) / 16) * (size_t)(K / 64) * kChUnit; }

cudaError_t chain_plan_build(const ChainItem* items, int n, int sms, ChainPlan* out) {
  ChainPlan p{};
  // levels: renumbered 0.. in order of first appearance (the list is level-sorted)
  std::vector<int> lev(n);
  int nlevels = 0;
  for (int i = 0; i < n; ++i) {
    if (i == 0 || items[i].level != items[i - 1].level) ++nlevels;
    lev[i] = nlevels - 1;
  }
  std::vector<size_t> off(n + 1, 0);
  int maxK = 64;
  for (int i = 0; i < n; ++i) {
    off[i + 1] = off[i] + chain_packed_bytes(items[i].N, items[i].K);
    maxK = std::max(maxK, items[i].K);
  }
  const int grid = std::max(1, sms);
  // Tiles (one 16-row block of one projection, cost K) are handed out level by
  // level: a level completes when its slowest CTA is done, so each level's
  // tiles are split on their own into `grid` contiguous runs of equal cost
  // (ends at the nearest tile boundary), and run r goes to CTA (r + rot) % grid
  // with rot advancing by a step coprime to the grid, so that the CTAs taking
  // one tile more than the others change from level to level. A CTA's tiles
  // of one projection are consecutive (one segment).
  std::vector<std::vector<ChainSeg>> per(grid);
  std::vector<int> level_tiles(nlevels, 0);
  int rot = 0, step = grid / 2 + 1;
  while (step > 1 && std::gcd(step, grid) != 1) --step;
  for (int i0 = 0; i0 < n;) {
    int i1 = i0;
    while (i1 < n && lev[i1] == lev[i0]) ++i1;
    std::vector<int> tp, tb;  // the level's tiles: projection, block
    std::vector<double> prefix{0.0};
    for (int i = i0; i < i1; ++i)
      for (int b = 0; b < (items[i].N + 15) / 16; ++b) {
        tp.push_back(i);
        tb.push_back(b);
        prefix.push_back(prefix.back() + items[i].K);
      }
    const int T = (int)tp.size();
    level_tiles[lev[i0]] = T;
    int t = 0;
    for (int r = 0; r < grid; ++r) {
      const double end_cost = prefix[T] * (r + 1) / grid;
      int e = (int)(std::lower_bound(prefix.begin(), prefix.end(), end_cost) - prefix.begin());
      if (e > T) e = T;
      if (e > 0 && end_cost - prefix[e - 1] < prefix[e] - end_cost) --e;  // nearest boundary
      if (r == grid - 1) e = T;
      e = std::max(e, t);
      auto& v = per[(r + rot) % grid];
      for (; t < e; ++t) {
        if (!v.empty() && v.back().proj == tp[t] && v.back().b1 == tb[t])
          v.back().b1 = tb[t] + 1;
        else
          v.push_back(ChainSeg{tp[t], tb[t], tb[t] + 1, lev[tp[t]]});
      }
    }
    rot = (rot + step) % grid;
    i0 = i1;
  }
  std::vector<ChainSeg> segs;
  std::vector<int> cta(grid + 1, 0);
  for (int c = 0; c < grid; ++c) {
    cta[c] = (int)segs.size();
    segs.insert(segs.end(), per[c].begin(), per[c].end());
  }
  cta[grid] = (int)segs.size();

  p.nproj = n;
  p.nlevels = nlevels;
  p.grid = grid;
  p.bfr_bytes = (uint32_t)(maxK / 64) * 128u;
  const size_t fixed = (size_t)p.bfr_bytes + p.bfr_bytes / 8;
  const size_t per_stage = kChStageBytes + kChRedBytes + 3 * 8;
  const size_t budget = (size_t)device_max_smem_optin() - 256;  // static shared: the abort flag
  if (budget < fixed + 2 * per_stage) return cudaErrorInvalidValue;
  p.ST = (int)std::min<size_t>(8, (budget - fixed) / per_stage);
  p.smem = fixed + (size_t)p.ST * per_stage;
  p.packed_bytes = off[n];

  cudaError_t e = cudaMalloc(&p.d_packed, off[n]);
  if (e == cudaSuccess) e = cudaMalloc(&p.d_proj, sizeof(ChainProj) * n);
  if (e == cudaSuccess) e = cudaMalloc(&p.d_seg, sizeof(ChainSeg) * std::max<size_t>(1, segs.size()));
  if (e == cudaSuccess) e = cudaMalloc(&p.d_cta, sizeof(int) * (grid + 1));
  if (e == cudaSuccess) e = cudaMalloc(&p.d_ltiles, sizeof(int) * nlevels);
  if (e == cudaSuccess) e = cudaMalloc(&p.d_cnt, sizeof(unsigned) * (nlevels + 1));
  std::vector<ChainProj> proj(n);
  for (int i = 0; i < n && e == cudaSuccess; ++i) {
    const ChainItem& it = items[i];
    ChainProj& q = proj[i];
    q.packed = p.d_packed + off[i];
    q.xsrc = it.xsrc;
    q.y = it.y;
    q.alpha = it.alpha;
    q.op = it.op;
    q.N = it.N;
    q.K = it.K;
    q.level = lev[i];
    const long long units = (long long)((it.N + 15) / 16) * (it.K / 64);
    w4a16_chain_repack_kernel<<<(unsigned)((units + 7) / 8), 256>>>(it.wq, it.scales, it.biases, it.N, it.K,
                                                                   p.d_packed + off[i]);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaMemcpy(p.d_proj, proj.data(), sizeof(ChainProj) * n, cudaMemcpyHostToDevice);
  if (e == cudaSuccess && !segs.empty())
    e = cudaMemcpy(p.d_seg, segs.data(), sizeof(ChainSeg) * segs.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(p.d_cta, cta.data(), sizeof(int) * (grid + 1), cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(p.d_ltiles, level_tiles.data(), sizeof(int) * nlevels, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(p.d_cnt, 0, sizeof(unsigned) * (nlevels + 1));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    chain_plan_free(&p);
    return e;
  }
  *out = p;
  return cudaSuccess;
}

void chain_plan_free(ChainPlan* p) {
  cudaFree(p->d_packed);
  cudaFree(p->d_proj);
  cudaFree(p->d_seg);
  cudaFree(p->d_cta);
  cudaFree(p->d_ltiles);
  cudaFree(p->d_cnt);
  cudaFree(p->d_trace);
  *p = ChainPlan{};
}

cudaError_t chain_launch(const ChainPlan& p, uint32_t* err, cudaStream_t stream) {
  ChainArgs a;
  a.proj = p.d_proj;
  a.seg = p.d_seg;
  a.cta_seg = p.d_cta;
  a.level_tiles = p.d_ltiles;
  a.cnt = p.d_cnt;
  a.nlevels = p.nlevels;
  a.ST = p.ST;
  a.bfr_bytes = p.bfr_bytes;
  a.err = err;
  a.trace = p.d_trace;
  cudaError_t e = allow_max_smem(w4a16_chain_kernel);
  if (e != cudaSuccess) return e;
  // every CTA must be resident at once (CTAs wait for each other's levels):
  // a cooperative launch, which the driver refuses rather than run partially
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kChThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, w4a16_chain_kernel, a);
}

cudaError_t chain_set_trace(ChainPlan* p, bool enable) {
  if (!enable) {
    cudaError_t e = cudaFree(p->d_trace);
    p->d_trace = nullptr;
    return e;
  }
  if (p->d_trace) return cudaSuccess;
  const size_t bytes = sizeof(unsigned long long) * (size_t)p->grid * p->nlevels * 4;
  cudaError_t e = cudaMalloc(&p->d_trace, bytes);
  if (e == cudaSuccess) e = cudaMemset(p->d_trace, 0, bytes);
  return e;
}

}  // namespace qg
