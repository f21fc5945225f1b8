// W8A8 int32 GEMM on the tensor cores through exact fp16 operands, M <= 16.
//
// C[m][n] = sum_k a[m][k] w[n][k] with int8 a, w ("How Uzu optimizes bytes and
// tokens per pass": 8-bit activations on the int8 matrix path, 16 verify rows).
// The int8 mma.sync path of GB300 measured 252 MAC/clk/SM, so the products run
// on the f16 path instead, exactly:
//  * A weight byte b becomes the fp16 1024 + (b + 128) with one xor and one
//    byte permute per two bytes (fp16 has an ulp of 1 in [1024, 2048)); an
//    activation becomes its own value in fp16 (|a| <= 128, exact).
//  * mma.sync.m16n8k16 (f16 in, fp32 accumulate) sums (1152 + b) a over a 64-k
//    group starting from -1152 sum a, so it ends at sum b a; every partial
//    sum is an integer below 2^24 in magnitude (1152 * 64 * 128 + 64 * 128^2),
//    hence exact in fp32, and is moved into an int32 accumulator per group.
//  * Layout as in the skinny W4A16 MMA kernel: one persistent CTA per SM, a
//    producer warp loads per 512-k stage the codes of 128 weight rows and the
//    stage's activations (128B-swizzled TMA tiles); warp w of 8 consumer warps
//    owns 64-k group w of every stage and all 128 rows (eight 16-row blocks)
//    and builds the group's B fragments from the landed activations once per
//    stage. The warps' partial tiles are added through shared memory and the
//    row tile's int32 results added into C with integer atomics (exact in any
//    order), so K may be split over CTAs; C is cleared before the launch.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

namespace {

constexpr int kW8Rows = 128;                          // weight rows (output columns) per tile
constexpr int kW8StageK = 512;                        // k per stage
constexpr int kW8Warps = 8;                           // consumer warps = 64-k groups per stage
constexpr int kW8Threads = 32 * (kW8Warps + 1);       // + the producer warp
constexpr uint32_t kW8Codes = kW8Rows * kW8StageK;    // 64 KB: [4 chunks][128 rows][128 B]
constexpr uint32_t kW8Acts = 16 * kW8StageK;          // 8 KB: [4 chunks][16 rows][128 B]
constexpr uint32_t kW8Stage = kW8Codes + kW8Acts;
constexpr uint32_t kW8Red = kW8Warps * 16 * 32 * 16;  // 64 KB: int32 partial tiles of all warps

struct W8MmaArgs {
  int32_t* c;
  int M, N, K;
  int ntiles, splits, kper, nunits, ST;
  uint32_t* err;
};

__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* tm, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// d = A B + C with C = (c0, c1) for both row halves (first k-step of a group)
__device__ __forceinline__ void mma16816_from(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1, float c0, float c1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %11, %10, %11};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void mma16816_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// four int8 weights (byte j = weight j) -> fp16 pairs (1152 + w0, 1152 + w1), (1152 + w2, 1152 + w3)
__device__ __forceinline__ void w8_to_f16x2_offset(uint32_t word, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = word ^ 0x80808080u;  // signed byte b -> b + 128 in 0..255
  lo = __byte_perm(u, 0x64646464u, 0x4140);  // bytes u0, 0x64, u1, 0x64: fp16 1024 + u
  hi = __byte_perm(u, 0x64646464u, 0x4342);
}

// four int8 activations -> exact fp16 pairs (a0, a1), (a2, a3): the offset form
// above minus 1152 (exact: integers below 2048 in magnitude)
__device__ __forceinline__ void a8_to_f16x2(uint32_t word, uint32_t& lo, uint32_t& hi) {
  uint32_t l, h;
  w8_to_f16x2_offset(word, l, h);
  constexpr uint32_t k1152 = 0x64806480u;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(l), "r"(k1152));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(h), "r"(k1152));
}

// D += A B in int32: m16n8k32, s8 operands (row-major A, column-major B)
__device__ __forceinline__ void mma16832_s8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                            uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace

__global__ void __launch_bounds__(kW8Threads, 1)
    w8a8_mma_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_a,
                    const W8MmaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  // shared layout: stages | red (64 KB) | barriers
  int32_t* red = reinterpret_cast<int32_t*>(gbase + a.ST * kW8Stage);
  uint64_t* full = reinterpret_cast<uint64_t*>(gbase + a.ST * kW8Stage + kW8Red);
  uint64_t* empty = full + a.ST;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kW8Warps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();  // C is cleared and a written before this kernel
  const int nstage = a.kper / kW8StageK;

  if (warp == kW8Warps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < a.nunits && ok; u += gridDim.x) {
        const int n0 = (u / a.splits) * kW8Rows, k0 = (u % a.splits) * a.kper;
        for (int s = 0; s < nstage; ++s) {
          const int st = issued % a.ST;
          if (issued >= a.ST) ok = mbar_wait(&empty[st], ((issued / a.ST) & 1) ^ 1, a.err, kErrGemvEmptyWait);
          if (!ok) break;
          const uint32_t sb = base + st * kW8Stage;
          mbar_arrive_expect_tx(&full[st], kW8Stage);
          const int kc = (k0 + s * kW8StageK) / 128;  // first 128-byte chunk of the stage
          tma_3d(sb, &tm_w, 0, n0, kc, &full[st]);
          tma_3d(sb + kW8Codes, &tm_a, 0, 0, kc, &full[st]);
          ++issued;
        }
      }
      for (int j = max(0, issued - a.ST); j < issued; ++j)
        mbar_wait(&full[j % a.ST], (j / a.ST) & 1, a.err, kErrGemvDrain);
    }
  } else {
    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, c = lane & 3;
    // the 16 bytes of group `warp` this lane reads in every 128-byte row: unit 4 (warp % 2) + c
    const uint32_t unit = 4u * (uint32_t)(warp & 1) + (uint32_t)c;
    const uint32_t chunk = (uint32_t)(warp >> 1);
    int sgc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < a.nunits; u += gridDim.x) {
      const int n0 = (u / a.splits) * kW8Rows;
      int yi[8][2][4];
#pragma unroll
      for (int rb = 0; rb < 8; ++rb)
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int e = 0; e < 4; ++e) yi[rb][t][e] = 0;
      for (int s = 0; s < nstage; ++s, ++sgc) {
        const int st = sgc % a.ST;
        if (ok) ok = mbar_wait(&full[st], (sgc / a.ST) & 1, a.err, kErrGemvFullWait);
        const uint32_t sb = base + st * kW8Stage;
        if (ok) {
          // B fragments of this group: activation rows g (tile 0) and g + 8 (tile 1),
          // k = 16c .. 16c + 15 of the group; step s4 uses k 16c + 4 s4 .. + 3
          uint32_t b[16];
          int asum[2];
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int n = g + 8 * t;
            const uint4 v = lds128(sb + kW8Codes + chunk * 2048 + n * 128 + ((unit ^ (uint32_t)(n & 7)) << 4));
            const uint32_t wds[4] = {v.x, v.y, v.z, v.w};
            int sa = 0;
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
              a8_to_f16x2(wds[s4], b[(s4 * 2 + t) * 2], b[(s4 * 2 + t) * 2 + 1]);
              sa = __dp4a((int)wds[s4], 0x01010101, sa);
            }
            sa += __shfl_xor_sync(0xFFFFFFFFu, sa, 1);
            sa += __shfl_xor_sync(0xFFFFFFFFu, sa, 2);
            asum[t] = sa;  // sum of a over the group for activation row n
          }
          // accumulator start per output column (activation row 8t + 2c, + 1): -1152 sum a
          float c0[2], c1[2];
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            c0[t] = -1152.f * (float)__shfl_sync(0xFFFFFFFFu, asum[t], 8 * c);
            c1[t] = -1152.f * (float)__shfl_sync(0xFFFFFFFFu, asum[t], 8 * c + 4);
          }
          const uint32_t cbase = sb + chunk * 16384;
#pragma unroll
          for (int rb = 0; rb < 8; ++rb) {
            const int r0 = 16 * rb + g;  // rows r0 and r0 + 8 share the swizzle (r & 7 = g)
            const uint32_t sw = (unit ^ (uint32_t)g) << 4;
            const uint4 w0 = lds128(cbase + r0 * 128 + sw);
            const uint4 w1 = lds128(cbase + (r0 + 8) * 128 + sw);
            const uint32_t x0[4] = {w0.x, w0.y, w0.z, w0.w}, x1[4] = {w1.x, w1.y, w1.z, w1.w};
            float acc[2][4];
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
              uint32_t a0l, a0h, a1l, a1h;
              w8_to_f16x2_offset(x0[s4], a0l, a0h);
              w8_to_f16x2_offset(x1[s4], a1l, a1h);
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                if (s4 == 0)
                  mma16816_from(acc[t], a0l, a1l, a0h, a1h, b[t * 2], b[t * 2 + 1], c0[t], c1[t]);
                else
                  mma16816_acc(acc[t], a0l, a1l, a0h, a1h, b[(s4 * 2 + t) * 2], b[(s4 * 2 + t) * 2 + 1]);
              }
            }
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
              for (int e = 0; e < 4; ++e) yi[rb][t][e] += __float2int_rn(acc[t][e]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
      // the 8 warps' partial tiles -> one tile (integers: any order is exact), added into C
      {
        int4* rv = reinterpret_cast<int4*>(red);
#pragma unroll
        for (int rb = 0; rb < 8; ++rb)
#pragma unroll
          for (int t = 0; t < 2; ++t)
            rv[(warp * 16 + rb * 2 + t) * 32 + lane] = make_int4(yi[rb][t][0], yi[rb][t][1], yi[rb][t][2], yi[rb][t][3]);
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      {
        const int et = threadIdx.x;  // 0..255: lane et % 32 of units 2 (et / 32), + 1
        const int ln = et & 31, u0 = 2 * (et >> 5);
        const int gg = ln >> 2, cc = ln & 3;
        const int4* rv = reinterpret_cast<const int4*>(red);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          int tot[4] = {0, 0, 0, 0};
#pragma unroll
          for (int w2 = 0; w2 < kW8Warps; ++w2) {
            const int4 v = rv[(w2 * 16 + u0 + h) * 32 + ln];
            tot[0] += v.x;
            tot[1] += v.y;
            tot[2] += v.z;
            tot[3] += v.w;
          }
          const int uu = u0 + h, rb = uu >> 1, t = uu & 1;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int n = n0 + 16 * rb + gg + 8 * (e >> 1);
            const int m = 8 * t + 2 * cc + (e & 1);
            if (m < a.M && n < a.N) atomicAdd(&a.c[(size_t)m * a.N + n], tot[e]);
          }
        }
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
    }
  }
  __syncthreads();
  pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// Fused: Hadamard -> int8 -> W8A8 -> dequant in one launch (w8a8_fused_kernel)
//
// y[m][n] = C[m][n] s_a[m] s_w[n] / 32 with (q_a, s_a) the block-32 randomized
// Hadamard + per-row int8 of x (bit-exact with hadamard32_quant_i8) and C =
// q_a w^T exact -- the whole int8 path of the Uzu article's "How Uzu optimizes
// bytes and tokens per pass", with no int8 round trip through a separate
// quantizer launch and no cleared accumulator.
//
// One cooperative launch, one CTA per SM (8 consumer warps + 1 producer warp):
//  1. transform: the M x K/32 blocks are split over the CTAs; a warp takes a
//     block (one element per lane, the five butterflies as shuffles in the
//     fixed order), the CTA's per-row maxima of |z| are taken in shared memory
//     and then into the rows' maxima in the workspace (an integer max on the
//     float bits: exact, any order). Grid barrier.
//  2. quantize: every CTA reads the M row maxima, s = max / 127 and q =
//     rint(z / s) (IEEE divisions), and writes its blocks' codes to the
//     workspace already in the order the product reads them. Grid barrier.
//  3. every CTA copies all of q_a (M <= 16 rows, 64 KB at K = 4096) into
//     shared memory with one bulk copy.
//  4. product: tiles of 16 weight rows x the whole K, one contiguous range of
//     tiles per CTA; a tile is one ring stage, 16 bulk copies of one row each
//     into rows padded to K + 64 bytes (every shared read conflict-free), and
//     the producer warp streams tiles from the start of the launch, so the
//     weight stream overlaps steps 1-3. Per 64-k group a warp runs four int8
//     mma.sync.m16n8k32 (weights and codes as stored, int32 accumulation:
//     exact, nothing to convert); at the end of a tile the 8 warps' int32
//     partials are added through shared memory (two buffers, one barrier per
//     tile) and each thread writes one y = float(C) s_a s_w / 32.
// The last CTA to finish zeroes the row maxima and the barrier counters, so the
// workspace stays ready for the next call.
// ---------------------------------------------------------------------------
namespace {

constexpr int kFzRows = 16;                             // weight rows per tile (= per stage)
constexpr int kFzMaxK = 4096;
constexpr uint32_t kFzQa = (kFzMaxK / 64) * 1024;       // q_a: [group][row g, g + 8][32 lanes][16 B]
constexpr uint32_t kFzRed = 2 * kW8Warps * 32 * 8 * 4;  // int32 partial tiles of the 8 warps, two buffers
constexpr unsigned long long kFzWaitNs = 1000000000ull;

struct W8FusedArgs {
  const uint16_t* x;
  const uint32_t* sign_bits;
  const int8_t* w;
  const float* sw;
  float* y;
  uint32_t* amax;   // [16] row maxima (float bits), zero between calls
  uint32_t* cnt;    // [4]: grid barriers 1 and 2, CTAs finished
  int8_t* qa;       // codes in product order, [K / 64][2][32][16]
  int M, N, K, ntiles, ST;
  int zcap;         // transformed blocks a CTA keeps: ceil(M K / 32 / grid)
  uint32_t pitch;   // shared row pitch of a tile: K + 64 bytes
  uint32_t* err;
};

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// grid barrier over all CTAs (cooperative launch): the consumer warps of a CTA
// have synchronized before thread 0 arrives; a bounded wait
__device__ __forceinline__ bool fz_grid_barrier(uint32_t* cnt, uint32_t* err) {
  __shared__ int ok_s;
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(cnt) : "memory");
    const uint64_t t0 = gtimer();
    int ok = 1;
    for (uint32_t i = 0;; ++i) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
      if (v >= gridDim.x) break;
      if ((i & 63) == 63 && gtimer() - t0 > kFzWaitNs) {
        report_error(err, kErrW8FusedBarrier);
        ok = 0;
        break;
      }
      if (i > 256) __nanosleep(32);
    }
    ok_s = ok;
  }
  asm volatile("bar.sync 1, 256;" ::: "memory");
  return ok_s != 0;
}

// one 64-k group for one lane: rows g, g + 8 of the tile, x rows g, g + 8
__device__ __forceinline__ void fz_group(int (&y0)[4], int (&y1)[4], uint32_t sb, uint32_t pitch, uint32_t qs,
                                         int gi, int g, int c, int lane) {
  const uint4 w0 = lds128(sb + g * pitch + gi * 64 + 16 * c);
  const uint4 w1 = lds128(sb + (g + 8) * pitch + gi * 64 + 16 * c);
  const uint4 q0 = lds128(qs + gi * 1024 + lane * 16);
  const uint4 q1 = lds128(qs + gi * 1024 + 512 + lane * 16);
  // two k = 32 steps: the lane's 16 bytes are (a0, a2) of step 0 and of step 1
  // for its rows, and the same bytes of the x rows are (b0, b1)
  mma16832_s8(y0, w0.x, w1.x, w0.y, w1.y, q0.x, q0.y);
  mma16832_s8(y1, w0.x, w1.x, w0.y, w1.y, q1.x, q1.y);
  mma16832_s8(y0, w0.z, w1.z, w0.w, w1.w, q0.z, q0.w);
  mma16832_s8(y1, w0.z, w1.z, w0.w, w1.w, q1.z, q1.w);
}

}  // namespace

__global__ void __launch_bounds__(kW8Threads, 1) w8a8_fused_kernel(const W8FusedArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float s_row[16];
  __shared__ unsigned cta_max[16];
  __shared__ __align__(8) uint64_t qbar;
  // shared layout: ring [ST][16 rows][K + 64] | q_a | red x 2 | barriers | z blocks
  const uint32_t stage_bytes = kFzRows * a.pitch;
  const uint32_t base = smem_u32(smem);
  const uint32_t qs = base + a.ST * stage_bytes;
  int32_t* red = reinterpret_cast<int32_t*>(smem + (size_t)a.ST * stage_bytes + kFzQa);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)a.ST * stage_bytes + kFzQa + kFzRed);
  uint64_t* empty = full + a.ST;
  float* zb = reinterpret_cast<float*>(smem + (size_t)a.ST * stage_bytes + kFzQa + kFzRed + 16 * a.ST);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = a.K, M = a.M, G = a.K / 64;
  const int t0 = (int)((long long)a.ntiles * blockIdx.x / gridDim.x);
  const int t1 = (int)((long long)a.ntiles * (blockIdx.x + 1) / gridDim.x);
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kW8Warps);
    }
    mbar_init(&qbar, 1);
    fence_mbar_init();
  }
  if (threadIdx.x < 16) cta_max[threadIdx.x] = 0u;
  __syncthreads();

  if (warp == kW8Warps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      bool ok = true;
      for (int t = t0; t < t1 && ok; ++t, ++issued) {
        const int st = issued % a.ST;
        if (issued >= a.ST) ok = mbar_wait(&empty[st], ((issued / a.ST) & 1) ^ 1, a.err, kErrGemvEmptyWait);
        if (!ok) break;
        const int rows = min(kFzRows, a.N - t * kFzRows);
        mbar_arrive_expect_tx(&full[st], (uint32_t)rows * K);
        uint8_t* dst = smem + (size_t)st * stage_bytes;
        for (int r = 0; r < rows; ++r)
          bulk_g2s_evict_first(dst + r * a.pitch, a.w + (size_t)(t * kFzRows + r) * K, K, &full[st], pol);
      }
      for (int j = max(0, issued - a.ST); j < issued; ++j)
        mbar_wait(&full[j % a.ST], (j / a.ST) & 1, a.err, kErrGemvDrain);
    }
  } else {
    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, c = lane & 3;
    bool ok = true;
    // 1. transform this CTA's blocks, row maxima
    const int nblk = M * (K / 32);
    const int b0 = (int)((long long)nblk * blockIdx.x / gridDim.x);
    const int b1 = (int)((long long)nblk * (blockIdx.x + 1) / gridDim.x);
    for (int j = b0 + warp, i = warp; j < b1; j += kW8Warps, i += kW8Warps) {
      const int m = j / (K / 32), kb = j % (K / 32);
      float v = bf16_bits_to_f32(a.x[(size_t)m * K + 32 * kb + lane]);
      if ((a.sign_bits[kb] >> lane) & 1u) v = -v;
#pragma unroll
      for (int h = 1; h < 32; h <<= 1) {
        const float p = __shfl_xor_sync(0xffffffffu, v, h);
        v = (lane & h) ? __fsub_rn(p, v) : __fadd_rn(v, p);
      }
      zb[32 * i + lane] = v;
      float mx = fabsf(v);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (lane == 0) atomicMax(&cta_max[m], __float_as_uint(mx));
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (threadIdx.x < M && cta_max[threadIdx.x] != 0u) atomicMax(&a.amax[threadIdx.x], cta_max[threadIdx.x]);
    asm volatile("bar.sync 1, 256;" ::: "memory");
    ok = fz_grid_barrier(&a.cnt[0], a.err);
    // 2. scales and this CTA's codes, written in product order: code (m, k) at
    //    group k / 64, half m / 8, lane 4 (m % 8) + (k % 64) / 16, byte k % 16
    if (threadIdx.x < 16) {
      unsigned bits;
      asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(bits) : "l"(&a.amax[threadIdx.x]) : "memory");
      s_row[threadIdx.x] = __fdiv_rn(__uint_as_float(bits), 127.0f);
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (ok) {
      for (int j = b0 + warp, i = warp; j < b1; j += kW8Warps, i += kW8Warps) {
        const int m = j / (K / 32), kb = j % (K / 32);
        const float sc = s_row[m];
        int8_t code = 0;
        if (sc > 0.f) {
          float r = rintf(__fdiv_rn(zb[32 * i + lane], sc));
          r = fminf(fmaxf(r, -127.f), 127.f);
          code = (int8_t)(int)r;
        }
        const int k = 32 * kb + lane;
        a.qa[(size_t)(k >> 6) * 1024 + (m >> 3) * 512 + (((m & 7) << 2) + ((k >> 4) & 3)) * 16 + (k & 15)] = code;
      }
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (ok) ok = fz_grid_barrier(&a.cnt[1], a.err);
    // 3. all of q_a into shared memory: one bulk copy (the codes of the other
    //    CTAs were published before the barrier; the copy reads them through
    //    the async proxy)
    if (threadIdx.x == 0 && ok) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      mbar_arrive_expect_tx(&qbar, (uint32_t)G * 1024);
      bulk_g2s(smem + (size_t)a.ST * stage_bytes, a.qa, (uint32_t)G * 1024, &qbar);
    }
    if (ok) ok = mbar_wait(&qbar, 0, a.err, kErrGemvFullWait);
    // 4. the product
    int tile_i = 0;
    for (int t = t0; t < t1; ++t, ++tile_i) {
      const int st = tile_i % a.ST;
      // four independent accumulator pairs (groups gi, gi + 8, gi + 16, gi + 24
      // of a round), so four MMA chains are in flight per warp
      int ya[4][2][4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int e = 0; e < 4; ++e) ya[u][0][e] = ya[u][1][e] = 0;
      if (ok) ok = mbar_wait(&full[st], (tile_i / a.ST) & 1, a.err, kErrGemvFullWait);
      if (ok) {
        const uint32_t sb = base + st * stage_bytes;
        int gi = warp;
        for (; gi + 3 * kW8Warps < G; gi += 4 * kW8Warps) {
#pragma unroll
          for (int u = 0; u < 4; ++u) fz_group(ya[u][0], ya[u][1], sb, a.pitch, qs, gi + u * kW8Warps, g, c, lane);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (gi + u * kW8Warps < G) fz_group(ya[u][0], ya[u][1], sb, a.pitch, qs, gi + u * kW8Warps, g, c, lane);
      }
      int y0[4], y1[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        y0[e] = (ya[0][0][e] + ya[1][0][e]) + (ya[2][0][e] + ya[3][0][e]);
        y1[e] = (ya[0][1][e] + ya[1][1][e]) + (ya[2][1][e] + ya[3][1][e]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      // the 8 warps' partial tiles added in warp order, then y = C s_a s_w / 32;
      // two buffers, so one barrier per tile orders both the writes before the
      // reads and this tile's reads before the next-but-one tile's writes
      int32_t* rt = red + (tile_i & 1) * (kW8Warps * 32 * 8);
      {
        int4* rv = reinterpret_cast<int4*>(rt);
        rv[(warp * 32 + lane) * 2] = make_int4(y0[0], y0[1], y0[2], y0[3]);
        rv[(warp * 32 + lane) * 2 + 1] = make_int4(y1[0], y1[1], y1[2], y1[3]);
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      {
        // thread -> (row r of the tile, x row m): fragment lane and element
        const int r = threadIdx.x >> 4, m = threadIdx.x & 15;
        const int tt = m >> 3, col = m & 7;
        const int L = ((r & 7) << 2) | (col >> 1);
        const int e = ((r >> 3) << 1) | (col & 1);
        int tot = 0;
#pragma unroll
        for (int w2 = 0; w2 < kW8Warps; ++w2) tot += rt[((w2 * 32 + L) * 2 + tt) * 4 + e];
        const int n = t * kFzRows + r;
        if (ok && m < M && n < a.N) a.y[(size_t)m * a.N + n] = (float)tot * s_row[m] * (a.sw[n] * 0.03125f);
      }
    }
  }
  __syncwarp();
  __syncthreads();
  // the last CTA to finish leaves the workspace zeroed for the next call
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(&a.cnt[2], 1u);
    if (prev == gridDim.x - 1) {
      for (int i = 0; i < 16; ++i) atomicExch(&a.amax[i], 0u);
      atomicExch(&a.cnt[0], 0u);
      atomicExch(&a.cnt[1], 0u);
      __threadfence();
      atomicExch(&a.cnt[2], 0u);
    }
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
bool w8a8_mma_ok(int M, int N, int K) {
  return M >= 1 && M <= 16 && N >= kW8Rows && K >= kW8StageK && K % kW8StageK == 0;
}

cudaError_t launch_w8a8_mma(const int8_t* a8, const int8_t* w8, int32_t* c, int M, int N, int K, uint32_t* err,
                            cudaStream_t stream, bool pdl) {
  const int sms = device_sm_count();
  W8MmaArgs a{};
  a.c = c;
  a.M = M;
  a.N = N;
  a.K = K;
  a.err = err;
  a.ntiles = (N + kW8Rows - 1) / kW8Rows;
  const int kstages = K / kW8StageK;
  // split K while twice the units still fit the SMs (integer atomics add the splits)
  a.splits = 1;
  while (a.ntiles * a.splits * 2 <= sms && kstages % (a.splits * 2) == 0) a.splits *= 2;
  a.kper = K / a.splits;
  a.nunits = a.ntiles * a.splits;
  a.ST = 2;
  const size_t smem = 1024 + (size_t)a.ST * kW8Stage + kW8Red + 16 * (size_t)a.ST;
  CUtensorMap tm_w, tm_a;
  // weights {128 B, N rows, K / 128 chunks} in [4][128][128 B] boxes; activations
  // {128 B, M rows, K / 128 chunks} in [4][16][128 B] boxes (rows past M read as zeros)
  if (!tmap_3d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w8, 128, (uint64_t)N, (uint64_t)K / 128, (uint64_t)K, 128, 128,
               kW8Rows, 4) ||
      !tmap_3d(&tm_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, a8, 128, (uint64_t)M, (uint64_t)K / 128, (uint64_t)K, 128, 128,
               16, 4))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(c, 0, sizeof(int32_t) * (size_t)M * N, stream);
  if (e != cudaSuccess) return e;
  e = allow_max_smem(w8a8_mma_kernel);
  if (e != cudaSuccess) return e;
  return launch_kernel(w8a8_mma_kernel, dim3(std::min(a.nunits, sms)), dim3(kW8Threads), smem, stream, pdl, tm_w,
                       tm_a, a);
}

bool w8a8_fused_ok(int M, int N, int K) {
  return M >= 1 && M <= 16 && N >= 1 && K >= 1024 && K % 1024 == 0 && K <= kFzMaxK;
}

size_t w8a8_fused_workspace_size(int M, int K) {
  (void)M;
  return 128 + 16 * (size_t)K;  // row maxima [16], barrier counters [4], pad | codes [16][K]
}

cudaError_t launch_w8a8_fused(const uint16_t* x, const uint32_t* sign_bits, const int8_t* w, const float* sw,
                              float* y, int M, int N, int K, void* ws, uint32_t* err, cudaStream_t stream) {
  W8FusedArgs a{};
  a.x = x;
  a.sign_bits = sign_bits;
  a.w = w;
  a.sw = sw;
  a.y = y;
  a.amax = static_cast<uint32_t*>(ws);
  a.cnt = a.amax + 16;
  a.qa = reinterpret_cast<int8_t*>(static_cast<uint8_t*>(ws) + 128);
  a.M = M;
  a.N = N;
  a.K = K;
  a.ntiles = (N + kFzRows - 1) / kFzRows;
  a.pitch = (uint32_t)K + 64;
  a.err = err;
  // every SM takes a share of the transform, also when there are fewer tiles
  const int grid = device_sm_count();
  const int nblk = M * (K / 32);
  a.zcap = (nblk + grid - 1) / grid;
  const size_t fixed = kFzQa + kFzRed + 128 * (size_t)a.zcap;
  const size_t stage = (size_t)kFzRows * a.pitch;
  const size_t budget = (size_t)device_max_smem_optin() - 256;
  if (budget < fixed + 2 * (stage + 16)) return cudaErrorInvalidValue;
  a.ST = (int)std::min<size_t>(4, (budget - fixed) / (stage + 16));
  const size_t smem = fixed + (size_t)a.ST * (stage + 16);
  cudaError_t e = allow_max_smem(w8a8_fused_kernel);
  if (e != cudaSuccess) return e;
  // CTAs wait for each other at the two grid barriers: a cooperative launch,
  // which the driver refuses rather than start partially
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kW8Threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, w8a8_fused_kernel, a);
}

}  // namespace qg
