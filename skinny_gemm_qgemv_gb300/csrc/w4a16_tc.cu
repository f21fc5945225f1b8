// W4A16 skinny GEMM on the 5th-generation tensor cores (tcgen05), M = 3..32.
//
// Y[m][n] = sum_k (s[n][g] q[n][k] + b[n][g]) X[m][k]: the skinny form of the
// affine 4-bit GEMV ("MLX Runner: An Inference Engine You Can Read", section
// "Architecture: one command buffer per token"), where several activation rows
// share one read of the weights ("Krill Teardown", section "Core mechanisms")
// and a 16-token verify batch gives the matrix units 16 rows of work (Uzu
// article, section "Producing several tokens from one model pass").
//
// GB300 design (one persistent CTA per SM, 10 warps):
//  warp 0      producer: TMA tensor loads per 512-k stage -- the X tile (bf16,
//              128B-swizzled, one box per 64-k group), the 4-bit codes of 128
//              weight rows (two 128B-swizzled boxes) and their fp16 scales and
//              biases -- into a ring of shared-memory stages (mbarrier tx).
//  warp 1      MMA issuer: per 64-k group, four tcgen05.mma.kind::f16
//              (M = 128 weight rows, N = 16 or 32 activation rows, K = 16) into a
//              fresh TMEM accumulator; owns the TMEM allocation.
//  warps 2..5  converters: decode each code word into eight bf16 values 128 + q
//              (exact) in natural k order and store them in the canonical
//              128B-swizzled K-major layout the MMA reads (A operand).
//  warps 6..9  epilogue: one weight row per thread (its TMEM lane); per group
//              it reads the accumulator (tcgen05.ld) and folds
//              y += s * acc + (b - 128 s) * sum_{k in g} x, the group-factored
//              affine dot product, in fp32. The weights are never rounded to
//              bf16: products are exact and only the fp32 sums round.
// Short matrices are split along K; the CTA finishing a row tile last (atomic
// counter, no waiting) adds the partial tiles in split order (deterministic).
// Every mbarrier wait is bounded; a timeout sets the device error word and a
// shared abort flag so all roles finish quickly and TMEM is released.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

namespace {

constexpr int kRows = 128;          // weight rows per tile = MMA M = TMEM lanes
constexpr int kStageK = 512;        // k per pipeline stage
constexpr int kGroupsPerStage = 8;  // 64-k groups per stage
constexpr int kNA = 8;              // A (converted weights) buffers in TMEM, 32 columns each
constexpr uint32_t kAccCols = 128;  // TMEM columns for accumulators: 128 / N buffers of N columns
constexpr uint32_t kTmemCols = 512; // accumulators at column 0, A buffers from column 128
constexpr int kThreads = 480;  // 1 producer + 2 MMA + 2 x 4 converter + 4 epilogue warps

struct TcArgs {
  int N, K, M;
  int ntiles, splits, kper, nunits;
  int ST;
  uint32_t stage_bytes;
  float* y;
  const uint16_t* x;
  float* partial;
  uint32_t* counters;
  uint32_t* err;
};

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  // tcgen05 shared-memory matrix descriptor, K-major, 128-byte swizzle:
  // start address >> 4, leading offset unused (1), stride between 8-row
  // groups 1024 B, descriptor version 1, swizzle mode 2 (128B).
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// 32 consecutive 32-bit TMEM columns of this thread's lane <- registers
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&v)[N]);

template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, float (&v)[32]) {
  float a[16], b[16];
  tmem_ld<16>(taddr, a);
  tmem_ld<16>(taddr + 16, b);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[i] = a[i];
    v[16 + i] = b[i];
  }
}

// Eight 4-bit codes (code i in bits 4i..4i+3) -> four bf16x2 registers in
// natural order: register j holds 128 + code 2j (low half) and 128 + code 2j+1
// (high half). The byte 0x43 above a code c in 0..15 is the bf16 of 128 + c.
__device__ __forceinline__ void nib8_to_bf16x2_natural(uint32_t w, uint32_t (&o)[4]) {
  const uint32_t even = w & 0x0F0F0F0Fu;         // codes 0, 2, 4, 6 in bytes 0..3
  const uint32_t odd = (w >> 4) & 0x0F0F0F0Fu;   // codes 1, 3, 5, 7
  const uint32_t t0 = __byte_perm(even, odd, 0x5140);  // codes 0, 1, 2, 3
  const uint32_t t1 = __byte_perm(even, odd, 0x7362);  // codes 4, 5, 6, 7
  constexpr uint32_t kMagic = 0x43004300u;
  o[0] = __byte_perm(t0, kMagic, 0x7150);
  o[1] = __byte_perm(t0, kMagic, 0x7352);
  o[2] = __byte_perm(t1, kMagic, 0x7150);
  o[3] = __byte_perm(t1, kMagic, 0x7352);
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Bounded wait that also honours the CTA-wide abort flag. Waiters off the
// MMA-issue critical path back off with a short sleep so their polling does not
// slow down the barrier operations of the issuing threads.
template <bool kBackoff>
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                              uint32_t* err, uint32_t code) {
  for (uint32_t i = 0; i < kMaxPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 1023u) == 1023u && *abort_flag) return false;
    if (kBackoff) __nanosleep(64);
  }
  report_error(err, code);
  *abort_flag = 1u;
  return false;
}

}  // namespace

template <int NT>
__global__ void __launch_bounds__(kThreads, 1)
    w4a16_tc_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_scales,
                    const __grid_constant__ CUtensorMap tm_biases, const __grid_constant__ CUtensorMap tm_x,
                    const TcArgs a) {
  constexpr int NB = (int)kAccCols / NT;  // TMEM accumulator buffers
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  // shared layout: stages | sx [K/64][NT] f32 | barriers
  const uint32_t s_stages = base;
  const int ngroups = a.kper / 64;
  const int nstage = a.kper / kStageK;
  const int gtotal = a.K / 64;
  float* sx = reinterpret_cast<float*>(gbase + a.ST * a.stage_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      gbase + ((a.ST * a.stage_bytes + sizeof(float) * gtotal * NT + 7) & ~(size_t)7));
  uint64_t* full = bars;
  uint64_t* empty = full + a.ST;
  uint64_t* afull = empty + a.ST;     // converted A of a group is in TMEM
  uint64_t* mmadone = afull + kNA;    // the MMAs of a group completed (A buffer free, accumulator ready)
  uint64_t* accempty = mmadone + kNA; // the epilogue has read an accumulator
  uint64_t* done = accempty + NB;     // [2] all MMAs of an issuing warp completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 2);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* is_last = tmem_slot + 2;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // per stage: [0, NT*1024) X tiles; codes 32 KB; scales, biases 2 KB each
  const uint32_t x_off = 0, c_off = NT * 1024, s_off = c_off + 32768, b_off = s_off + 2048;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 12);  // 8 converter warps + 4 epilogue warps
    }
    for (int i = 0; i < kNA; ++i) {
      mbar_init(&afull[i], 4);
      mbar_init(&mmadone[i], 1);
    }
    for (int i = 0; i < NB; ++i) mbar_init(&accempty[i], 4);
    mbar_init(&done[0], 1);
    mbar_init(&done[1], 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // sum of x over every 64-k group of the whole K, per activation row, once
  // per CTA (all threads; the activations may come from the previous kernel)
  pdl_wait();
  for (int idx = threadIdx.x; idx < gtotal * NT; idx += kThreads) {
    const int g = idx / NT, m = idx % NT;
    float t = 0.f;
    if (m < a.M) {
      const uint4* xp = reinterpret_cast<const uint4*>(a.x + (size_t)m * a.K + 64 * g);
      uint4 c[8];
#pragma unroll
      for (int v = 0; v < 8; ++v) c[v] = xp[v];
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const uint32_t e[4] = {c[v].x, c[v].y, c[v].z, c[v].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) t += bf16_bits_to_f32(e[h] & 0xFFFFu) + bf16_bits_to_f32(e[h] >> 16);
      }
    }
    sx[idx] = t;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int issued = 0;
      for (int ui = 0, u = blockIdx.x; u < a.nunits && !*abort_flag; ++ui, u += gridDim.x) {
        const int tile = u / a.splits, split = u % a.splits;
        const int n0 = tile * kRows, k0 = split * a.kper;
        for (int s = 0; s < nstage; ++s) {
          const int sg = ui * nstage + s, st = sg % a.ST;
          if (sg >= a.ST &&
              !wait_or_abort<true>(&empty[st], ((sg / a.ST) & 1) ^ 1, abort_flag, a.err, kErrTcEmptyWait))
            break;
          const uint32_t sb = s_stages + st * a.stage_bytes;
          mbar_arrive_expect_tx(&full[st], a.stage_bytes);
          const int kk = k0 + s * kStageK;
          // X viewed as {64 k, rows, K/64}: one box = the stage's eight [NT][128 B] tiles;
          // codes viewed as {128 B, rows, K/256}: one box = two [128][128 B] tiles
          tma_load_3d(sb + x_off, &tm_x, 0, 0, kk / 64, &full[st]);
          tma_load_3d(sb + c_off, &tm_codes, 0, n0, kk / 256, &full[st]);
          tma_load_2d(sb + s_off, &tm_scales, kk / 64, n0, &full[st]);
          tma_load_2d(sb + b_off, &tm_biases, kk / 64, n0, &full[st]);
          ++issued;
        }
      }
      // every issued copy must land before the CTA exits
      for (int j = max(0, issued - a.ST); j < issued; ++j)
        mbar_wait(&full[j % a.ST], (j / a.ST) & 1, a.err, kErrTcDrain);
    }
  } else if (warp <= 2) {
    // ------------------------------------------------- MMA issuers: warp 1 even groups, warp 2 odd
    if (lane == 0) {
      const int parity_set = warp - 1;
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NT >> 3) << 17) |
                             ((uint32_t)(kRows >> 4) << 24);
      bool ok = true;
      for (int ui = 0, u = blockIdx.x; u < a.nunits && ok; ++ui, u += gridDim.x) {
        for (int g = parity_set; g < ngroups && ok; g += 2) {
          const int gg = ui * ngroups + g;
          const int sg = ui * nstage + g / kGroupsPerStage, st = sg % a.ST;
          const int ab = gg % kNA, nb = gg % NB;
          ok = wait_or_abort<false>(&full[st], (sg / a.ST) & 1, abort_flag, a.err, kErrTcFullWait);
          ok = ok && wait_or_abort<false>(&afull[ab], (gg / kNA) & 1, abort_flag, a.err, kErrTcMmaWait);
          if (ok && gg >= NB)
            ok = wait_or_abort<false>(&accempty[nb], ((gg / NB) & 1) ^ 1, abort_flag, a.err, kErrTcAccWait);
          if (!ok) break;
          tc_fence_after();
          const uint32_t at = tbase + kAccCols + ab * 32;
          const uint64_t bd = sw128_desc(s_stages + st * a.stage_bytes + x_off + (g % kGroupsPerStage) * NT * 128);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) mma_bf16_tmem_a(tbase + nb * NT, at + 8 * ks, bd + 2 * ks, idesc, ks > 0);
          mma_commit(&mmadone[ab]);
        }
      }
      mma_commit(&done[parity_set]);
      mbar_wait(&done[parity_set], 0, a.err, kErrTcDrain);
    }
  } else if (warp < 11) {
    // ------------------------------------- converters: warps 3..6 even groups, 7..10 odd groups
    // a warp may only touch TMEM lanes 32 * (warp % 4) .. + 31: row = its lane
    const int set = (warp - 3) >> 2;
    const int r = (warp & 3) * 32 + lane;  // weight row of the tile, 0..127
    const uint32_t rsw = r & 7;
    const uint32_t tlane = tbase + ((uint32_t)((warp & 3) * 32) << 16) + kAccCols;
    for (int ui = 0, u = blockIdx.x; u < a.nunits; ++ui, u += gridDim.x) {
      for (int g = set; g < ngroups; g += 2) {
        const int gg = ui * ngroups + g;
        const int sg = ui * nstage + g / kGroupsPerStage, st = sg % a.ST;
        const int ab = gg % kNA;
        if (!*abort_flag && g % kGroupsPerStage <= 1)
          wait_or_abort<true>(&full[st], (sg / a.ST) & 1, abort_flag, a.err, kErrTcFullWait);
        if (!*abort_flag && gg >= kNA)
          wait_or_abort<true>(&mmadone[ab], ((gg / kNA) & 1) ^ 1, abort_flag, a.err, kErrTcMmaWait);
        tc_fence_after();
        if (!*abort_flag) {
          const int j = g % kGroupsPerStage;
          const uint32_t row = s_stages + st * a.stage_bytes + c_off + (j >> 2) * 16384 + r * 128;
          const uint32_t c0 = 2 * (j & 3);
          const uint4 lo = lds128(row + ((c0 ^ rsw) << 4));
          const uint4 hi = lds128(row + (((c0 + 1) ^ rsw) << 4));
          const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
          uint32_t o[32];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            uint32_t t4[4];
            nib8_to_bf16x2_natural(w[i], t4);
#pragma unroll
            for (int c = 0; c < 4; ++c) o[4 * i + c] = t4[c];
          }
          tmem_st32(tlane + ab * 32, o);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&afull[ab]);
          // this set's last group of the stage
          if (g % kGroupsPerStage >= kGroupsPerStage - 2 || g + 2 >= ngroups) mbar_arrive(&empty[st]);
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 11..14)
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int et = threadIdx.x - 352;  // 0..127
    const uint32_t tlane = tbase + ((uint32_t)(q * 32) << 16);
    for (int ui = 0, u = blockIdx.x; u < a.nunits; ++ui, u += gridDim.x) {
      const int tile = u / a.splits, split = u % a.splits;
      const int n0 = tile * kRows;
      const float* sxu = sx + (size_t)(split * ngroups) * NT;
      float yacc[NT];
#pragma unroll
      for (int m = 0; m < NT; ++m) yacc[m] = 0.f;
      for (int g = 0; g < ngroups; ++g) {
        const int gg = ui * ngroups + g;
        const int sg = ui * nstage + g / kGroupsPerStage, st = sg % a.ST;
        const int nb = gg % NB, ab = gg % kNA;
        // the epilogue releases accumulators on the MMA critical path: no backoff
        if (!*abort_flag && g % kGroupsPerStage == 0)
          wait_or_abort<false>(&full[st], (sg / a.ST) & 1, abort_flag, a.err, kErrTcFullWait);
        if (!*abort_flag) wait_or_abort<false>(&mmadone[ab], (gg / kNA) & 1, abort_flag, a.err, kErrTcAccWait);
        tc_fence_after();
        float acc[NT];
        tmem_ld<NT>(tlane + nb * NT, acc);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&accempty[nb]);
        const uint32_t sb = s_stages + st * a.stage_bytes;
        const int j = g % kGroupsPerStage;
        const float s = f16_bits_to_f32(lds16(sb + s_off + row * 16 + 2 * j));
        const float b = f16_bits_to_f32(lds16(sb + b_off + row * 16 + 2 * j));
        const float c = fmaf(-128.f, s, b);
#pragma unroll
        for (int m = 0; m < NT; ++m) yacc[m] = fmaf(s, acc[m], fmaf(c, sxu[g * NT + m], yacc[m]));
        __syncwarp();
        if (lane == 0 && (j == kGroupsPerStage - 1 || g == ngroups - 1)) mbar_arrive(&empty[st]);
      }
      const int n = n0 + row;
      if (a.splits == 1) {
        if (n < a.N) {
#pragma unroll
          for (int m = 0; m < NT; ++m)
            if (m < a.M) a.y[(size_t)m * a.N + n] = yacc[m];
        }
      } else {
        float* part = a.partial + (size_t)u * NT * kRows;
#pragma unroll
        for (int m = 0; m < NT; ++m) part[m * kRows + row] = yacc[m];
        __threadfence();
        epi_bar();
        if (et == 0) *is_last = (atomicAdd(&a.counters[tile], 1u) == (uint32_t)(a.splits - 1)) ? 1u : 0u;
        epi_bar();
        if (*is_last) {
          __threadfence();
          if (n < a.N) {
            for (int m = 0; m < a.M; ++m) {
              float t = 0.f;
              for (int s2 = 0; s2 < a.splits; ++s2)
                t += __ldcg(a.partial + ((size_t)(tile * a.splits + s2) * NT + m) * kRows + row);
              a.y[(size_t)m * a.N + n] = t;
            }
          }
          if (et == 0) a.counters[tile] = 0u;
        }
        epi_bar();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_launch_dependents();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kTmemCols));
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3D view {inner, rows, chunks}: element (i, r, c) at ptr + r * row_bytes + c * chunk_bytes + i * elem
bool make_map3(CUtensorMap* tm, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t rows,
               uint64_t chunks, uint64_t row_bytes, uint64_t chunk_bytes, uint32_t box_inner, uint32_t box_rows,
               uint32_t box_chunks) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {inner, rows, chunks};
  cuuint64_t strides[2] = {row_bytes, chunk_bytes};
  cuuint32_t box[3] = {box_inner, box_rows, box_chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(tm, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map(CUtensorMap* tm, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t outer,
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(tm, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct TcPlan {
  int NT, ntiles, splits, kper, nunits, ST;
  uint32_t stage_bytes;
  size_t smem, ws_partial, ws_counters;
};

TcPlan tc_plan(int M, int N, int K, int sms) {
  TcPlan p;
  p.NT = M <= 16 ? 16 : 32;
  p.ntiles = (N + kRows - 1) / kRows;
  const int kstages = K / kStageK;
  // split K until every SM has a unit, keeping each split a whole number of stages
  p.splits = 1;
  while (p.ntiles * p.splits < sms && p.splits * 2 <= kstages && kstages % (p.splits * 2) == 0) p.splits *= 2;
  p.kper = K / p.splits;
  p.nunits = p.ntiles * p.splits;
  p.stage_bytes = (uint32_t)(p.NT * 1024 + 36864);
  const size_t fixed = 1024 + sizeof(float) * (size_t)(K / 64) * p.NT + 256;
  const size_t budget = 224 * 1024;
  p.ST = (int)std::min<size_t>(4, (budget - fixed) / p.stage_bytes);
  p.smem = fixed + (size_t)p.ST * p.stage_bytes;
  p.ws_partial = p.splits > 1 ? sizeof(float) * (size_t)p.nunits * p.NT * kRows : 0;
  p.ws_counters = p.splits > 1 ? sizeof(uint32_t) * (size_t)p.ntiles : 0;
  return p;
}

}  // namespace

bool tc_path_ok(int M, int N, int K) {
  return M >= 3 && M <= 32 && N >= 1 && K % kStageK == 0 && K >= kStageK && K <= 32768;
}

size_t tc_workspace_size(int M, int N, int K) {
  if (!tc_path_ok(M, N, K)) return 0;
  const TcPlan p = tc_plan(M, N, K, device_sm_count());
  return p.ws_partial + ((p.ws_counters + 255) & ~(size_t)255) + (p.ws_partial ? 256 : 0);
}

template <int NT>
static cudaError_t launch_tc_nt(const CUtensorMap* maps, const TcArgs& a, const TcPlan& p, int grid,
                                cudaStream_t stream, bool pdl) {
  auto kern = w4a16_tc_kernel<NT>;
  cudaError_t e = allow_max_smem(kern);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(grid), dim3(kThreads), p.smem, stream, pdl, maps[0], maps[1], maps[2], maps[3],
                       a);
}

cudaError_t launch_w4a16_tc(const uint32_t* wq, const uint16_t* sc, const uint16_t* bi, const uint16_t* x,
                            float* y, int M, int N, int K, void* ws, size_t ws_bytes, uint32_t* err,
                            cudaStream_t stream, bool pdl) {
  const int sms = device_sm_count();
  const TcPlan p = tc_plan(M, N, K, sms);
  if (ws_bytes < tc_workspace_size(M, N, K)) return cudaErrorInvalidValue;
  CUtensorMap maps[4];
  const bool ok =
      make_map3(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, 128, (uint64_t)N, (uint64_t)K / 256, (uint64_t)K / 2,
                128, 128, kRows, 2) &&
      make_map(&maps[1], CU_TENSOR_MAP_DATA_TYPE_UINT16, sc, (uint64_t)K / 64, (uint64_t)N, (uint64_t)K / 32, 8,
               kRows, CU_TENSOR_MAP_SWIZZLE_NONE) &&
      make_map(&maps[2], CU_TENSOR_MAP_DATA_TYPE_UINT16, bi, (uint64_t)K / 64, (uint64_t)N, (uint64_t)K / 32, 8,
               kRows, CU_TENSOR_MAP_SWIZZLE_NONE) &&
      make_map3(&maps[3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, 64, (uint64_t)M, (uint64_t)K / 64, (uint64_t)K * 2,
                128, 64, (uint32_t)p.NT, kGroupsPerStage);
  if (!ok) return cudaErrorInvalidValue;
  TcArgs a;
  a.N = N;
  a.K = K;
  a.M = M;
  a.ntiles = p.ntiles;
  a.splits = p.splits;
  a.kper = p.kper;
  a.nunits = p.nunits;
  a.ST = p.ST;
  a.stage_bytes = p.stage_bytes;
  a.y = y;
  a.x = x;
  a.partial = p.splits > 1 ? static_cast<float*>(ws) : nullptr;
  a.counters = p.splits > 1 ? reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + p.ws_partial) : nullptr;
  a.err = err;
  if (p.splits > 1) {
    cudaError_t e = cudaMemsetAsync(a.counters, 0, p.ws_counters, stream);
    if (e != cudaSuccess) return e;
  }
  const int grid = std::min(p.nunits, sms);
  if (p.NT == 16) return launch_tc_nt<16>(maps, a, p, grid, stream, pdl);
  return launch_tc_nt<32>(maps, a, p, grid, stream, pdl);
}

}  // namespace qg
