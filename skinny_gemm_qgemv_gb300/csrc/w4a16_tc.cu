// W4A16 skinny GEMM on the 5th-generation tensor cores (tcgen05), M = 3..32.
//
// Y[m][n] = sum_k (s[n][g] q[n][k] + b[n][g]) X[m][k]: the skinny form of the
// affine 4-bit GEMV ("MLX Runner: An Inference Engine You Can Read", section
// "Architecture: one command buffer per token"), where several activation rows
// share one read of the weights ("Krill Teardown", section "Core mechanisms")
// and a 16-token verify batch gives the matrix units 16 rows of work (Uzu
// article, section "Producing several tokens from one model pass").
//
// GB300 design (one persistent CTA per SM, 15 warps). The roles hand work to
// each other in chunks of 256 k (four 64-k groups): every mbarrier operation
// costs tens to hundreds of cycles under load, so one hand-off per group would
// pace the whole pipeline.
//  warp 0       producer: TMA tensor loads per 512-k stage -- the X tile (bf16,
//               128B-swizzled, one box per 64-k group), the 4-bit codes of 128
//               weight rows (two 128B-swizzled boxes, one per chunk) and their
//               fp16 scales and biases -- into a ring of shared-memory stages.
//  warps 1, 2   MMA issuers (groups 0-1 / 2-3 of every chunk): per group four
//               tcgen05.mma.kind::f16 (M = 128 weight rows, N = 16 or 32
//               activation rows, K = 16) with A read from TMEM, each group into
//               its own accumulator; one commit per chunk. They learn that A is
//               converted and that an accumulator buffer was read from shared
//               counters, and need no wait on the stage itself (the converters
//               waited for it before converting).
//  warps 3..10  converters, all on every chunk (warps 3..6 its groups 0-1,
//               7..10 groups 2-3): decode each code word into eight bf16 values
//               128 + q (exact) in natural k order and store them into TMEM as
//               the A operand (row = lane); two A buffers let the next chunk be
//               decoded while the MMAs read the current one.
//  warps 11..14 epilogue: one weight row per thread (its TMEM lane); per chunk
//               it reads the four accumulators (tcgen05.ld) and folds
//               y += s * acc + (b - 128 s) * sum_{k in g} x, the group-factored
//               affine dot product, in fp32. The weights are never rounded to
//               bf16: products are exact and only the fp32 sums round. The
//               sums of x per group come from the landed X tile, computed by
//               the same warps while the chunk's MMAs run.
// TMEM: columns 0..255 hold the accumulators (chunk buffers of 4 x N columns),
// 256..511 two A chunk buffers of 4 x 32 columns.
// A grouped launch walks the full-K row tiles of many projections, one
// contiguous equal-cost range per CTA, reading each projection's tensor maps
// from a descriptor in device memory.
// Short matrices are split along K while twice the units still fit the SMs
// (each unit then pipelines several stages); the CTA finishing a row tile last
// (atomic counter, no waiting) adds the partial tiles in split order
// (deterministic) and resets the counter, so the workspace needs clearing only
// before its first use.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

namespace {

constexpr int kRows = 128;          // weight rows per tile = MMA M = TMEM lanes
constexpr int kStageK = 512;        // k per pipeline stage
constexpr int kGroupsPerStage = 8;  // 64-k groups per stage
constexpr int kChunkK = 256;        // k per hand-off between the roles: one 128-byte row of codes
constexpr int kChunkGroups = 4;     // 64-k groups per chunk
constexpr int kChunksPerStage = kStageK / kChunkK;
constexpr int kNAB = 2;             // A (converted weights) chunk buffers in TMEM, 128 columns each
constexpr uint32_t kAccCols = 256;  // TMEM columns for accumulators: chunk buffers of 4 x N columns
constexpr uint32_t kACol = 256;     // first TMEM column of the A buffers
constexpr uint32_t kTmemCols = 512;
constexpr int kThreads = 480;  // 1 producer + 2 MMA + 8 converter + 4 epilogue warps

// One projection of a grouped launch, as the kernel reads it from global
// memory; the tensor maps need 64-byte alignment (CUtensorMap is declared with 128).
struct TcGemv {
  CUtensorMap codes, scales, biases, x;
  float* y;
  const uint16_t* xraw;  // the activations (mma path: read by the B-fragment pass)
  uint32_t* frag;        // mma path: B fragments of X, K * 32 bytes
  float* tab;            // mma path: per 64-k group offsets, sums of x and 2^sigma
  int N, M, K;
  int unit0, unit_end;  // its row tiles in the launch's unit numbering
};
static_assert(alignof(TcGemv) >= 64, "tensor maps need 64-byte alignment");

struct TcArgs {
  int N, K, M;
  int ntiles, splits, kper, nunits;
  int ST;
  uint32_t stage_bytes;
  float* y;
  float* partial;
  uint32_t* counters;
  uint32_t* err;
  const uint32_t* frag;  // mma path, one matrix: B fragments and group table
  const float* tab;
  // grouped launch (null for one matrix): per-projection descriptors, the
  // first unit of every CTA's range ([grid + 1]) and the projection of that unit
  const TcGemv* gemvs;
  const int* cta_unit0;
  const int* cta_gemv0;
};

// The units one CTA works on, in order: for one matrix a grid-stride walk over
// its (128-row tile, K split) pairs; for a grouped launch a contiguous range of
// full-K row tiles of the group's projections, the projections in group order.
struct UnitWalk {
  int u, end, stride, g;
  int tile, n0, k0, kper, N, M;
  float* y;
  const uint32_t* frag;
  const float* tab;
  __device__ __forceinline__ explicit UnitWalk(const TcArgs& a) {
    if (a.gemvs) {
      u = a.cta_unit0[blockIdx.x];
      end = a.cta_unit0[blockIdx.x + 1];
      stride = 1;
      g = a.cta_gemv0[blockIdx.x];
    } else {
      u = blockIdx.x;
      end = a.nunits;
      stride = gridDim.x;
      g = 0;
    }
    load(a);
  }
  __device__ __forceinline__ bool valid() const { return u < end; }
  __device__ __forceinline__ void next(const TcArgs& a) {
    u += stride;
    load(a);
  }
  __device__ __forceinline__ void load(const TcArgs& a) {
    if (u >= end) return;
    if (a.gemvs) {
      while (u >= a.gemvs[g].unit_end) ++g;
      const TcGemv& d = a.gemvs[g];
      tile = u - d.unit0;
      k0 = 0;
      kper = d.K;
      N = d.N;
      M = d.M;
      y = d.y;
      frag = d.frag;
      tab = d.tab;
    } else {
      tile = u / a.splits;
      k0 = (u % a.splits) * a.kper;
      kper = a.kper;
      N = a.N;
      M = a.M;
      y = a.y;
      frag = a.frag;
      tab = a.tab;
    }
    n0 = tile * kRows;
  }
};

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  // tcgen05 shared-memory matrix descriptor, K-major, 128-byte swizzle:
  // start address >> 4, leading offset unused (1), stride between 8-row
  // groups 1024 B, descriptor version 1, swizzle mode 2 (128B).
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}


__device__ __forceinline__ void tensormap_acquire(const CUtensorMap* tm) {
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(reinterpret_cast<uint64_t>(tm))
               : "memory");
}

__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// 32 consecutive 32-bit TMEM columns of this thread's lane <- registers (no wait)
__device__ __forceinline__ void tmem_st32_nowait(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// G groups x N accumulator columns of this thread's lane (G * N = 64): sixteen
// columns per load, one wait for all of them; the values are only touched
// after the wait.
template <int G, int N>
__device__ __forceinline__ void tmem_ld_groups(uint32_t taddr, uint32_t (&r)[G][N]) {
#pragma unroll
  for (int j = 0; j < G; ++j) {
#pragma unroll
    for (int h = 0; h < N / 16; ++h) {
      uint32_t* o = &r[j][16 * h];
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
          : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]), "=r"(o[4]), "=r"(o[5]), "=r"(o[6]), "=r"(o[7]),
            "=r"(o[8]), "=r"(o[9]), "=r"(o[10]), "=r"(o[11]), "=r"(o[12]), "=r"(o[13]), "=r"(o[14]), "=r"(o[15])
          : "r"(taddr + j * N + 16 * h));
    }
  }
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < G; ++j)
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[j][i]));
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
__device__ __forceinline__ uint32_t ld_acquire_s32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add_s32(uint32_t* p, uint32_t v) {
  asm volatile("red.release.cta.shared::cta.add.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ bool wait_count(const uint32_t* p, uint32_t target, volatile uint32_t* abort_flag,
                                           uint32_t* err, uint32_t code) {
  for (uint32_t i = 0; i < (kMaxPolls << 6); ++i) {
    if ((int32_t)(ld_acquire_s32(p) - target) >= 0) return true;
    if ((i & 1023u) == 1023u && *abort_flag) return false;
  }
  report_error(err, code);
  *abort_flag = 1u;
  return false;
}

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
  constexpr int NACC = (int)kAccCols / (kChunkGroups * NT);  // accumulator chunk buffers in TMEM
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  // shared layout: stages | sx [2][4 groups][NT] f32 (x sums of a chunk) | barriers
  const uint32_t s_stages = base;
  float* sx = reinterpret_cast<float*>(gbase + a.ST * a.stage_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      gbase + ((a.ST * a.stage_bytes + sizeof(float) * 2 * kChunkGroups * NT + 7) & ~(size_t)7));
  uint64_t* full = bars;
  uint64_t* empty = full + a.ST;
  uint64_t* accfull = empty + a.ST;    // the MMAs of a chunk completed: accumulators ready, A buffer free
  uint64_t* done = accfull + NACC;     // [2] all MMAs of an issuing warp completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 2);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* is_last = tmem_slot + 2;
  // Hand-offs to the MMA issuers are monotonic shared-memory counters (release
  // add / acquire load): polling one costs a shared load, where an mbarrier
  // try_wait costs a few hundred cycles while the converters keep the shared
  // memory pipe busy, and the issuers wait on every chunk.
  uint32_t* conv_cnt = tmem_slot + 4;       // [kNAB][2] converter warps done with half an A buffer
  uint32_t* epi_cnt = conv_cnt + 2 * kNAB;  // [NACC] epilogue warps done reading an accumulator buffer

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // per stage: [0, NT*1024) X tiles; codes 32 KB; scales, biases 2 KB each
  const uint32_t x_off = 0, c_off = NT * 1024, s_off = c_off + 32768, b_off = s_off + 2048;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 12);  // 8 converter warps + 4 epilogue warps
    }
    for (int i = 0; i < NACC; ++i) {
      mbar_init(&accfull[i], 2);  // one commit per MMA warp
    }
    mbar_init(&done[0], 1);
    mbar_init(&done[1], 1);
    *abort_flag = 0u;
    for (int i = 0; i < 2 * kNAB + NACC; ++i) conv_cnt[i] = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // the activations may come from the previous kernel
  pdl_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int issued = 0, fenced = -1;
      for (UnitWalk w(a); w.valid() && !*abort_flag; w.next(a)) {
        const int nstage = w.kper / kStageK;
        if (a.gemvs && w.g != fenced) {
          // the descriptors were written through the generic proxy (a host copy,
          // possibly into memory that held other descriptors before): make the
          // TMA unit see their current contents
          const TcGemv* d = &a.gemvs[w.g];
          tensormap_acquire(&d->codes);
          tensormap_acquire(&d->scales);
          tensormap_acquire(&d->biases);
          tensormap_acquire(&d->x);
          fenced = w.g;
        }
        const CUtensorMap* mc = a.gemvs ? &a.gemvs[w.g].codes : &tm_codes;
        const CUtensorMap* ms = a.gemvs ? &a.gemvs[w.g].scales : &tm_scales;
        const CUtensorMap* mb = a.gemvs ? &a.gemvs[w.g].biases : &tm_biases;
        const CUtensorMap* mx = a.gemvs ? &a.gemvs[w.g].x : &tm_x;
        for (int s = 0; s < nstage; ++s) {
          const int sg = issued, st = sg % a.ST;
          if (sg >= a.ST &&
              !wait_or_abort<true>(&empty[st], ((sg / a.ST) & 1) ^ 1, abort_flag, a.err, kErrTcEmptyWait))
            break;
          const uint32_t sb = s_stages + st * a.stage_bytes;
          mbar_arrive_expect_tx(&full[st], a.stage_bytes);
          const int kk = w.k0 + s * kStageK;
          // X viewed as {64 k, rows, K/64}: one box = the stage's eight [NT][128 B] tiles;
          // codes viewed as {128 B, rows, K/256}: one box = two [128][128 B] tiles (one per chunk)
          tma_load_3d(sb + x_off, mx, 0, 0, kk / 64, &full[st]);
          tma_load_3d(sb + c_off, mc, 0, w.n0, kk / 256, &full[st]);
          tma_load_2d(sb + s_off, ms, kk / 64, w.n0, &full[st]);
          tma_load_2d(sb + b_off, mb, kk / 64, w.n0, &full[st]);
          ++issued;
        }
      }
      // every issued copy must land before the CTA exits
      for (int j = max(0, issued - a.ST); j < issued; ++j)
        mbar_wait(&full[j % a.ST], (j / a.ST) & 1, a.err, kErrTcDrain);
    }
    __syncwarp();  // the lane's role loop ends here: the warp reaches the final barrier converged
  } else if (warp <= 2) {
    // ------------------------- MMA issuers: warp 1 groups 0, 1 of every chunk, warp 2 groups 2, 3
    if (lane == 0) {
      const int h = warp - 1;
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NT >> 3) << 17) |
                             ((uint32_t)(kRows >> 4) << 24);
      bool ok = true;
      int gcb = 0, sgb = 0;  // chunks and stages of the CTA's earlier units
      for (UnitWalk w(a); w.valid() && ok; w.next(a)) {
        const int nchunk = w.kper / kChunkK;
        for (int c = 0; c < nchunk && ok; ++c) {
          const int gc = gcb + c;
          const int sg = sgb + c / kChunksPerStage, st = sg % a.ST;
          const int ab = gc % kNAB, nb = gc % NACC;
          ok = wait_count(&conv_cnt[2 * ab + h], 4u * (uint32_t)(gc / kNAB + 1), abort_flag, a.err, kErrTcMmaWait);
          if (ok && gc >= NACC)
            ok = wait_count(&epi_cnt[nb], 4u * (uint32_t)(gc / NACC), abort_flag, a.err, kErrTcAccWait);
          if (!ok) break;
          tc_fence_after();
          const uint32_t xs = s_stages + st * a.stage_bytes + x_off;
#pragma unroll
          for (int jj = 0; jj < kChunkGroups / 2; ++jj) {
            const int j = 2 * h + jj;
            const int gi = (c % kChunksPerStage) * kChunkGroups + j;  // group within the stage
            const uint32_t at = tbase + kACol + ab * (kChunkGroups * 32) + j * 32;
            const uint32_t dt = tbase + nb * (kChunkGroups * NT) + j * NT;
            const uint64_t bd = sw128_desc(xs + gi * NT * 128);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) mma_bf16_tmem_a(dt, at + 8 * ks, bd + 2 * ks, idesc, ks > 0);
          }
          mma_commit(&accfull[nb]);
        }
        gcb += nchunk;
        sgb += nchunk / kChunksPerStage;
      }
      mma_commit(&done[h]);
      mbar_wait(&done[h], 0, a.err, kErrTcDrain);
    }
    __syncwarp();  // the lane's role loop ends here: the warp reaches the final barrier converged
  } else if (warp < 11) {
    // ------------------------------------------ converters: warps 3..10, every chunk
    // a warp may only touch TMEM lanes 32 * (warp % 4) .. + 31: row = its lane;
    // warps 3..6 decode groups 0, 1 of a chunk, warps 7..10 groups 2, 3
    const int h = (warp - 3) >> 2;
    const int r = (warp & 3) * 32 + lane;  // weight row of the tile, 0..127
    const uint32_t rsw = r & 7;
    const uint32_t tlane = tbase + ((uint32_t)((warp & 3) * 32) << 16) + kACol;
    int gcb = 0, sgb = 0;
    for (UnitWalk w(a); w.valid(); w.next(a)) {
      const int nchunk = w.kper / kChunkK;
      for (int c = 0; c < nchunk; ++c) {
        const int gc = gcb + c;
        const int sg = sgb + c / kChunksPerStage, st = sg % a.ST;
        const int ab = gc % kNAB;
        if (!*abort_flag && c % kChunksPerStage == 0)
          wait_or_abort<true>(&full[st], (sg / a.ST) & 1, abort_flag, a.err, kErrTcFullWait);
        // the A buffer is free once the MMAs of chunk gc - kNAB completed
        if (!*abort_flag && gc >= kNAB) {
          const int pc = gc - kNAB;
          wait_or_abort<true>(&accfull[pc % NACC], (pc / NACC) & 1, abort_flag, a.err, kErrTcMmaWait);
        }
        tc_fence_after();
        if (!*abort_flag) {
          // the chunk's 256 k of this row: one 128-byte swizzled row of the codes tile
          const uint32_t row = s_stages + st * a.stage_bytes + c_off + (c % kChunksPerStage) * 16384 + r * 128;
#pragma unroll
          for (int jj = 0; jj < kChunkGroups / 2; ++jj) {
            const int j = 2 * h + jj;
            const uint32_t c0 = 2 * j;
            const uint4 lo = lds128(row + ((c0 ^ rsw) << 4));
            const uint4 hi = lds128(row + (((c0 + 1) ^ rsw) << 4));
            const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
            uint32_t o[32];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              uint32_t t4[4];
              nib8_to_bf16x2_natural(w[i], t4);
#pragma unroll
              for (int q = 0; q < 4; ++q) o[4 * i + q] = t4[q];
            }
            tmem_st32_nowait(tlane + ab * (kChunkGroups * 32) + j * 32, o);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          red_release_add_s32(&conv_cnt[2 * ab + h], 1u);
          if (c % kChunksPerStage == kChunksPerStage - 1) mbar_arrive(&empty[st]);
        }
      }
      gcb += nchunk;
      sgb += nchunk / kChunksPerStage;
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 11..14)
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int et = threadIdx.x - 352;  // 0..127 (warps 11..14)
    const uint32_t tlane = tbase + ((uint32_t)(q * 32) << 16);
    int gcb = 0, sgb = 0;
    for (UnitWalk w(a); w.valid(); w.next(a)) {
      const int nchunk = w.kper / kChunkK;
      uint64_t yacc2[NT / 2];  // activation rows (2p, 2p + 1)
#pragma unroll
      for (int q2 = 0; q2 < NT / 2; ++q2) yacc2[q2] = 0ull;
      for (int c = 0; c < nchunk; ++c) {
        const int gc = gcb + c;
        const int sg = sgb + c / kChunksPerStage, st = sg % a.ST;
        const int nb = gc % NACC;
        // the epilogue releases accumulators on the MMA critical path: no backoff
        if (!*abort_flag && c % kChunksPerStage == 0)
          wait_or_abort<false>(&full[st], (sg / a.ST) & 1, abort_flag, a.err, kErrTcFullWait);
        const int j0 = (c % kChunksPerStage) * kChunkGroups;  // first group of the chunk within the stage
        float* sxc = sx + (c & 1) * (kChunkGroups * NT);
        {
          // x sums of the chunk's groups while its MMAs run: a (group, activation
          // row) pair per thread (N = 32) or per two threads (N = 16), from the
          // row's 128 bytes of the landed X tile in any order
          constexpr int kPer = 128 / (kChunkGroups * NT);  // threads per sum: 2 or 1
          const int p = et / kPer, part = et % kPer;
          const uint32_t src = s_stages + st * a.stage_bytes + x_off + ((j0 + p / NT) * NT + p % NT) * 128;
          const uint32_t sw = (uint32_t)(p % NT) & 7;  // the tile's 128-byte swizzle of this row
          float t0 = 0.f, t1 = 0.f;
#pragma unroll
          for (int v = 0; v < 8 / kPer; ++v) {
            // physical 16-byte units part * 4 + v, spread over the banks by the swizzle
            const uint4 c4 = lds128(src + ((((uint32_t)(part * (8 / kPer) + v)) ^ sw) << 4));
            t0 += bf16_bits_to_f32(c4.x & 0xFFFFu) + bf16_bits_to_f32(c4.x >> 16);
            t1 += bf16_bits_to_f32(c4.y & 0xFFFFu) + bf16_bits_to_f32(c4.y >> 16);
            t0 += bf16_bits_to_f32(c4.z & 0xFFFFu) + bf16_bits_to_f32(c4.z >> 16);
            t1 += bf16_bits_to_f32(c4.w & 0xFFFFu) + bf16_bits_to_f32(c4.w >> 16);
          }
          float t = t0 + t1;
          if (kPer == 2) t += __shfl_xor_sync(0xFFFFFFFFu, t, 1);
          if (part == 0) sxc[p] = t;
          epi_bar();
        }
        if (!*abort_flag) wait_or_abort<false>(&accfull[nb], (gc / NACC) & 1, abort_flag, a.err, kErrTcAccWait);
        tc_fence_after();
        const uint32_t sb = s_stages + st * a.stage_bytes;
        const uint2 s4 = lds64(sb + s_off + row * 16 + 2 * j0);
        const uint2 b4 = lds64(sb + b_off + row * 16 + 2 * j0);
        const uint32_t sv[2] = {s4.x, s4.y}, bv[2] = {b4.x, b4.y};
        // 64 accumulator columns per batch: all four groups (N = 16) or two (N = 32)
        constexpr int G = 64 / NT;
#pragma unroll
        for (int j1 = 0; j1 < kChunkGroups; j1 += G) {
          uint32_t acc[G][NT];
          tmem_ld_groups<G, NT>(tlane + nb * (kChunkGroups * NT) + j1 * NT, acc);
          if (j1 + G == kChunkGroups) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) red_release_add_s32(&epi_cnt[nb], 1u);
          }
#pragma unroll
          for (int jj = 0; jj < G; ++jj) {
            const int j = j1 + jj;
            const float s = f16_bits_to_f32((sv[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
            const float b = f16_bits_to_f32((bv[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
            const float cc = fmaf(-128.f, s, b);
            const uint64_t s2 = pair2(__float_as_uint(s), __float_as_uint(s));
            const uint64_t c2 = pair2(__float_as_uint(cc), __float_as_uint(cc));
            const uint64_t* sxg = reinterpret_cast<const uint64_t*>(sxc + j * NT);
#pragma unroll
            for (int q2 = 0; q2 < NT / 2; ++q2)
              yacc2[q2] = ffma2(s2, pair2(acc[jj][2 * q2], acc[jj][2 * q2 + 1]), ffma2(c2, sxg[q2], yacc2[q2]));
          }
        }
        if (c % kChunksPerStage == kChunksPerStage - 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[st]);
        }
      }
      float yacc[NT];
#pragma unroll
      for (int q2 = 0; q2 < NT / 2; ++q2) unpair2(yacc2[q2], yacc[2 * q2], yacc[2 * q2 + 1]);
      const int n = w.n0 + row;
      if (a.gemvs || a.splits == 1) {
        if (n < w.N) {
#pragma unroll
          for (int m = 0; m < NT; ++m)
            if (m < w.M) w.y[(size_t)m * w.N + n] = yacc[m];
        }
      } else {
        const int tile = w.tile;
        float* part = a.partial + (size_t)w.u * NT * kRows;
#pragma unroll
        for (int m = 0; m < NT; ++m) part[m * kRows + row] = yacc[m];
        __threadfence();
        epi_bar();
        if (et == 0) *is_last = (atomicAdd(&a.counters[tile], 1u) == (uint32_t)(a.splits - 1)) ? 1u : 0u;
        epi_bar();
        if (*is_last) {
          __threadfence();
          if (n < a.N) {
            // eight activation rows at a time: eight independent loads per split
            for (int m0 = 0; m0 < a.M; m0 += 8) {
              float t[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) t[i] = 0.f;
              for (int s2 = 0; s2 < a.splits; ++s2) {
                const float* ps = a.partial + ((size_t)(tile * a.splits + s2) * NT + m0) * kRows + row;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  if (m0 + i < NT) t[i] += __ldcg(ps + i * kRows);
              }
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (m0 + i < a.M) a.y[(size_t)(m0 + i) * a.N + n] = t[i];
            }
          }
          if (et == 0) a.counters[tile] = 0u;
        }
        epi_bar();
      }
      gcb += nchunk;
      sgb += nchunk / kChunksPerStage;
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
// Skinny GEMM with warp-level MMA, M <= 16 (w4a16_mma_kernel)
//
// At N = 16 activation rows one tcgen05.mma (M = 128, K = 16) costs its issuing
// thread about 44 cycles whatever N is, and its A operand has to be handed from
// converter warps to the issuer through TMEM; the resulting chain of hand-offs
// sets the tcgen05 kernel's period. Here every consumer warp decodes its own
// weights into registers and multiplies them with mma.sync.m16n8k16 (f16 in,
// fp32 accumulate), so no role waits on another within a stage:
//  * The same TMA stages as the tcgen05 kernel carry the codes (128 rows x
//    512 k, 128B-swizzled), the fp16 scales and biases, and -- instead of the
//    X tile -- the stage's B fragments, prepared once per call by
//    w4a16_mma_prep_kernel (below) for the whole matrix.
//  * Warp w of the 8 consumer warps owns 64-k group w of every stage and all
//    128 rows (eight 16-row blocks): the B fragments of its group are loaded
//    once per stage and reused by all row blocks.
//  * A codes word gives four fp16x2 registers with one shift and four lop3:
//    (1024 + q) for codes 0, 4 / 2, 6 and (1024 + 16 q) for codes 1, 5 / 3, 7
//    (exact). Lane (g, c) takes words 2c, 2c + 1 of rows g and g + 8 of a row
//    block; the k order inside a group is permuted the same way in A and B, and
//    the B fragment of a (1024 + 16 q) slot holds x / 16, so one accumulator
//    per output collects 1024 X_A + 64 X_B + sum q x': it starts at minus that
//    offset (from the table), so the MMA result is sum q x' directly.
//  * Per group: y += s * 2^sigma * acc + b * sum x, in paired fp32 FMAs; at the
//    end of a 128-row tile the eight warps' partial sums are added in warp
//    order through shared memory (deterministic).
//  * Up to 8 activation rows the kernel computes one 8-column n tile (MNT = 1:
//    half the MMAs and folds of MNT = 2), and MMA row g reads weight row
//    2 (g % 4) + g / 4 of each 8-row half, which spreads the 16 lanes of one
//    shared-load phase over distinct banks.
// ---------------------------------------------------------------------------
constexpr int kMmaWarps = 8;                           // consumer warps = 64-k groups per stage
constexpr int kMmaThreads = 32 * (kMmaWarps + 1);      // + 1 producer warp
constexpr uint32_t kMmaFragStage = 8 * 2048;           // B fragments of one stage: 8 groups x 2 KB
constexpr uint32_t kMmaStageBytes = 32768 + 4096 + kMmaFragStage;  // codes, scales + biases, fragments
constexpr uint32_t kMmaRedBytes = kMmaWarps * 16 * 32 * 16;        // 64 KB: partial tiles of all warps
constexpr int kMmaTab = 48;                            // floats per group: offset[16], sum x[16], 2^sigma

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = A B + c, with the accumulator input in registers of its own
__device__ __forceinline__ void mma_16816_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                            uint32_t b0, uint32_t b1, const float (&c)[4]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %11, %12, %13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ void f16x2_to_f32(uint32_t v, float& lo, float& hi) {
  asm("{.reg .f16 l, h; mov.b32 {l, h}, %2; cvt.f32.f16 %0, l; cvt.f32.f16 %1, h;}" : "=f"(lo), "=f"(hi) : "r"(v));
}

struct MmaPrepArgs {
  const TcGemv* gemvs;  // grouped launch (null: one matrix)
  int ngemv;
  const uint16_t* x;    // one matrix
  uint32_t* frag;
  float* tab;
  int M, K;
};

// B fragments of X for every 64-k group: one warp per group. Lane (g, c) covers
// activation rows g and g + 8 at k = 16c .. 16c + 15 of the group (words 2c and
// 2c + 1); step s = 0..3 of the group uses word 2c + (s >> 1) and codes
// j = 2 (s & 1) (slots 2c, 2c + 1 <- codes j, j + 4) and j + 1 (slots 2c + 8,
// 2c + 9 <- codes j + 1, j + 5, divided by 16). sigma is per group: the
// group's largest |x| (over all rows) just below 2^15 after scaling.
__global__ void __launch_bounds__(256) w4a16_mma_prep_kernel(const MmaPrepArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = blockIdx.x * 8 + warp;
  const uint16_t* x = a.x;
  uint32_t* frag = a.frag;
  float* tab = a.tab;
  int M = a.M, K = a.K;
  if (a.gemvs) {
    const TcGemv& d = a.gemvs[blockIdx.y];
    x = d.xraw;
    frag = d.frag;
    tab = d.tab;
    M = d.M;
    K = d.K;
  }
  pdl_wait();  // x may come from the previous kernel
  if (gi < K / 64) {
    const int g = lane >> 2, c = lane & 3;
    const int k0 = gi * 64 + 16 * c;
    float v[2][16];
    float amax = 0.f;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int m = g + 8 * t;
      uint4 u0 = make_uint4(0, 0, 0, 0), u1 = make_uint4(0, 0, 0, 0);
      if (m < M) {
        const uint4* p = reinterpret_cast<const uint4*>(x + (size_t)m * K + k0);
        u0 = p[0];
        u1 = p[1];
      }
      const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[t][2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
        v[t][2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[t][i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const int sig = fp16_prescale_exp(amax);
    const float down = pow2f(-sig), down16 = pow2f(-sig - 4);
    uint32_t b[16];
    float off[2] = {0.f, 0.f}, sx[2] = {0.f, 0.f};
#pragma unroll
    for (int t = 0; t < 2; ++t) {
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int wb = 8 * (s >> 1), j = 2 * (s & 1);  // the word's first value in v, first code
        const uint32_t b0 = f16x2_of(v[t][wb + j] * down, v[t][wb + j + 4] * down);
        const uint32_t b1 = f16x2_of(v[t][wb + j + 1] * down16, v[t][wb + j + 5] * down16);
        b[(s * 2 + t) * 2] = b0;
        b[(s * 2 + t) * 2 + 1] = b1;
        float l0, h0, l1, h1;
        f16x2_to_f32(b0, l0, h0);
        f16x2_to_f32(b1, l1, h1);
        off[t] += (l0 + h0) + (l1 + h1);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) sx[t] += v[t][i];
    }
    // fragments: [u][lane][4] of this group, 16-byte units contiguous over the lanes
    uint4* fg = reinterpret_cast<uint4*>(frag + (size_t)gi * 512);
#pragma unroll
    for (int u = 0; u < 4; ++u) fg[u * 32 + lane] = make_uint4(b[4 * u], b[4 * u + 1], b[4 * u + 2], b[4 * u + 3]);
    // per row: 1024 x (the sum of its fragment values), the sum of x; lanes of one row add up
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      off[t] += __shfl_xor_sync(0xFFFFFFFFu, off[t], 1);
      off[t] += __shfl_xor_sync(0xFFFFFFFFu, off[t], 2);
      sx[t] += __shfl_xor_sync(0xFFFFFFFFu, sx[t], 1);
      sx[t] += __shfl_xor_sync(0xFFFFFFFFu, sx[t], 2);
    }
    float* tg = tab + (size_t)gi * kMmaTab;
    if (c == 0) {
      tg[g] = 1024.f * off[0];
      tg[g + 8] = 1024.f * off[1];
      tg[16 + g] = sx[0];
      tg[16 + g + 8] = sx[1];
    }
    if (lane == 0) tg[32] = pow2f(sig);
  }
  pdl_launch_dependents();
}

// MNT: n tiles of 8 activation rows that carry rows (1: M <= 8, 2: M <= 16)
template <int MNT>
__global__ void __launch_bounds__(kMmaThreads, 1)
    w4a16_mma_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_scales,
                     const __grid_constant__ CUtensorMap tm_biases, const TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  // shared layout: stages | red (64 KB) | barriers
  const uint32_t s_stages = base;
  float* red = reinterpret_cast<float*>(gbase + a.ST * kMmaStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(gbase + a.ST * kMmaStageBytes + kMmaRedBytes);
  uint64_t* empty = full + a.ST;
  volatile uint32_t* is_last = reinterpret_cast<uint32_t*>(empty + a.ST);
  // per stage: codes [2 chunks][128 rows][128 B] | scales [128][8] | biases [128][8] | fragments
  constexpr uint32_t c_off = 0, s_off = 32768, b_off = s_off + 2048, f_off = b_off + 2048;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kMmaWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();  // the fragments come from the preparation kernel

  if (warp == kMmaWarps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int issued = 0, fenced = -1;
      bool ok = true;
      for (UnitWalk w(a); w.valid() && ok; w.next(a)) {
        const int nstage = w.kper / kStageK;
        if (a.gemvs && w.g != fenced) {
          const TcGemv* d = &a.gemvs[w.g];
          tensormap_acquire(&d->codes);
          tensormap_acquire(&d->scales);
          tensormap_acquire(&d->biases);
          fenced = w.g;
        }
        const CUtensorMap* mc = a.gemvs ? &a.gemvs[w.g].codes : &tm_codes;
        const CUtensorMap* ms = a.gemvs ? &a.gemvs[w.g].scales : &tm_scales;
        const CUtensorMap* mb = a.gemvs ? &a.gemvs[w.g].biases : &tm_biases;
        for (int s = 0; s < nstage; ++s) {
          const int sg = issued, st = sg % a.ST;
          if (sg >= a.ST) ok = mbar_wait(&empty[st], ((sg / a.ST) & 1) ^ 1, a.err, kErrTcEmptyWait);
          if (!ok) break;
          const uint32_t sb = s_stages + st * kMmaStageBytes;
          mbar_arrive_expect_tx(&full[st], kMmaStageBytes);
          const int kk = w.k0 + s * kStageK;
          tma_load_3d(sb + c_off, mc, 0, w.n0, kk / 256, &full[st]);
          tma_load_2d(sb + s_off, ms, kk / 64, w.n0, &full[st]);
          tma_load_2d(sb + b_off, mb, kk / 64, w.n0, &full[st]);
          bulk_g2s(gbase + (sb - s_stages) + f_off, w.frag + (size_t)(kk / 64) * 512, kMmaFragStage, &full[st]);
          ++issued;
        }
      }
      for (int j = max(0, issued - a.ST); j < issued; ++j)
        mbar_wait(&full[j % a.ST], (j / a.ST) & 1, a.err, kErrTcDrain);
    }
    __syncwarp();  // the lane's role loop ends here: the warp reaches the final barrier converged
  } else {
    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, c = lane & 3;
    const int et = threadIdx.x;  // 0..255
    int sgc = 0;                 // stages consumed
    bool ok = true;
    for (UnitWalk w(a); w.valid(); w.next(a)) {
      const int nstage = w.kper / kStageK;
      uint64_t y2[8][2][2];  // [row block][n tile][rows g, g + 8]: (col 2c, col 2c + 1)
#pragma unroll
      for (int rb = 0; rb < 8; ++rb)
#pragma unroll
        for (int t = 0; t < 2; ++t) y2[rb][t][0] = y2[rb][t][1] = 0ull;
      // this warp's group in a stage: offsets and sums of x of its output
      // columns and 2^sigma, loaded one stage ahead (the table is in L2)
      float2 no0, no1, nx0, nx1;
      float nup;
      auto load_tab = [&](int s) {
        const float* tg = w.tab + (size_t)((w.k0 + s * kStageK) / 64 + warp) * kMmaTab;
        no0 = __ldg(reinterpret_cast<const float2*>(tg + 2 * c));
        no1 = __ldg(reinterpret_cast<const float2*>(tg + 8 + 2 * c));
        nx0 = __ldg(reinterpret_cast<const float2*>(tg + 16 + 2 * c));
        nx1 = __ldg(reinterpret_cast<const float2*>(tg + 24 + 2 * c));
        nup = __ldg(tg + 32);
      };
      load_tab(0);
      for (int s = 0; s < nstage; ++s, ++sgc) {
        const int st = sgc % a.ST;
        const float2 o0 = no0, o1 = no1, x0 = nx0, x1 = nx1;
        const float up = nup;
        if (s + 1 < nstage) load_tab(s + 1);
        if (ok) ok = mbar_wait(&full[st], (sgc / a.ST) & 1, a.err, kErrTcFullWait);
        const uint32_t sb = s_stages + st * kMmaStageBytes;
        if (ok) {
          uint32_t b[16];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint4 v = lds128(sb + f_off + warp * 2048 + (u * 32 + lane) * 16);
            b[4 * u] = v.x;
            b[4 * u + 1] = v.y;
            b[4 * u + 2] = v.z;
            b[4 * u + 3] = v.w;
          }
          const uint64_t sxp[2] = {pair2(__float_as_uint(x0.x), __float_as_uint(x0.y)),
                                   pair2(__float_as_uint(x1.x), __float_as_uint(x1.y))};
          // every row block's accumulators start at minus the group's offsets
          const float negc[2][4] = {{-o0.x, -o0.y, -o0.x, -o0.y}, {-o1.x, -o1.y, -o1.x, -o1.y}};
          // codes of group `warp`: chunk warp / 4, 32-byte segment warp % 4 of each 128-byte row;
          // words 2c, 2c + 1 are 8 bytes of 16-byte unit 2 (warp % 4) + c / 2
          const uint32_t cu = 2u * (uint32_t)(warp & 3) + ((uint32_t)c >> 1);
          const uint32_t cbase = sb + c_off + (uint32_t)(warp >> 2) * 16384 + 8u * (uint32_t)(c & 1);
#pragma unroll
          for (int rb = 0; rb < 8; ++rb) {
            // One n tile: MMA row g is weight row pg = 2 (g % 4) + g / 4 of each
            // half of the block, so the 16 lanes of one shared-load phase
            // (g = 0..3 or 4..7) read rows whose swizzled 32-byte segments fall
            // in different banks (with row g, rows g and g ^ 1 share two 16-byte
            // units); measured slower with two n tiles, which keep row g. Rows
            // r0 and r0 + 8 share the swizzle (r & 7 = pg).
            const int pg = MNT == 1 ? 2 * (g & 3) + (g >> 2) : g;
            const int r0 = 16 * rb + pg;
            const uint32_t sw = (cu ^ (uint32_t)pg) << 4;
            const uint2 w0 = lds64(cbase + r0 * 128 + sw);
            const uint2 w1 = lds64(cbase + (r0 + 8) * 128 + sw);
            uint32_t q00[4], q01[4], q10[4], q11[4];  // [row][word]
            nib8_to_f16x2_offset(w0.x, q00);
            nib8_to_f16x2_offset(w0.y, q01);
            nib8_to_f16x2_offset(w1.x, q10);
            nib8_to_f16x2_offset(w1.y, q11);
            float acc[2][4];
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
              const uint32_t* qa = (s4 >> 1) ? q01 : q00;
              const uint32_t* qb = (s4 >> 1) ? q11 : q10;
              const int p = 2 * (s4 & 1);
#pragma unroll
              for (int t = 0; t < MNT; ++t) {
                if (s4 == 0)
                  mma_16816_c(acc[t], qa[p], qb[p], qa[p + 1], qb[p + 1], b[t * 2], b[t * 2 + 1], negc[t]);
                else
                  mma_16816(acc[t], qa[p], qb[p], qa[p + 1], qb[p + 1], b[(s4 * 2 + t) * 2], b[(s4 * 2 + t) * 2 + 1]);
              }
            }
            const float s0 = f16_bits_to_f32(lds16(sb + s_off + r0 * 16 + 2 * warp));
            const float s1 = f16_bits_to_f32(lds16(sb + s_off + (r0 + 8) * 16 + 2 * warp));
            const float bb0 = f16_bits_to_f32(lds16(sb + b_off + r0 * 16 + 2 * warp));
            const float bb1 = f16_bits_to_f32(lds16(sb + b_off + (r0 + 8) * 16 + 2 * warp));
            const float cf0 = s0 * up, cf1 = s1 * up;
            const uint64_t c0 = pair2(__float_as_uint(cf0), __float_as_uint(cf0));
            const uint64_t c1 = pair2(__float_as_uint(cf1), __float_as_uint(cf1));
            const uint64_t d0 = pair2(__float_as_uint(bb0), __float_as_uint(bb0));
            const uint64_t d1 = pair2(__float_as_uint(bb1), __float_as_uint(bb1));
#pragma unroll
            for (int t = 0; t < MNT; ++t) {  // an n tile without rows stays zero
              y2[rb][t][0] = ffma2(c0, pair2(__float_as_uint(acc[t][0]), __float_as_uint(acc[t][1])),
                                   ffma2(d0, sxp[t], y2[rb][t][0]));
              y2[rb][t][1] = ffma2(c1, pair2(__float_as_uint(acc[t][2]), __float_as_uint(acc[t][3])),
                                   ffma2(d1, sxp[t], y2[rb][t][1]));
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
      // the 8 warps' partial tiles -> one tile, summed in warp order
      {
        uint4* rv = reinterpret_cast<uint4*>(red);
#pragma unroll
        for (int rb = 0; rb < 8; ++rb)
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            float e0, e1, e2, e3;
            unpair2(y2[rb][t][0], e0, e1);
            unpair2(y2[rb][t][1], e2, e3);
            rv[(warp * 16 + rb * 2 + t) * 32 + lane] =
                make_uint4(__float_as_uint(e0), __float_as_uint(e1), __float_as_uint(e2), __float_as_uint(e3));
          }
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      {
        // thread et: lane et % 32 of units 2 (et / 32), 2 (et / 32) + 1 (row block, n tile)
        const int ln = et & 31, u0 = 2 * (et >> 5);
        const int gg = ln >> 2, cc = ln & 3;
        const uint4* rv = reinterpret_cast<const uint4*>(red);
        float tot[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 4; ++e) tot[h][e] = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kMmaWarps; ++w2)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 v = rv[(w2 * 16 + u0 + h) * 32 + ln];
            tot[h][0] += __uint_as_float(v.x);
            tot[h][1] += __uint_as_float(v.y);
            tot[h][2] += __uint_as_float(v.z);
            tot[h][3] += __uint_as_float(v.w);
          }
        const bool whole = a.gemvs || a.splits == 1;
        float* part = whole ? nullptr : a.partial + (size_t)w.u * 16 * kRows;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int uu = u0 + h, rb = uu >> 1, t = uu & 1;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int row = 16 * rb + (MNT == 1 ? 2 * (gg & 3) + (gg >> 2) : gg) + 8 * (e >> 1);
            const int m = 8 * t + 2 * cc + (e & 1);
            if (whole) {
              if (m < w.M && w.n0 + row < w.N) w.y[(size_t)m * w.N + w.n0 + row] = tot[h][e];
            } else {
              part[m * kRows + row] = tot[h][e];
            }
          }
        }
        if (!whole) {
          // split K: the CTA that finishes a row tile last adds the partial tiles in split order
          __threadfence();
          asm volatile("bar.sync 1, 256;" ::: "memory");
          if (et == 0) *is_last = (atomicAdd(&a.counters[w.tile], 1u) == (uint32_t)(a.splits - 1)) ? 1u : 0u;
          asm volatile("bar.sync 1, 256;" ::: "memory");
          if (*is_last) {
            __threadfence();
            for (int q = et; q < 16 * kRows; q += 256) {
              const int m = q / kRows, row = q % kRows;
              float acc = 0.f;
              for (int s2 = 0; s2 < a.splits; ++s2)
                acc += __ldcg(a.partial + (size_t)(w.tile * a.splits + s2) * 16 * kRows + q);
              if (m < w.M && w.n0 + row < w.N) w.y[(size_t)m * w.N + w.n0 + row] = acc;
            }
            if (et == 0) a.counters[w.tile] = 0u;
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
// Host side
// ---------------------------------------------------------------------------
namespace {

// split-K happens only while 2 x tiles <= SMs, so a few hundred counters cover it
constexpr size_t kCounterBytes = 1024;

// codes {128 B, N rows, K/256 chunks} in [128][128 B] boxes (two per stage),
// scales and biases {K/64, N} in [128][8] boxes, X {64 k, M rows, K/64 groups}
// in [8][NT][64] boxes (one per stage), the rows past M read as zeros
bool tc_maps(CUtensorMap (&maps)[4], const uint32_t* wq, const uint16_t* sc, const uint16_t* bi, const uint16_t* x,
             int M, int N, int K, int NT) {
  return tmap_3d(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, 128, (uint64_t)N, (uint64_t)K / 256, (uint64_t)K / 2,
                 128, 128, kRows, 2) &&
         tmap_2d(&maps[1], CU_TENSOR_MAP_DATA_TYPE_UINT16, sc, (uint64_t)K / 64, (uint64_t)N, (uint64_t)K / 32, 8,
                 kRows, CU_TENSOR_MAP_SWIZZLE_NONE) &&
         tmap_2d(&maps[2], CU_TENSOR_MAP_DATA_TYPE_UINT16, bi, (uint64_t)K / 64, (uint64_t)N, (uint64_t)K / 32, 8,
                 kRows, CU_TENSOR_MAP_SWIZZLE_NONE) &&
         tmap_3d(&maps[3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, 64, (uint64_t)M, (uint64_t)K / 64, (uint64_t)K * 2,
                 128, 64, (uint32_t)NT, kGroupsPerStage);
}

int stages_for(int NT, uint32_t stage_bytes, size_t* smem) {
  const size_t fixed = 1024 + 512;  // alignment slack, barriers
  const size_t budget = 224 * 1024;
  const size_t sx_bytes = sizeof(float) * 2 * kChunkGroups * NT;
  const int ST = (int)std::min<size_t>(4, (budget - fixed - sx_bytes) / stage_bytes);
  *smem = fixed + sx_bytes + (size_t)ST * stage_bytes;
  return ST;
}

struct TcPlan {
  int NT, ntiles, splits, kper, nunits, ST;
  bool mma;  // M <= 16: the warp-level MMA kernel
  uint32_t stage_bytes;
  size_t smem, ws_partial, ws_counters, ws_frag, ws_tab;
};

// shared memory of the mma kernel with ST stages: alignment slack, stages, the
// 64 KB reduction buffer, barriers
size_t mma_smem(int ST) { return 1024 + (size_t)ST * kMmaStageBytes + kMmaRedBytes + 16 * (size_t)ST + 64; }

int mma_stages() {
  int ST = 4;
  while (ST > 2 && mma_smem(ST) > (size_t)device_max_smem_optin()) --ST;
  return ST;
}

template <int MNT>
cudaError_t launch_mma(dim3 grid, size_t smem, cudaStream_t stream, bool pdl, const CUtensorMap* maps,
                       const TcArgs& a) {
  cudaError_t e = allow_max_smem(w4a16_mma_kernel<MNT>);
  if (e != cudaSuccess) return e;
  return launch_kernel(w4a16_mma_kernel<MNT>, grid, dim3(kMmaThreads), smem, stream, pdl, maps[0], maps[1], maps[2],
                       a);
}

TcPlan tc_plan(int M, int N, int K, int sms) {
  TcPlan p;
  p.NT = M <= 16 ? 16 : 32;
  p.mma = M <= 16;
  p.ntiles = (N + kRows - 1) / kRows;
  const int kstages = K / kStageK;
  // split K until every SM has a unit, keeping each split a whole number of stages
  p.splits = 1;
  while (p.ntiles * p.splits * 2 <= sms && p.splits * 2 <= kstages && kstages % (p.splits * 2) == 0) p.splits *= 2;
  p.kper = K / p.splits;
  p.nunits = p.ntiles * p.splits;
  p.stage_bytes = (uint32_t)(p.NT * 1024 + 36864);
  p.ST = stages_for(p.NT, p.stage_bytes, &p.smem);
  p.ws_frag = p.ws_tab = 0;
  if (p.mma) {
    p.stage_bytes = kMmaStageBytes;
    p.ST = mma_stages();
    p.smem = mma_smem(p.ST);
    p.ws_frag = (size_t)K * 32;                       // B fragments: 2 KB per 64-k group
    p.ws_tab = (size_t)(K / 64) * kMmaTab * 4;        // offsets, sums of x, 2^sigma per group
  }
  p.ws_partial = p.splits > 1 ? sizeof(float) * (size_t)p.nunits * p.NT * kRows : 0;
  // the counters sit at a fixed place (the workspace's first bytes) for every
  // shape, so a later call never finds partial sums of another shape there
  p.ws_counters = (p.splits > 1 || p.mma) ? kCounterBytes : 0;
  return p;
}

}  // namespace

bool tc_path_ok(int M, int N, int K) {
  return M >= 3 && M <= 32 && N >= 1 && K % kStageK == 0 && K >= kStageK && K <= 32768;
}

size_t tc_workspace_size(int M, int N, int K) {
  if (!tc_path_ok(M, N, K)) return 0;
  const TcPlan p = tc_plan(M, N, K, device_sm_count());
  return p.ws_counters + p.ws_frag + p.ws_tab + p.ws_partial;
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
  if (!tc_maps(maps, wq, sc, bi, x, M, N, K, p.NT)) return cudaErrorInvalidValue;
  TcArgs a{};
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
  // workspace: counters | B fragments | group table | partial tiles
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  a.counters = p.splits > 1 ? reinterpret_cast<uint32_t*>(wsb) : nullptr;
  uint8_t* after = wsb + p.ws_counters;
  a.frag = p.mma ? reinterpret_cast<uint32_t*>(after) : nullptr;
  a.tab = p.mma ? reinterpret_cast<float*>(after + p.ws_frag) : nullptr;
  a.partial = p.splits > 1 ? reinterpret_cast<float*>(after + p.ws_frag + p.ws_tab) : nullptr;
  a.err = err;
  a.gemvs = nullptr;
  a.cta_unit0 = nullptr;
  a.cta_gemv0 = nullptr;
  // the counters start at zero (caller contract) and the last arriver of every
  // tile resets its counter, so no clearing launch is needed between calls
  const int grid = std::min(p.nunits, sms);
  if (p.mma) {
    MmaPrepArgs pa{};
    pa.x = x;
    pa.frag = const_cast<uint32_t*>(a.frag);
    pa.tab = const_cast<float*>(a.tab);
    pa.M = M;
    pa.K = K;
    cudaError_t e = launch_kernel(w4a16_mma_prep_kernel, dim3((K / 64 + 7) / 8), dim3(256), 0, stream, pdl, pa);
    if (e != cudaSuccess) return e;
    return M <= 8 ? launch_mma<1>(dim3(grid), p.smem, stream, pdl, maps, a)
                  : launch_mma<2>(dim3(grid), p.smem, stream, pdl, maps, a);
  }
  if (p.NT == 16) return launch_tc_nt<16>(maps, a, p, grid, stream, pdl);
  return launch_tc_nt<32>(maps, a, p, grid, stream, pdl);
}

// ---------------------------------------------------------------------------
// Grouped launch: the row tiles of every projection, full K each, in one
// persistent grid; each CTA takes a contiguous range of equal cost.
// ---------------------------------------------------------------------------
int tc_group_check(const TcGroupItem* list, int n) {
  // a grouped launch also takes M = 2 (single calls of M <= 2 go to the GEMV
  // kernel): the activation tile is padded to 16 rows either way
  for (int i = 0; i < n; ++i)
    if (!(list[i].M == 2 ? tc_path_ok(3, list[i].N, list[i].K) : tc_path_ok(list[i].M, list[i].N, list[i].K)))
      return 1;
  for (int i = 1; i < n; ++i)
    if ((list[i].M <= 16) != (list[0].M <= 16)) return 2;
  return 0;
}

cudaError_t tc_group_plan_build(const TcGroupItem* list, int n, int sms, TcGroupPlan* out) {
  if (n < 1 || tc_group_check(list, n) != 0) return cudaErrorInvalidValue;
  TcGroupPlan p{};
  p.NT = list[0].M <= 16 ? 16 : 32;
  p.mma = list[0].M <= 16 ? 1 : 0;
  p.mma_nt = 1;  // n tiles of 8 rows the MMA kernel computes: the group's largest M
  for (int i = 0; i < n; ++i)
    if (list[i].M > 8) p.mma_nt = 2;
  std::vector<TcGemv> g(n);
  long long units = 0;
  size_t scratch = 0;  // mma path: every projection's B fragments and group table
  for (int i = 0; i < n; ++i) scratch += (size_t)list[i].K * 32 + (size_t)(list[i].K / 64) * kMmaTab * 4;
  for (int i = 0; i < n; ++i) {
    const TcGroupItem& it = list[i];
    CUtensorMap maps[4];
    if (!tc_maps(maps, it.wq, it.scales, it.biases, it.x, it.M, it.N, it.K, p.NT)) return cudaErrorInvalidValue;
    TcGemv& d = g[i];
    d.codes = maps[0];
    d.scales = maps[1];
    d.biases = maps[2];
    d.x = maps[3];
    d.y = it.y;
    d.xraw = it.x;
    d.frag = nullptr;
    d.tab = nullptr;
    d.N = it.N;
    d.M = it.M;
    d.K = it.K;
    p.max_groups = std::max(p.max_groups, it.K / 64);
    d.unit0 = (int)units;
    units += (it.N + kRows - 1) / kRows;
    if (units >= (1LL << 30)) return cudaErrorInvalidValue;
    d.unit_end = (int)units;
  }
  // a unit costs its stages plus about one stage of hand-over at its end
  std::vector<long long> cum(units + 1, 0);
  for (const TcGemv& d : g)
    for (int u = d.unit0; u < d.unit_end; ++u) cum[u + 1] = cum[u] + d.K / kStageK + 1;
  const int grid = (int)std::max<long long>(1, std::min<long long>(sms, units));
  std::vector<int> cta(2 * grid + 1);
  cta[0] = 0;
  for (int c = 1; c < grid; ++c) {
    const long long target = cum[units] * c / grid;
    cta[c] = (int)(std::lower_bound(cum.begin(), cum.end(), target) - cum.begin());
    cta[c] = std::max(cta[c], cta[c - 1]);
  }
  cta[grid] = (int)units;
  for (int c = 0, gi = 0; c < grid; ++c) {
    while (gi + 1 < n && cta[c] >= g[gi].unit_end) ++gi;
    cta[grid + 1 + c] = gi;
  }
  p.ngemv = n;
  p.grid = grid;
  p.stage_bytes = (uint32_t)(p.NT * 1024 + 36864);
  p.ST = stages_for(p.NT, p.stage_bytes, &p.smem);
  cudaError_t e;
  if (p.mma) {
    p.stage_bytes = kMmaStageBytes;
    p.ST = mma_stages();
    p.smem = mma_smem(p.ST);
    e = cudaMalloc(&p.d_scratch, scratch);
    if (e != cudaSuccess) return e;
    uint8_t* q = static_cast<uint8_t*>(p.d_scratch);
    for (TcGemv& d : g) {
      d.frag = reinterpret_cast<uint32_t*>(q);
      q += (size_t)d.K * 32;
      d.tab = reinterpret_cast<float*>(q);
      q += (size_t)(d.K / 64) * kMmaTab * 4;
    }
  }
  e = cudaMalloc(&p.d_gemvs, sizeof(TcGemv) * n);
  if (e != cudaSuccess) {
    if (p.d_scratch) cudaFree(p.d_scratch);
    return e;
  }
  e = cudaMalloc(&p.d_cta, sizeof(int) * cta.size());
  if (e != cudaSuccess) {
    cudaFree(p.d_gemvs);
    if (p.d_scratch) cudaFree(p.d_scratch);
    return e;
  }
  e = cudaMemcpy(p.d_gemvs, g.data(), sizeof(TcGemv) * n, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(p.d_cta, cta.data(), sizeof(int) * cta.size(), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(p.d_gemvs);
    cudaFree(p.d_cta);
    if (p.d_scratch) cudaFree(p.d_scratch);
    return e;
  }
  *out = p;
  return cudaSuccess;
}

void tc_group_plan_free(TcGroupPlan* p) {
  if (p->d_gemvs) cudaFree(p->d_gemvs);
  if (p->d_cta) cudaFree(p->d_cta);
  if (p->d_scratch) cudaFree(p->d_scratch);
  p->d_gemvs = nullptr;
  p->d_cta = nullptr;
  p->d_scratch = nullptr;
}

cudaError_t tc_group_launch(const TcGroupPlan& p, uint32_t* err, cudaStream_t stream, bool pdl) {
  TcArgs a{};
  a.splits = 1;
  a.ST = p.ST;
  a.stage_bytes = p.stage_bytes;
  a.err = err;
  a.gemvs = static_cast<const TcGemv*>(p.d_gemvs);
  a.cta_unit0 = p.d_cta;
  a.cta_gemv0 = p.d_cta + p.grid + 1;
  // the kernel reads every projection's maps from its descriptor
  CUtensorMap unused[4];
  std::memset(unused, 0, sizeof(unused));
  TcPlan tp{};
  tp.smem = p.smem;
  if (p.mma) {
    // B fragments of every projection's X, then the grid over all row tiles
    MmaPrepArgs pa{};
    pa.gemvs = a.gemvs;
    pa.ngemv = p.ngemv;
    cudaError_t e = launch_kernel(w4a16_mma_prep_kernel, dim3((p.max_groups + 7) / 8, p.ngemv), dim3(256), 0,
                                  stream, pdl, pa);
    if (e != cudaSuccess) return e;
    return p.mma_nt == 1 ? launch_mma<1>(dim3(p.grid), p.smem, stream, pdl, unused, a)
                         : launch_mma<2>(dim3(p.grid), p.smem, stream, pdl, unused, a);
  }
  if (p.NT == 16) return launch_tc_nt<16>(unused, a, tp, p.grid, stream, pdl);
  return launch_tc_nt<32>(unused, a, tp, p.grid, stream, pdl);
}

}  // namespace qg
