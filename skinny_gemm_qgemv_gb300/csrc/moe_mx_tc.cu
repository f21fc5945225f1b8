// MXFP4 routed-expert MoE layer on the 5th-generation tensor cores with
// hardware block scaling (tcgen05.mma kind::mxf8f6f4, block_scale): batches of
// 33 to 64 tokens (prefill-sized batches; up to 32 tokens the warp-level MMA
// kernels of moe_mx_mma.cu are faster on this workload).
//
// "Running Kimi K3 (2.8T) on one Apple Silicon Mac" (Deltafin), section "How it
// works": the router picks 16 experts per token and only the selected experts'
// weights are read; section "Technical approach / compute": the expert GEMV
// applies the E2M1 codes and their E8M0 block scales in the same pass as the
// multiply. Here that pass is the tensor core's own block-scaled MMA: the
// weights enter it exactly as stored (E2M1 codes, one E8M0 scale per 32), so no
// instruction decodes a weight.
//
// The activations of an MMA must be a block-scaled 8-bit format too. A vector
// v is written as a sum of e4m3 terms, each with one E8M0 scale per 32
// elements: t1 = rn(v / 2^s1), r = v - t1 2^s1, t2 = rn(r / 2^s2), ... The
// products are exact in the tensor core and only the fp32 sums round. Two
// terms carry a bf16 x exactly (bf16 has 8 significant bits, e4m3 4, and the
// residual after the first term has at most 4) except for elements more than
// 2^14 below their block's largest, which keep an error below 2^-20 of it;
// three terms carry the fp32 p h of the down product to about 2^-13 of each
// element. A token owns 2 (gate/up) or 3 (down) consecutive MMA columns, the
// sum of whose results is its value; an expert multiplies only the 16-column
// blocks that hold its tokens (one MMA over the span from the first to the
// last such block).
//
// Three launches:
//  * route: CTA 0 finds every token's top-k (warp radix select on
//    order-preserving keys, ties to the lower expert index) with its softmax
//    weights, the list of distinct selected experts, per (expert, token) the
//    pair or -1, and per expert its column spans; the other CTAs write x as
//    the two-term operand image.
//  * gate/up: persistent, one CTA per SM. A unit is (selected expert, 128
//    rows of I) for both matrices; the units' 256-k stages form one list that
//    the CTAs split into equal contiguous ranges (a unit cut by a range
//    boundary is finished by whichever CTA adds its part last, summing the
//    parts in CTA order). Three rings in shared memory: weight slots (one
//    matrix, 128 rows x 256 k: E2M1 codes unpacked to a byte each by the tensor
//    map, 128B-swizzled), x operand slots (the stage's column span), and
//    512-k windows (the x scale rows); the weight rows' E8M0 bytes are read by
//    the scale warps themselves, a few windows ahead, with plain loads.
//    Warp roles: a TMA producer; an MMA issuer (per 32 k one MMA into the gate
//    and one into the up accumulator in TMEM); four scale warps (each thread
//    one weight row: its window's E8M0 bytes into TMEM with tcgen05.st, in the
//    layout the MMA reads: row m at lane m, column base + m / 32, one byte per
//    32-k block selected by the instruction); four epilogue warps (tcgen05.ld
//    of a finished unit: g, u per token, h = silu(g) u in fp32, p h as the
//    down's three-term operand image).
//  * down: the same machinery over units of 128 rows of H whose stages walk
//    every selected expert; the MMA columns are the batch's tokens (zero where
//    a token did not pick the expert), so one TMEM accumulator collects
//    y_t = sum_j p_j W_d[e_j] h_j over all experts of the layer. A unit's first
//    stage in a CTA multiplies every column, which starts the accumulator.
// Every wait is bounded; on a timeout a kernel records a code in the error
// word, stops issuing work, lets its copies and MMAs land and exits.
// Every wait is bounded; on a timeout a kernel records a code in the error
// word, stops issuing work, lets its copies and MMAs land and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include "moe_route.cuh"
#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

namespace {

constexpr int kTcWarps = 11;  // weight producer, MMA issuer, 4 epilogue, 4 scale warps, operand producer
constexpr int kNW = 3;        // window slots
constexpr int kTcThreads = 32 * kTcWarps;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: accumulators in [0, 256): two buffers (b at 128 b; gate/up: g
// at +0, u at +64) while the batch's columns fit, else one (gate/up: g at 0,
// u at 128); scale windows of 64 columns from 256: SFA | SFA (up) | SFB
constexpr uint32_t kSfCol = 256;
constexpr uint32_t kSfWin = 64;
constexpr size_t kTcSmemMax = 227 * 1024;
constexpr int kImgThreads = 1024;

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  // tcgen05 shared-memory matrix descriptor, K-major, 128-byte swizzle:
  // start >> 4, leading offset unused (1), 1024 B between 8-row groups,
  // descriptor version 1, swizzle mode 2.
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ void mma_mx(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d),
      "l"(ad), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc));
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// The 16 E8M0 bytes of this thread's weight row for one 512-k window (four
// words, one per group of four 32-k blocks) into 16 columns of its lane, word g
// in all four columns 4g .. 4g + 3: the MMA for group g (scale address
// base + 4g) reads row m's word at column base + 4g + m / 32, so every row
// finds its own word and every address stays 4-column aligned.
__device__ __forceinline__ void tmem_st_sfa(uint32_t taddr, uint4 v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %1, %1, %1, %2, %2, %2, %2, %3, %3, %3, %3, %4, %4, %4, "
      "%4};" ::"r"(taddr),
      "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
      : "memory");
}
// The E8M0 scales of the B operand (the MMA's columns) for one 512-k window:
// lane L gets, for group g and j = 0..3, the word of column L % 32 + 32 j at
// column base + 4g + j. The MMA for group g (scale address base + 4g) reads
// column n's word at column base + 4g + n / 32 of lane n (or of lane n % 32:
// both hold it).
__device__ __forceinline__ void tmem_st_sfb(uint32_t taddr, const uint4 (&c)[4]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(c[0].x), "r"(c[1].x), "r"(c[2].x), "r"(c[3].x), "r"(c[0].y), "r"(c[1].y), "r"(c[2].y), "r"(c[3].y),
      "r"(c[0].z), "r"(c[1].z), "r"(c[2].z), "r"(c[3].z), "r"(c[0].w), "r"(c[1].w), "r"(c[2].w), "r"(c[3].w)
      : "memory");
}
// The same for up to 256 columns: group g at base + 8g, column n's word at
// base + 8g + n / 32 (j = 0..7)
__device__ __forceinline__ void tmem_st_sfb8(uint32_t taddr, const uint4 (&c)[8]) {
  uint32_t w[32];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    w[j] = c[j].x;
    w[8 + j] = c[j].y;
    w[16 + j] = c[j].z;
    w[24 + j] = c[j].w;
  }
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "r"(w[8]),
      "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]), "r"(w[16]),
      "r"(w[17]), "r"(w[18]), "r"(w[19]), "r"(w[20]), "r"(w[21]), "r"(w[22]), "r"(w[23]), "r"(w[24]),
      "r"(w[25]), "r"(w[26]), "r"(w[27]), "r"(w[28]), "r"(w[29]), "r"(w[30]), "r"(w[31])
      : "memory");
}
// 16 zero columns of this thread's lane
__device__ __forceinline__ void tmem_st_zero16(uint32_t taddr) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, "
      "%1};" ::"r"(taddr),
      "r"(0u)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 16 consecutive 32-bit columns of this thread's lane, waited for
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&f)[16]) {
  uint32_t v[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(v[i]);
}
__device__ __forceinline__ uint4 ldg_nc16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
constexpr int kSfAhead = 4;  // windows of weight-row scales a scale warp holds in registers

__device__ __forceinline__ void tma_3d_hint(uint32_t dst, const void* tm, int x, int y, int z, uint64_t* bar,
                                            uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst), "l"(src),
      "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Bounded mbarrier wait that also gives up once another role set the CTA's
// abort flag.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                              uint32_t* err, uint32_t code) {
  for (uint32_t i = 0; i < kMaxPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort_flag) return false;
  }
  report_error(err, code);
  *abort_flag = 1u;
  return false;
}

// 2^e for -127 <= e <= 127 (2^-127 as the fp32 subnormal)
__device__ __forceinline__ float pow2_any(int e) {
  return e >= -126 ? __int_as_float((e + 127) << 23) : __int_as_float(0x00400000);
}

// One e4m3 term of v over the warp's 32 lanes (one 32-element block): the
// block scale 2^s puts the largest |v| in (224, 448]; the lane's code is
// rn(v / 2^s) and v becomes the residual v - code 2^s (exact in fp32). The
// block's E8M0 byte s + 127 is returned in every lane.
__device__ __forceinline__ uint32_t e4m3_term(float& v, uint32_t& sbyte) {
  float m = fabsf(v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  int s = 0;
  if (m > 0.f) {
    int e;
    const float f = frexpf(m, &e);  // m = f 2^e, f in [0.5, 1)
    s = max(f <= 0.875f ? e - 9 : e - 8, -127);
  }
  const float qv = v * pow2_any(-s);
  uint16_t pk;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pk) : "f"(0.f), "f"(qv));
  const uint32_t code = pk & 0xFFu;
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)code));
  float back;
  asm("{.reg .b16 lo, hi; mov.b32 {lo, hi}, %1; cvt.f32.f16 %0, lo;}" : "=f"(back) : "r"(h2));
  v -= back * pow2_any(s);
  sbyte = (uint32_t)(s + 127);
  return code;
}

// The scale rows of MMA columns L % 32 + 32 j (j = 0..3) of a B span starting at
// image row r0, from a window's [rows][16 B] scales in shared memory; rows past
// the image hold unit scales
__device__ __forceinline__ void load_sfb(uint32_t src, int r0, int nrows, int lane, uint4 (&c)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int row = r0 + (lane & 31) + 32 * j;
    c[j] = row < nrows ? lds128(src + 16u * (uint32_t)row) : make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
  }
}

// The same for eight rows (up to 256 columns)
__device__ __forceinline__ void load_sfb8(uint32_t src, int r0, int nrows, int lane, uint4 (&c)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int row = r0 + (lane & 31) + 32 * j;
    c[j] = row < nrows ? lds128(src + 16u * (uint32_t)row) : make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
  }
}

// Byte offset of element (row n, column k) in an operand image of N rows:
// [k / 128][N][128 B], the 16-byte unit (k % 128) / 16 of row n stored at
// position ((k % 128) / 16) ^ (n % 8) -- the 128B-swizzled K-major layout the
// MMA reads, so a stage of KS columns is one contiguous KS * N byte copy.
__device__ __forceinline__ uint32_t img_off(int k, int n, int N) {
  return ((uint32_t)(k >> 7) * (uint32_t)N + (uint32_t)n) * 128u + (((((uint32_t)k >> 4) & 7u) ^ ((uint32_t)n & 7u)) << 4) +
         ((uint32_t)k & 15u);
}

}  // namespace


// ---------------------------------------------------------------------------
// route + x operand image
// ---------------------------------------------------------------------------
struct TcRouteArgs {
  const float* logits;   // [T][E]
  const uint16_t* x;     // [T][H] bf16
  int T, H, E, top_k, Ng;
  int32_t* idx;          // [T][k]
  float* wts;            // [T][k]
  int32_t* elist;        // [D] selected experts, ascending
  int32_t* nexp;         // D
  int32_t* epair;        // [D][T] pair t * k + j, or -1
  int32_t* gspan;        // [D] first | last << 16 16-column block of the expert's tokens (gate/up)
  int32_t* dspan;        // [D] the same for the down's three columns per token
  uint8_t* ximg;         // [H / 128][Ng][128] two-term e4m3 image of x (rows 2t, 2t + 1)
  uint8_t* xsf;          // [H / 512][Ng][16] E8M0 of the image rows per 512-k window
  uint32_t* gcnt;        // [ngcnt] gate/up unit counters (zeroed here)
  uint32_t* dcnt;        // [ndcnt] down unit counters
  int ngcnt, ndcnt;
};

template <int PER>
__global__ void __launch_bounds__(kImgThreads) moe_tc_route_kernel(const TcRouteArgs a) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();  // the logits and x may come from the previous kernel; the workspace is free
  if (blockIdx.x > 0) {
    // x as two e4m3 terms per element: one warp per (token, 32-element block);
    // the padding rows 2T .. Ng - 1 are zero with unit scales
    const int nkb = a.H >> 5;
    const int tasks = (a.Ng >> 1) * nkb;
    for (int task = (blockIdx.x - 1) * 32 + warp; task < tasks; task += (gridDim.x - 1) * 32) {
      const int t = task / nkb, kb = task - t * nkb, k = 32 * kb + lane;
      float v = t < a.T ? bf16_bits_to_f32(a.x[(size_t)t * a.H + k]) : 0.f;
      uint32_t s0, s1;
      const uint32_t c0 = e4m3_term(v, s0);
      const uint32_t c1 = e4m3_term(v, s1);
      a.ximg[img_off(k, 2 * t, a.Ng)] = (uint8_t)c0;
      a.ximg[img_off(k, 2 * t + 1, a.Ng)] = (uint8_t)c1;
      if (lane == 0) {
        uint8_t* sf = a.xsf + ((size_t)(kb >> 4) * a.Ng + 2 * t) * 16 + (kb & 15);
        sf[0] = (uint8_t)s0;
        sf[16] = (uint8_t)s1;
      }
    }
    pdl_launch_dependents();
    return;
  }
  __shared__ uint32_t sel_k[32][32];
  __shared__ int sel_e[32][32];
  __shared__ int pe[kImgThreads];    // expert of pair p = t * top_k + slot
  __shared__ int mark[kImgThreads];  // expert selected, then its slot in the list
  __shared__ int wsum[33];
  for (int i = tid; i < a.ngcnt; i += kImgThreads) a.gcnt[i] = 0u;
  for (int i = tid; i < a.ndcnt; i += kImgThreads) a.dcnt[i] = 0u;
  mark[tid] = 0;
  __syncthreads();
  for (int t = warp; t < a.T; t += 32)
    route_token<PER>(a.logits + (size_t)t * a.E, a.E, a.top_k, lane, sel_k[warp], sel_e[warp],
                     a.idx + (size_t)t * a.top_k, a.wts + (size_t)t * a.top_k, pe + t * a.top_k);
  __syncthreads();
  const int P = a.T * a.top_k;
  for (int p = tid; p < P; p += kImgThreads) mark[pe[p]] = 1;
  __syncthreads();
  int D;
  const int sel = tid < a.E ? mark[tid] : 0;
  const int slot = cta_exclusive_scan(sel, wsum, D);
  if (sel) a.elist[slot] = tid;
  if (tid < a.E) mark[tid] = slot;
  for (int i = tid; i < D * a.T; i += kImgThreads) a.epair[i] = -1;
  __syncthreads();
  for (int p = tid; p < P; p += kImgThreads) a.epair[mark[pe[p]] * a.T + p / a.top_k] = p;
  __syncthreads();
  // column spans: token t owns gate/up columns 2t, 2t + 1 and down columns 3t .. 3t + 2
  for (int d = tid; d < D; d += kImgThreads) {
    int glo = 1 << 20, ghi = -1, dlo = 1 << 20, dhi = -1;
    for (int t = 0; t < a.T; ++t)
      if (a.epair[d * a.T + t] >= 0) {
        glo = min(glo, t >> 3);
        ghi = max(ghi, t >> 3);
        dlo = min(dlo, (3 * t) >> 4);
        dhi = max(dhi, (3 * t + 2) >> 4);
      }
    a.gspan[d] = glo | (ghi << 16);
    a.dspan[d] = dlo | (dhi << 16);
  }
  if (tid == 0) a.nexp[0] = D;
  pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// shared pieces of the two expert kernels
// ---------------------------------------------------------------------------
namespace {

constexpr int kKS = 256;              // k per stage
constexpr uint32_t kASlot = 32768;    // one weight matrix, 128 rows x 256 k, one byte per code
constexpr uint32_t kIdBase = (5u << 7) | (1u << 23) | ((128u >> 4) << 24);  // E2M1 x E4M3, E8M0, M = 128

// the contiguous stage range [q0, q1) of this CTA out of `total`, with the
// common range length P
struct StageRange {
  int q0, q1, P;
  __device__ StageRange(int total) {
    P = (total + (int)gridDim.x - 1) / (int)gridDim.x;
    q0 = min(total, (int)blockIdx.x * P);
    q1 = min(total, q0 + P);
  }
};

// CTAs holding part of unit u (stages [u S, (u + 1) S)) under range length P,
// and which of a CTA's two partial slots holds it (0: the first unit of the
// CTA's range, 1: its last)
__device__ __forceinline__ void unit_ctas(int u, int S, int P, int& cf, int& cl) {
  cf = (u * S) / P;
  cl = ((u + 1) * S - 1) / P;
}
__device__ __forceinline__ int part_slot(int c, int u, int S, int P) { return u == (c * P) / S ? 0 : 1; }

__device__ __forceinline__ void span_of(int v, int& lo, int& nb) {
  lo = v & 0xFFFF;
  nb = 16 * ((v >> 16) - lo + 1);
}

}  // namespace

// ---------------------------------------------------------------------------
// gate/up + SwiGLU + the down's operand image
// ---------------------------------------------------------------------------
struct TcGuArgs {
  const uint8_t* gs;     // gate E8M0 [E][I][H / 32]
  const uint8_t* us;     // up E8M0
  const uint8_t* ximg;   // x operand image [H / 128][Ng][128]
  const uint8_t* xsf;    // x scale rows [H / 512][Ng][16]
  const int32_t* elist;  // [D]
  const int32_t* nexp;
  const int32_t* epair;  // [D][T]
  const int32_t* gspan;  // [D]
  const float* wts;      // [P]
  float* h;              // [P][I] fp32
  uint8_t* dimg;         // [D][I / 128][Nd][128] three-term image of p h
  uint8_t* dsf;          // [D][I / 512][Nd][16] its scale rows
  float* part;           // [grid][2 slots][2 (g, u)][T][128]
  uint32_t* cnt;         // [D * I / 128]
  uint32_t* err;
  int T, H, I, Ng, Nd, ST, NB;  // weight slots, x operand slots
  int NA;                       // accumulator buffers (1 or 2)
  uint32_t WB;                  // window slot bytes (the x scale rows, 16 per row)
};


__global__ void __launch_bounds__(kTcThreads, 1)
    moe_tc_gu_kernel(const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_u,
                     const TcGuArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const int T = a.T, H = a.H, I = a.I, Ng = a.Ng, ST = a.ST, NB = a.NB;
  // shared layout: weight slots | x operand slots | windows | barriers
  const uint32_t sA = base, sB = sA + ST * kASlot, sW = sB + NB * Ng * kKS;
  uint64_t* afull = reinterpret_cast<uint64_t*>(gbase + (sW - base) + kNW * a.WB);
  uint64_t* aempty = afull + ST;
  uint64_t* bfull = aempty + ST;  // [NB]
  uint64_t* bempty = bfull + NB;
  uint64_t* wfull = bempty + NB;  // [kNW] window data landed
  uint64_t* wempty = wfull + kNW; // [kNW] the window's MMAs completed
  uint64_t* sff = wempty + kNW;   // [kNW] the window's scales are in TMEM
  uint64_t* accf = sff + kNW;     // [2] an accumulator buffer holds a finished unit (part)
  uint64_t* acce = accf + 2;      // [2] the epilogue read an accumulator buffer
  uint64_t* done = acce + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* is_last = tmem_slot + 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < ST; ++i) {
      mbar_init(&afull[i], 1);
      mbar_init(&aempty[i], 1);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(&bfull[i], 1);
      mbar_init(&bempty[i], 1);
    }
    for (int i = 0; i < kNW; ++i) {
      mbar_init(&wfull[i], 1);
      mbar_init(&wempty[i], 1);
      mbar_init(&sff[i], 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accf[i], 1);
      mbar_init(&acce[i], 4);
    }
    mbar_init(done, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  pdl_wait();  // the expert list and the x image come from the route kernel
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const int RT = I >> 7, S = H / kKS;  // S is even: a 512-k window is two stages
  const int D = *a.nexp;
  const StageRange R(D * RT * S);
  const int q0 = R.q0, q1 = R.q1;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int na = 0, nw = 0;  // weight slots and windows issued
      for (int q = q0; q < q1 && !*abort_flag; ++q) {
        const int u = q / S, j = q - u * S, d = u / RT, r = u - d * RT;
        const int row = __ldg(a.elist + d) * I + 128 * r;
        if (q == q0 || (j & 1) == 0) {
          const int wsl = nw % kNW;
          if (nw >= kNW && !wait_or_abort(&wempty[wsl], ((nw / kNW) & 1) ^ 1, abort_flag, a.err, kErrMoeWait)) break;
          const uint32_t sw = sW + wsl * a.WB;
          mbar_arrive_expect_tx(&wfull[wsl], 16u * Ng);
          bulk_load(sw, a.xsf + (size_t)(j >> 1) * Ng * 16, 16u * Ng, &wfull[wsl]);
          ++nw;
        }
        bool stop = false;
        for (int mat = 0; mat < 2; ++mat) {
          const int st = na % ST;
          if (na >= ST && !wait_or_abort(&aempty[st], ((na / ST) & 1) ^ 1, abort_flag, a.err, kErrMoeWait)) {
            stop = true;
            break;
          }
          mbar_arrive_expect_tx(&afull[st], kASlot / 2);
          tma_3d_hint(sA + st * kASlot, mat ? &tm_u : &tm_g, 0, row, 2 * j, &afull[st], pol);
          ++na;
        }
        if (stop) break;
      }
      // copies still in flight land before the CTA may exit
      for (int k = max(0, na - ST); k < na; ++k) mbar_wait(&afull[k % ST], (k / ST) & 1, a.err, kErrMoeWait);
      for (int k = max(0, nw - kNW); k < nw; ++k) mbar_wait(&wfull[k % kNW], (k / kNW) & 1, a.err, kErrMoeWait);
    }
    __syncwarp();  // the lane's role loop ends here: the warp reaches the final barrier converged
  } else if (warp == 10) {
    // ------------------------------------------------------------ x operand producer
    if (lane == 0) {
      int nbi = 0;
      for (int q = q0; q < q1 && !*abort_flag; ++q) {
        const int u = q / S, j = q - u * S, d = u / RT;
        const int bsl = nbi % NB;
        if (nbi >= NB && !wait_or_abort(&bempty[bsl], ((nbi / NB) & 1) ^ 1, abort_flag, a.err, kErrMoeWait)) break;
        int lo, nb;
        span_of(__ldg(a.gspan + d), lo, nb);
        const uint32_t sb = sB + bsl * Ng * kKS;
        mbar_arrive_expect_tx(&bfull[bsl], (uint32_t)nb * kKS);
        for (int c = 0; c < 2; ++c)
          bulk_load(sb + c * nb * 128, a.ximg + ((size_t)(2 * j + c) * Ng + 16 * lo) * 128, nb * 128, &bfull[bsl]);
        ++nbi;
      }
      for (int k = max(0, nbi - NB); k < nbi; ++k) mbar_wait(&bfull[k % NB], (k / NB) & 1, a.err, kErrMoeWait);
    }
    __syncwarp();  // the lane's role loop ends here: the warp reaches the final barrier converged
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int i = 0, na = 0, uc = -1, wc = -1, b = 0, wsl = 0;
      uint32_t acc_on = 0;
      for (int q = q0; q < q1 && !*abort_flag; ++q, ++i) {
        const int u = q / S, j = q - u * S, d = u / RT;
        if (q == q0 || j == 0) {
          ++uc;
          b = uc % a.NA;
          if (uc >= a.NA && !wait_or_abort(&acce[b], ((uc / a.NA) & 1) ^ 1, abort_flag, a.err, kErrMoeWait)) break;
          acc_on = 0;
        }
        if (q == q0 || (j & 1) == 0) {
          ++wc;
          wsl = wc % kNW;
          if (!wait_or_abort(&sff[wsl], (wc / kNW) & 1, abort_flag, a.err, kErrMoeWait)) break;
        }
        const uint32_t sfw = tbase + kSfCol + kSfWin * wsl;
        const int bsl = i % NB;
        if (!wait_or_abort(&bfull[bsl], (i / NB) & 1, abort_flag, a.err, kErrMoeWait)) break;
        int lo, nb;
        span_of(__ldg(a.gspan + d), lo, nb);
        const uint64_t bd0 = sw128_desc(sB + bsl * Ng * kKS);
        const uint32_t bchunk = (uint32_t)nb * 8;  // descriptor units between the two 128-k chunks
        const uint32_t idn = (uint32_t)(nb >> 3) << 17;
        const uint32_t g0 = (uint32_t)(j & 1) * 2;  // first scale group of this stage in its window
        const int uoff = a.NA == 2 ? 64 : 128;      // the up accumulator's column offset
        bool stop = false;
        for (int mat = 0; mat < 2; ++mat, ++na) {
          const int st = na % ST;
          if (!wait_or_abort(&afull[st], (na / ST) & 1, abort_flag, a.err, kErrMoeWait)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint64_t ad0 = sw128_desc(sA + st * kASlot);
          const uint32_t dcol = tbase + (uint32_t)(b * 128 + mat * uoff + 16 * lo);
          const uint32_t sfa = sfw + 16 * mat;
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const uint32_t c = jj >> 2, kk = jj & 3;
            mma_mx(dcol, ad0 + c * 1024 + 2 * kk, bd0 + c * bchunk + 2 * kk, kIdBase | idn | (kk << 4) | (kk << 29),
                   sfa + 4 * (g0 + c), sfw + 32 + 4 * (g0 + c), acc_on | (jj > 0 ? 1u : 0u));
          }
          tc_commit(&aempty[st]);
        }
        if (stop) break;
        tc_commit(&bempty[bsl]);
        if ((j & 1) == 1 || q + 1 == q1) tc_commit(&wempty[wsl]);
        if (j == S - 1 || q + 1 == q1) tc_commit(&accf[b]);
        acc_on = 1;
      }
      // every MMA this thread issued completes before TMEM is released
      tc_commit(done);
      mbar_wait(done, 0, a.err, kErrMoeWait);
    }
    __syncwarp();  // the lane's role loop ends here: the warp reaches the final barrier converged
  } else if (warp >= 6) {
    // ------------------------------------------------------------ scale warps
    // thread = weight row m of the 128-row tile; TMEM lane quarter = warp % 4.
    // Per 512-k window the thread's 16 E8M0 bytes of its gate and up row are
    // read from global memory kSfAhead windows ahead (plain loads keep the TMA
    // unit free for the weights); they and the x scale rows of the window
    // (landed in the window slot) go to TMEM in the layout the MMA reads.
    // Reusing a window slot implies its previous window's MMAs completed, so
    // its TMEM columns are free too.
    const int qd = warp & 3, m = 32 * qd + lane;
    const uint32_t tq = tbase + ((uint32_t)(32 * qd) << 16) + kSfCol;
    const size_t rowb = (size_t)(H / 32);
    const int nwin = q0 < q1 ? (q1 - 1) / 2 - q0 / 2 + 1 : 0;
    auto wstart = [&](int k) { return k == 0 ? q0 : 2 * (q0 / 2 + k); };
    auto load = [&](int k, uint4& ga, uint4& ua) {
      const int q = wstart(k), u = q / S, j = q - u * S, d = u / RT, r = u - d * RT;
      const size_t row = (size_t)__ldg(a.elist + d) * I + 128 * r + m;
      ga = ldg_nc16(a.gs + row * rowb + 16 * (j >> 1));
      ua = ldg_nc16(a.us + row * rowb + 16 * (j >> 1));
    };
    uint4 ga[kSfAhead], ua[kSfAhead];
#pragma unroll
    for (int t = 0; t < kSfAhead; ++t)
      if (t < nwin) load(t, ga[t], ua[t]);
    bool stop = false;
    for (int k0 = 0; k0 < nwin && !stop && !*abort_flag; k0 += kSfAhead) {
#pragma unroll
      for (int t = 0; t < kSfAhead; ++t) {
        const int k = k0 + t;
        if (k >= nwin || stop) break;
        const int wsl = k % kNW;
        if (!wait_or_abort(&wfull[wsl], (k / kNW) & 1, abort_flag, a.err, kErrMoeWait)) {
          stop = true;
          break;
        }
        tc_fence_after();
        const int d = (wstart(k) / S) / RT;
        int lo, nb;
        span_of(__ldg(a.gspan + d), lo, nb);
        uint4 cb[4];
        load_sfb(sW + wsl * a.WB, 16 * lo, Ng, lane, cb);
        tmem_st_sfa(tq + kSfWin * wsl, ga[t]);
        tmem_st_sfa(tq + kSfWin * wsl + 16, ua[t]);
        tmem_st_sfb(tq + kSfWin * wsl + 32, cb);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sff[wsl]);
        if (k + kSfAhead < nwin) load(k + kSfAhead, ga[t], ua[t]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int qd = warp & 3, m = 32 * qd + lane;
    const int et = threadIdx.x - 64;  // 0..127
    const uint32_t tl = tbase + ((uint32_t)(32 * qd) << 16);
    const int Nd = a.Nd;
    const size_t dimg_e = (size_t)I * Nd;  // bytes of one expert's image
    const size_t dsf_e = (size_t)(I / 512) * Nd * 16;  // bytes of one expert's scale rows
    // g, u of 8 tokens t0.. of row i of unit (d, r): h, and p h as three e4m3 terms
    auto finish = [&](int d, int i, int t0, const float (&g8)[8], const float (&u8)[8]) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int t = t0 + k;
        if (t >= T) break;
        const int p = __ldg(a.epair + d * T + t);
        float v = 0.f;
        if (p >= 0) {
          const float gv = g8[k], uv = u8[k];
          const float hv = gv / (1.f + expf(-gv)) * uv;
          a.h[(size_t)p * I + i] = hv;
          v = __ldg(a.wts + p) * hv;
        }
#pragma unroll
        for (int term = 0; term < 3; ++term) {
          uint32_t sb;
          const uint32_t c = e4m3_term(v, sb);
          const int n = 3 * t + term;
          a.dimg[d * dimg_e + img_off(i, n, Nd)] = (uint8_t)c;
          if (lane == 0) a.dsf[d * dsf_e + ((size_t)(i >> 9) * Nd + n) * 16 + ((i >> 5) & 15)] = (uint8_t)sb;
        }
      }
    };
    // padding columns 3T .. Nd - 1 of the down operand: zero, unit scale
    auto pad = [&](int d, int i) {
      for (int n = 3 * T; n < Nd; ++n) {
        a.dimg[d * dimg_e + img_off(i, n, Nd)] = 0;
        if (lane == 0) a.dsf[d * dsf_e + ((size_t)(i >> 9) * Nd + n) * 16 + ((i >> 5) & 15)] = 127;
      }
    };
    int uc = -1;
    const int ufirst = q0 < q1 ? q0 / S : 0, ulast = q0 < q1 ? (q1 - 1) / S : -1;
    for (int u = ufirst; u <= ulast && !*abort_flag; ++u) {
      ++uc;
      const int b = uc % a.NA;
      if (!wait_or_abort(&accf[b], (uc / a.NA) & 1, abort_flag, a.err, kErrMoeWait)) break;
      tc_fence_after();
      const int d = u / RT, r = u - d * RT, i = 128 * r + m;
      int cf, cl;
      unit_ctas(u, S, R.P, cf, cl);
      const uint32_t dg = tl + (uint32_t)(b * 128), du = dg + (a.NA == 2 ? 64 : 128);
      if (cf == cl) {
        // the whole unit ran here
        for (int t0 = 0; t0 < T; t0 += 8) {
          float vg[16], vu[16], g8[8], u8[8];
          tmem_ld16(dg + 2 * t0, vg);
          tmem_ld16(du + 2 * t0, vu);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            g8[k] = vg[2 * k] + vg[2 * k + 1];
            u8[k] = vu[2 * k] + vu[2 * k + 1];
          }
          finish(d, i, t0, g8, u8);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce[b]);
        pad(d, i);
      } else {
        // part of the unit: g, u per token into this CTA's slot; the CTA
        // adding the last part sums them in CTA order
        const int slot = part_slot(blockIdx.x, u, S, R.P);
        float* pp = a.part + (size_t)(blockIdx.x * 2 + slot) * 2 * T * 128;
        for (int t0 = 0; t0 < T; t0 += 8) {
          float vg[16], vu[16];
          tmem_ld16(dg + 2 * t0, vg);
          tmem_ld16(du + 2 * t0, vu);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (t0 + k < T) {
              pp[(size_t)(t0 + k) * 128 + m] = vg[2 * k] + vg[2 * k + 1];
              pp[(size_t)(T + t0 + k) * 128 + m] = vu[2 * k] + vu[2 * k + 1];
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce[b]);
        __threadfence();
        epi_bar();
        if (et == 0) *is_last = (atomicAdd(&a.cnt[u], 1u) == (uint32_t)(cl - cf)) ? 1u : 0u;
        epi_bar();
        if (*is_last) {
          __threadfence();
          for (int t0 = 0; t0 < T; t0 += 8) {
            float g8[8], u8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) g8[k] = u8[k] = 0.f;
            for (int c = cf; c <= cl; ++c) {
              const float* qp = a.part + (size_t)(c * 2 + part_slot(c, u, S, R.P)) * 2 * T * 128;
#pragma unroll
              for (int k = 0; k < 8; ++k)
                if (t0 + k < T) {
                  g8[k] += __ldcg(qp + (size_t)(t0 + k) * 128 + m);
                  u8[k] += __ldcg(qp + (size_t)(T + t0 + k) * 128 + m);
                }
            }
            finish(d, i, t0, g8, u8);
          }
          pad(d, i);
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
// down + routing-weighted combine
// ---------------------------------------------------------------------------
struct TcDnArgs {
  const uint8_t* ds;     // down E8M0 [E][H][I / 32]
  const uint8_t* dimg;   // [D][I / 128][Nd][128]
  const uint8_t* dsf;    // [D][I / 512][Nd][16]
  const int32_t* elist;
  const int32_t* nexp;
  const int32_t* dspan;  // [D]
  float* y;              // [T][H]
  float* part;           // [grid][2 slots][T][128]
  uint32_t* cnt;         // [H / 128]
  uint32_t* err;
  int T, H, I, Nd, ST, NB;  // weight slots, operand slots
  int NA;                   // accumulator buffers (1 or 2)
  uint32_t WB;              // window slot bytes (the h scale rows, 16 per row)
};


__global__ void __launch_bounds__(kTcThreads, 1)
    moe_tc_dn_kernel(const __grid_constant__ CUtensorMap tm_d, const TcDnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const int T = a.T, H = a.H, I = a.I, Nd = a.Nd, ST = a.ST, NB = a.NB;
  // shared layout: weight slots | operand slots | windows | barriers
  const uint32_t sA = base, sB = sA + ST * kASlot, sW = sB + NB * Nd * kKS;
  uint64_t* afull = reinterpret_cast<uint64_t*>(gbase + (sW - base) + kNW * a.WB);
  uint64_t* aempty = afull + ST;
  uint64_t* bfull = aempty + ST;  // [NB]
  uint64_t* bempty = bfull + NB;
  uint64_t* wfull = bempty + NB;  // [kNW]
  uint64_t* wempty = wfull + kNW;
  uint64_t* sff = wempty + kNW;
  uint64_t* accf = sff + kNW;
  uint64_t* acce = accf + 2;
  uint64_t* done = acce + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* is_last = tmem_slot + 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < ST; ++i) {
      mbar_init(&afull[i], 1);
      mbar_init(&aempty[i], 1);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(&bfull[i], 1);
      mbar_init(&bempty[i], 1);
    }
    for (int i = 0; i < kNW; ++i) {
      mbar_init(&wfull[i], 1);
      mbar_init(&wempty[i], 1);
      mbar_init(&sff[i], 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accf[i], 1);
      mbar_init(&acce[i], 4);
    }
    mbar_init(done, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  pdl_wait();  // the operand images come from gate/up
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const int SI = I / kKS;  // stages per expert of a unit (even)
  const int D = *a.nexp;
  const int S = D * SI;    // stages per unit (128 rows of H over every selected expert)
  const StageRange R((H >> 7) * S);
  const int q0 = R.q0, q1 = R.q1;
  // columns multiplied for expert d: the span of its tokens (the epilogue
  // warps zero an accumulator before its unit, so every MMA accumulates)
  auto span = [&](int d, int& lo, int& nb) { span_of(__ldg(a.dspan + d), lo, nb); };

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int na = 0, nw = 0;  // weight copies and windows issued
      for (int q = q0; q < q1 && !*abort_flag; ++q) {
        const int r = q / S, j = q - r * S, d = j / SI, jj = j - d * SI;
        const int row = __ldg(a.elist + d) * H + 128 * r;
        if (q == q0 || (jj & 1) == 0) {
          const int wsl = nw % kNW;
          if (nw >= kNW && !wait_or_abort(&wempty[wsl], ((nw / kNW) & 1) ^ 1, abort_flag, a.err, kErrMoeWait)) break;
          const uint32_t sw = sW + wsl * a.WB;
          mbar_arrive_expect_tx(&wfull[wsl], 16u * Nd);
          bulk_load(sw, a.dsf + ((size_t)d * (I / 512) + (jj >> 1)) * Nd * 16, 16u * Nd, &wfull[wsl]);
          ++nw;
        }
        const int st = na % ST;
        if (na >= ST && !wait_or_abort(&aempty[st], ((na / ST) & 1) ^ 1, abort_flag, a.err, kErrMoeWait)) break;
        mbar_arrive_expect_tx(&afull[st], kASlot / 2);
        tma_3d_hint(sA + st * kASlot, &tm_d, 0, row, 2 * jj, &afull[st], pol);
        ++na;
      }
      // copies still in flight land before the CTA may exit
      for (int k = max(0, na - ST); k < na; ++k) mbar_wait(&afull[k % ST], (k / ST) & 1, a.err, kErrMoeWait);
      for (int k = max(0, nw - kNW); k < nw; ++k) mbar_wait(&wfull[k % kNW], (k / kNW) & 1, a.err, kErrMoeWait);
    }
    __syncwarp();  // the lane's role loop ends here: the warp reaches the final barrier converged
  } else if (warp == 10) {
    // ------------------------------------------------------------ h operand producer
    if (lane == 0) {
      int nbi = 0;
      for (int q = q0; q < q1 && !*abort_flag; ++q) {
        const int r = q / S, j = q - r * S, d = j / SI, jj = j - d * SI;
        (void)r;
        const int bs = nbi % NB;
        if (nbi >= NB && !wait_or_abort(&bempty[bs], ((nbi / NB) & 1) ^ 1, abort_flag, a.err, kErrMoeWait)) break;
        int lo, nb;
        span(d, lo, nb);
        const uint32_t sb = sB + bs * Nd * kKS;
        mbar_arrive_expect_tx(&bfull[bs], (uint32_t)nb * kKS);
        for (int c = 0; c < 2; ++c)
          bulk_load(sb + c * nb * 128, a.dimg + (size_t)d * I * Nd + ((size_t)(2 * jj + c) * Nd + 16 * lo) * 128,
                    nb * 128, &bfull[bs]);
        ++nbi;
      }
      for (int k = max(0, nbi - NB); k < nbi; ++k) mbar_wait(&bfull[k % NB], (k / NB) & 1, a.err, kErrMoeWait);
    }
    __syncwarp();  // the lane's role loop ends here: the warp reaches the final barrier converged
  } else if (warp == 1) {
    if (lane == 0) {
      int i = 0, uc = -1, wc = -1, b = 0, wsl = 0;
      for (int q = q0; q < q1 && !*abort_flag; ++q, ++i) {
        const int r = q / S, j = q - r * S, d = j / SI, jj = j - d * SI;
        (void)r;
        if (q == q0 || j == 0) {
          // the epilogue warps zeroed this buffer (at start, or after reading it)
          ++uc;
          b = uc % a.NA;
          if (!wait_or_abort(&acce[b], (uc / a.NA) & 1, abort_flag, a.err, kErrMoeWait)) break;
        }
        if (q == q0 || (jj & 1) == 0) {
          ++wc;
          wsl = wc % kNW;
          if (!wait_or_abort(&sff[wsl], (wc / kNW) & 1, abort_flag, a.err, kErrMoeWait)) break;
        }
        const uint32_t sfw = tbase + kSfCol + kSfWin * wsl;
        const int st = i % ST, bs = i % NB;
        if (!wait_or_abort(&afull[st], (i / ST) & 1, abort_flag, a.err, kErrMoeWait)) break;
        if (!wait_or_abort(&bfull[bs], (i / NB) & 1, abort_flag, a.err, kErrMoeWait)) break;
        tc_fence_after();
        int lo, nb;
        span(d, lo, nb);
        const uint64_t ad0 = sw128_desc(sA + st * kASlot), bd0 = sw128_desc(sB + bs * Nd * kKS);
        const uint32_t bchunk = (uint32_t)nb * 8;
        const uint32_t idn = (uint32_t)(nb >> 3) << 17;
        const uint32_t dcol = tbase + (uint32_t)(b * 128 + 16 * lo);
        const uint32_t g0 = (uint32_t)(jj & 1) * 2;
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2) {
          const uint32_t c = k2 >> 2, kk = k2 & 3;
          mma_mx(dcol, ad0 + c * 1024 + 2 * kk, bd0 + c * bchunk + 2 * kk, kIdBase | idn | (kk << 4) | (kk << 29),
                 sfw + 4 * (g0 + c), sfw + 32 + 8 * (g0 + c), 1u);
        }
        tc_commit(&aempty[st]);
        tc_commit(&bempty[bs]);
        if ((jj & 1) == 1 || q + 1 == q1) tc_commit(&wempty[wsl]);
        if (j == S - 1 || q + 1 == q1) tc_commit(&accf[b]);
      }
      tc_commit(done);
      mbar_wait(done, 0, a.err, kErrMoeWait);
    }
    __syncwarp();  // the lane's role loop ends here: the warp reaches the final barrier converged
  } else if (warp >= 6) {
    // scale warps: as in gate/up, one weight matrix
    const int qd = warp & 3, m = 32 * qd + lane;
    const uint32_t tq = tbase + ((uint32_t)(32 * qd) << 16) + kSfCol;
    const size_t rowb = (size_t)(I / 32);
    const int nwin = q0 < q1 ? (q1 - 1) / 2 - q0 / 2 + 1 : 0;
    auto wstart = [&](int k) { return k == 0 ? q0 : 2 * (q0 / 2 + k); };
    auto load = [&](int k) {
      const int q = wstart(k), r = q / S, j = q - r * S, d = j / SI, jj = j - d * SI;
      const size_t row = (size_t)__ldg(a.elist + d) * H + 128 * r + m;
      return ldg_nc16(a.ds + row * rowb + 16 * (jj >> 1));
    };
    uint4 ca[kSfAhead];
#pragma unroll
    for (int t = 0; t < kSfAhead; ++t)
      if (t < nwin) ca[t] = load(t);
    bool stop = false;
    for (int k0 = 0; k0 < nwin && !stop && !*abort_flag; k0 += kSfAhead) {
#pragma unroll
      for (int t = 0; t < kSfAhead; ++t) {
        const int k = k0 + t;
        if (k >= nwin || stop) break;
        const int wsl = k % kNW;
        if (!wait_or_abort(&wfull[wsl], (k / kNW) & 1, abort_flag, a.err, kErrMoeWait)) {
          stop = true;
          break;
        }
        tc_fence_after();
        const int q = wstart(k);
        const int d = (q - (q / S) * S) / SI;
        int lo, nb;
        span(d, lo, nb);
        uint4 cb[8];
        load_sfb8(sW + wsl * a.WB, 16 * lo, Nd, lane, cb);
        tmem_st_sfa(tq + kSfWin * wsl, ca[t]);
        tmem_st_sfb8(tq + kSfWin * wsl + 32, cb);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sff[wsl]);
        if (k + kSfAhead < nwin) ca[t] = load(k + kSfAhead);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue: y = sum of the token's 3 columns
    const int qd = warp & 3, m = 32 * qd + lane;
    const int et = threadIdx.x - 64;
    const uint32_t tl = tbase + ((uint32_t)(32 * qd) << 16);
    const int n3 = 3 * T;
    // both accumulator buffers start at zero
    for (int bb = 0; bb < a.NA; ++bb)
      for (int c0 = 0; c0 < Nd; c0 += 16) tmem_st_zero16(tl + (uint32_t)(bb * 128 + c0));
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0)
      for (int bb = 0; bb < a.NA; ++bb) mbar_arrive(&acce[bb]);
    int uc = -1;
    const int ufirst = q0 < q1 ? q0 / S : 0, ulast = q0 < q1 ? (q1 - 1) / S : -1;
    for (int u = ufirst; u <= ulast && !*abort_flag; ++u) {
      ++uc;
      const int b = uc % a.NA;
      if (!wait_or_abort(&accf[b], (uc / a.NA) & 1, abort_flag, a.err, kErrMoeWait)) break;
      tc_fence_after();
      int cf, cl;
      unit_ctas(u, S, R.P, cf, cl);
      const bool whole = cf == cl;
      float* dst;
      size_t tstride;
      if (whole) {
        dst = a.y + 128 * u + m;
        tstride = (size_t)H;
      } else {
        dst = a.part + (size_t)(blockIdx.x * 2 + part_slot(blockIdx.x, u, S, R.P)) * T * 128 + m;
        tstride = 128;
      }
      float run = 0.f;
      for (int c0 = 0; c0 < n3; c0 += 16) {
        float v[16];
        tmem_ld16(tl + (uint32_t)(b * 128 + c0), v);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int n = c0 + k;
          if (n < n3) {
            run += v[k];
            if (n % 3 == 2) {
              dst[(size_t)(n / 3) * tstride] = run;
              run = 0.f;
            }
          }
        }
      }
      for (int c0 = 0; c0 < Nd; c0 += 16) tmem_st_zero16(tl + (uint32_t)(b * 128 + c0));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[b]);
      if (!whole) {
        __threadfence();
        epi_bar();
        if (et == 0) *is_last = (atomicAdd(&a.cnt[u], 1u) == (uint32_t)(cl - cf)) ? 1u : 0u;
        epi_bar();
        if (*is_last) {
          __threadfence();
          for (int t = 0; t < T; ++t) {
            float sum = 0.f;
            for (int c = cf; c <= cl; ++c)
              sum += __ldcg(a.part + ((size_t)(c * 2 + part_slot(c, u, S, R.P)) * T + t) * 128 + m);
            a.y[(size_t)t * H + 128 * u + m] = sum;
          }
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
// host side
// ---------------------------------------------------------------------------
namespace {

struct TcPlan {
  int Ng, Nd, stg, nbg, std_, nbd, grid;
  size_t smem_g, smem_d;
};

constexpr size_t kBarBytes = 512;  // barriers, TMEM slot, flags

int round16(int v) { return (v + 15) & ~15; }

TcPlan tc_plan(int T, int sms) {
  TcPlan p{};
  p.Ng = std::max(16, round16(2 * T));
  p.Nd = std::max(16, round16(3 * T));
  p.grid = sms;
  const size_t avail = kTcSmemMax - 1024 - kBarBytes;
  // weight slots fill what the operand slots (NB of the widest span) and the
  // windows leave; the operand slot count is the one that leaves the most
  // weight slots (ties: more operand slots)
  auto plan = [&](int n, int& st, int& nb) {
    const size_t win = ((size_t)16 * n + 1023) & ~(size_t)1023;
    st = 0;
    nb = 0;
    for (int b = 4; b >= 2; --b) {
      const size_t fixed = (size_t)b * n * kKS + kNW * win;
      const int s = (int)std::min<size_t>(8, (avail - fixed) / kASlot);
      if (s > st) {
        st = s;
        nb = b;
      }
    }
    return 1024 + (size_t)st * kASlot + (size_t)nb * n * kKS + kNW * win + kBarBytes;
  };
  p.smem_g = plan(p.Ng, p.stg, p.nbg);
  p.smem_d = plan(p.Nd, p.std_, p.nbd);
  return p;
}

template <typename K>
cudaError_t allow_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

bool moe_mx_tc_ok(int T, int H, int I, int E, int top_k) {
  if (T < 1 || T > 64 || E < 1 || E > 1024 || top_k < 1 || top_k > 32 || top_k > E) return false;
  if (T * top_k > kImgThreads) return false;  // the router's per-pair tables
  if (H < 512 || I < 512 || H % 512 || I % 512) return false;
  if ((long long)E * I >= (1ll << 31) || (long long)E * H >= (1ll << 31)) return false;
  const TcPlan p = tc_plan(T, device_sm_count());
  return p.stg >= 3 && p.std_ >= 3 && p.Ng <= 128 && p.Nd <= 192;
}

MoeTcLayout moe_tc_layout(int T, int H, int I, int E, int top_k, size_t off) {
  MoeTcLayout L{};
  const TcPlan p = tc_plan(T, device_sm_count());
  const size_t P = (size_t)T * top_k, Dmax = std::min<size_t>(E, P);
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = (off + bytes + 255) & ~(size_t)255;
    return o;
  };
  L.elist = take(4 * Dmax);
  L.nexp = take(16);
  L.epair = take(4 * Dmax * T);
  L.gspan = take(4 * Dmax);
  L.dspan = take(4 * Dmax);
  L.ximg = take((size_t)H * p.Ng);
  L.xsf = take((size_t)(H / 512) * p.Ng * 16);
  L.dimg = take(Dmax * I * p.Nd);
  L.dsf = take(Dmax * (I / 512) * p.Nd * 16);
  L.gpart = take((size_t)p.grid * 2 * 2 * T * 128 * 4);
  L.dpart = take((size_t)p.grid * 2 * T * 128 * 4);
  L.gcnt = take(4 * Dmax * (I / 128));
  L.dcnt = take(4 * (size_t)(H / 128));
  L.end = off;
  return L;
}

cudaError_t launch_moe_mx_tc(const uint16_t* x, const float* logits, const uint8_t* gq, const uint8_t* gs,
                             const uint8_t* uq, const uint8_t* us, const uint8_t* dq, const uint8_t* ds, int T,
                             int H, int I, int E, int top_k, float* y, int32_t* idx, float* wts, uint8_t* ws,
                             const MoeTcLayout& L, float* h, uint32_t* err, cudaStream_t stream, bool pdl) {
  const int sms = device_sm_count();
  const TcPlan p = tc_plan(T, sms);
  const size_t P = (size_t)T * top_k, Dmax = std::min<size_t>(E, P);
  auto I32 = [&](size_t o) { return reinterpret_cast<int32_t*>(ws + o); };
  auto U32 = [&](size_t o) { return reinterpret_cast<uint32_t*>(ws + o); };
  const TcRouteArgs ra{logits, x, T, H, E, top_k, p.Ng, idx, wts, I32(L.elist), I32(L.nexp), I32(L.epair),
                       I32(L.gspan), I32(L.dspan), ws + L.ximg, ws + L.xsf, U32(L.gcnt), U32(L.dcnt),
                       (int)(Dmax * (I / 128)), H / 128};
  const int tasks = (p.Ng / 2) * (H / 32);
  const int nimg = std::max(1, std::min(64, (tasks + 127) / 128));
  cudaError_t e;
  if (E <= 128)
    e = launch_kernel(moe_tc_route_kernel<4>, dim3(1 + nimg), dim3(kImgThreads), 0, stream, pdl, ra);
  else if (E <= 512)
    e = launch_kernel(moe_tc_route_kernel<16>, dim3(1 + nimg), dim3(kImgThreads), 0, stream, pdl, ra);
  else
    e = launch_kernel(moe_tc_route_kernel<32>, dim3(1 + nimg), dim3(kImgThreads), 0, stream, pdl, ra);
  if (e != cudaSuccess) return e;
  CUtensorMap tm_g, tm_u, tm_d;
  // E2M1 codes as {128 codes, rows, 128-code chunks}, unpacked to one byte per code in
  // shared memory; one box = 128 rows x 256 codes
  if (!tmap_3d(&tm_g, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, gq, 128, (uint64_t)E * I, H / 128, H / 2, 64, 128,
               128, 2) ||
      !tmap_3d(&tm_u, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, uq, 128, (uint64_t)E * I, H / 128, H / 2, 64, 128,
               128, 2) ||
      !tmap_3d(&tm_d, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, dq, 128, (uint64_t)E * H, I / 128, I / 2, 64, 128,
               128, 2))
    return cudaErrorInvalidValue;
  const TcGuArgs ga{gs, us, ws + L.ximg, ws + L.xsf, I32(L.elist), I32(L.nexp), I32(L.epair), I32(L.gspan), wts, h,
                    ws + L.dimg, ws + L.dsf, reinterpret_cast<float*>(ws + L.gpart), U32(L.gcnt), err,
                    T, H, I, p.Ng, p.Nd, p.stg, p.nbg, p.Ng <= 64 ? 2 : 1,
                    (uint32_t)((16 * p.Ng + 1023) & ~1023)};
  if ((e = allow_smem(moe_tc_gu_kernel, p.smem_g)) != cudaSuccess) return e;
  e = launch_kernel(moe_tc_gu_kernel, dim3(p.grid), dim3(kTcThreads), p.smem_g, stream, pdl, tm_g, tm_u, ga);
  if (e != cudaSuccess) return e;
  const TcDnArgs da{ds, ws + L.dimg, ws + L.dsf, I32(L.elist), I32(L.nexp), I32(L.dspan), y,
                    reinterpret_cast<float*>(ws + L.dpart), U32(L.dcnt), err, T, H, I, p.Nd, p.std_, p.nbd,
                    p.Nd <= 128 ? 2 : 1, (uint32_t)((16 * p.Nd + 1023) & ~1023)};
  if ((e = allow_smem(moe_tc_dn_kernel, p.smem_d)) != cudaSuccess) return e;
  return launch_kernel(moe_tc_dn_kernel, dim3(p.grid), dim3(kTcThreads), p.smem_d, stream, pdl, tm_d, da);
}

}  // namespace qg
