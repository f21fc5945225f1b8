// W8A16 row-int8 GEMV: y[n] = s[n] * sum_k q[n][k] x[k].
//
// "Running Kimi K3 (2.8T) on one Apple Silicon Mac" (Deltafin), section
// "Technical approach / compute" and its table of exact-path improvements: the
// packed int8 output head multiplies the row-int8 checkpoint directly (one
// scale per row, a weight-only quantized matmul) instead of an fp32 head and
// its dequantization. One byte per weight: the kernel is bound by HBM.
//
// GB300 design:
//  * Each CTA first turns x into fp16 scaled by an exact power of two 2^-sigma
//    (sigma from max |x|: the largest value lands in [2^14, 2^15)) and keeps it
//    in shared memory as two arrays, the first and second 8 values of every
//    16-value chunk, so a lane's two 16-byte loads of a chunk are conflict-free.
//  * A warp takes 4 rows at a time (grid-stride over row groups); lane l reads
//    16 weight bytes of each row per step with a streaming 128-bit load (chunks
//    l, l + 32, ...), so one warp instruction moves 512 contiguous bytes.
//  * int8 -> fp16 exactly: u = q xor 0x80 (= q + 128 as an unsigned byte),
//    byte permute with 0x64 gives fp16 1024 + u = 1152 + q, and a paired fp16
//    subtract of 1152 leaves q. Products q * x' are exact in fp32
//    (fma.rn.f32.f16); the row's lane sums are added with a transposed
//    butterfly and y = s * 2^sigma * sum.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

namespace {

constexpr int kW8gThreads = 512;
constexpr int kW8gWarps = kW8gThreads / 32;
constexpr int kW8gRows = 4;  // rows per warp step

// two int8 codes (bytes b, b + 1 of w) -> fp16x2 (q_b, q_b+1), exact
template <int PAIR>
__device__ __forceinline__ uint32_t i8x2_to_f16x2(uint32_t w_xor) {
  // fp16 bits 0x6400 | u = 1024 + u; u = q + 128
  const uint32_t biased = __byte_perm(w_xor, 0x64646464u, PAIR == 0 ? 0x4140u : 0x4342u);
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(biased), "r"(0x64806480u));  // - (1152, 1152)
  return r;
}

__device__ __forceinline__ float fma_lo(uint32_t a, uint32_t b, float acc) {
  asm("{.reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;}"
      : "+f"(acc)
      : "r"(a), "r"(b));
  return acc;
}
__device__ __forceinline__ float fma_hi(uint32_t a, uint32_t b, float acc) {
  asm("{.reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, ah, bh, %0;}"
      : "+f"(acc)
      : "r"(a), "r"(b));
  return acc;
}

// acc += sum of the 8 products of one weight half-chunk (8 codes) with x
__device__ __forceinline__ float dot8(uint32_t w0, uint32_t w1, const uint4 xv, float acc) {
  const uint32_t u0 = w0 ^ 0x80808080u, u1 = w1 ^ 0x80808080u;
  const uint32_t q0 = i8x2_to_f16x2<0>(u0), q1 = i8x2_to_f16x2<1>(u0);
  const uint32_t q2 = i8x2_to_f16x2<0>(u1), q3 = i8x2_to_f16x2<1>(u1);
  acc = fma_lo(q0, xv.x, acc);
  acc = fma_hi(q0, xv.x, acc);
  acc = fma_lo(q1, xv.y, acc);
  acc = fma_hi(q1, xv.y, acc);
  acc = fma_lo(q2, xv.z, acc);
  acc = fma_hi(q2, xv.z, acc);
  acc = fma_lo(q3, xv.w, acc);
  acc = fma_hi(q3, xv.w, acc);
  return acc;
}

}  // namespace

__global__ void __launch_bounds__(kW8gThreads, 2)
    w8a16_gemv_kernel(const int8_t* __restrict__ wq, const float* __restrict__ scales,
                      const uint16_t* __restrict__ x, float* __restrict__ y, int N, int K) {
  extern __shared__ uint4 xs[];  // [K / 16] first halves, then [K / 16] second halves of the chunks
  __shared__ float wmax[kW8gWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunks = K / 16;
  pdl_wait();  // x may come from the previous kernel
  // max |x| over the vector
  const uint4* x4 = reinterpret_cast<const uint4*>(x);
  float m = 0.f;
  for (int i = threadIdx.x; i < K / 8; i += kW8gThreads) {
    const uint4 v = __ldg(x4 + i);
    const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      m = fmaxf(m, fmaxf(fabsf(bf16_bits_to_f32(vv[j] & 0xFFFFu)), fabsf(bf16_bits_to_f32(vv[j] >> 16))));
  }
  m = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m)));  // non-negative: uint order
  if (lane == 0) wmax[warp] = m;
  __syncthreads();
  m = 0.f;
#pragma unroll
  for (int w = 0; w < kW8gWarps; ++w) m = fmaxf(m, wmax[w]);
  const int sig = fp16_prescale_exp(m);
  const float sc = pow2f(-sig);
  // x * 2^-sigma in fp16 (exact scaling), chunk halves in two arrays
  for (int i = threadIdx.x; i < K / 8; i += kW8gThreads) {
    const uint4 v = __ldg(x4 + i);
    uint4 o;
    o.x = pack2(__half_as_ushort(__float2half_rn(bf16_bits_to_f32(v.x & 0xFFFFu) * sc)),
                __half_as_ushort(__float2half_rn(bf16_bits_to_f32(v.x >> 16) * sc)));
    o.y = pack2(__half_as_ushort(__float2half_rn(bf16_bits_to_f32(v.y & 0xFFFFu) * sc)),
                __half_as_ushort(__float2half_rn(bf16_bits_to_f32(v.y >> 16) * sc)));
    o.z = pack2(__half_as_ushort(__float2half_rn(bf16_bits_to_f32(v.z & 0xFFFFu) * sc)),
                __half_as_ushort(__float2half_rn(bf16_bits_to_f32(v.z >> 16) * sc)));
    o.w = pack2(__half_as_ushort(__float2half_rn(bf16_bits_to_f32(v.w & 0xFFFFu) * sc)),
                __half_as_ushort(__float2half_rn(bf16_bits_to_f32(v.w >> 16) * sc)));
    xs[(i & 1) * chunks + (i >> 1)] = o;
  }
  __syncthreads();
  pdl_launch_dependents();
  const float up = pow2f(sig);
  const int nwarps = gridDim.x * kW8gWarps;
  for (int r0 = (blockIdx.x * kW8gWarps + warp) * kW8gRows; r0 < N; r0 += nwarps * kW8gRows) {
    float acc[kW8gRows];
#pragma unroll
    for (int r = 0; r < kW8gRows; ++r) acc[r] = 0.f;
    const int8_t* base = wq + (size_t)r0 * K;
#pragma unroll 2
    for (int c = lane; c < chunks; c += 32) {
      const uint4 xa = xs[c], xb = xs[chunks + c];
      uint4 w[kW8gRows];
#pragma unroll
      for (int r = 0; r < kW8gRows; ++r)
        w[r] = r0 + r < N ? ldg_stream128(base + (size_t)r * K + 16 * c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int r = 0; r < kW8gRows; ++r) {
        acc[r] = dot8(w[r].x, w[r].y, xa, acc[r]);
        acc[r] = dot8(w[r].z, w[r].w, xb, acc[r]);
      }
    }
    const float tot = transposed_warp_sum<kW8gRows>(acc, lane);
    const int row = r0 + transposed_row<kW8gRows>(lane);
    if (lane < kW8gRows * 8 && (lane & 7) == 0 && row < N) y[row] = __ldg(scales + row) * up * tot;
  }
}

cudaError_t launch_w8a16_gemv(const int8_t* wq, const float* scales, const uint16_t* x, float* y, int N, int K,
                              cudaStream_t stream, bool pdl) {
  if (N < 1 || K < 16 || K % 16) return cudaErrorInvalidValue;
  const size_t smem = (size_t)K * 2;
  cudaError_t e = allow_max_smem(w8a16_gemv_kernel);
  if (e != cudaSuccess) return e;
  const int groups = (N + kW8gRows - 1) / kW8gRows;
  const int grid = std::min(2 * device_sm_count(), (groups + kW8gWarps - 1) / kW8gWarps);
  return launch_kernel(w8a16_gemv_kernel, dim3(grid), dim3(kW8gThreads), smem, stream, pdl, wq, scales, x, y, N, K);
}

}  // namespace qg
