// Device-side building blocks shared by the sm_103a kernels of libqgemv:
// mbarrier / bulk-copy PTX wrappers with bounded waits, the device error word,
// and the bit-level decoders of the stored formats.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "qgemv.h"

namespace qg {

// ---------------------------------------------------------------------------
// Error codes written to the device error word when a bounded wait gives up.
// ---------------------------------------------------------------------------
enum DeviceError : uint32_t {
  kErrNone = 0,
  kErrGemvFullWait = 0x101,
  kErrGemvEmptyWait = 0x102,
  kErrGemvDrain = 0x103,
  kErrTcFullWait = 0x201,
  kErrTcEmptyWait = 0x202,
  kErrTcMmaWait = 0x203,
  kErrTcAccWait = 0x204,
  kErrTcDrain = 0x205,
  kErrMoeWait = 0x301,
  kErrChainFullWait = 0x401,
  kErrChainEmptyWait = 0x402,
  kErrChainDrain = 0x403,
  kErrChainLevelWait = 0x404,
  kErrW8FusedBarrier = 0x405,
  kErrSelftestBarrier = 0x501,
  kErrSelftestFlag = 0x502,
};

// Upper bound on polls of one mbarrier phase before a kernel reports a timeout
// (each poll is a try_wait that may suspend ~0.5-1 us in hardware), about
// a few seconds: far beyond any legitimate wait in these kernels.
constexpr uint32_t kMaxPolls = 1u << 22;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void report_error(uint32_t* err, uint32_t code) {
  if (err) atomicCAS(err, 0u, code);
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete. Returns false
// (after recording `code` in the error word) if it did not complete within
// `polls` polls.
__device__ __forceinline__ bool mbar_wait_n(uint64_t* bar, uint32_t parity, uint32_t* err, uint32_t code,
                                            uint32_t polls) {
  for (uint32_t i = 0; i < polls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  report_error(err, code);
  return false;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* err, uint32_t code) {
  return mbar_wait_n(bar, parity, err, code, kMaxPolls);
}

// ---------------------------------------------------------------------------
// Bulk (non-tensor) async copy global -> shared, completing on an mbarrier.
// Both addresses 16-byte aligned, size a multiple of 16.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Same with an L2 eviction-priority hint (weights streamed once: evict first).
__device__ __forceinline__ void bulk_g2s_evict_first(void* smem_dst, const void* gsrc, uint32_t bytes,
                                                     uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, "
      "[%3], %4;" ::"r"(smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch (no-ops when launched without the attribute).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Shared-memory vector loads
// ---------------------------------------------------------------------------
// TMA tiled load of a 2D box into shared memory, completing on an mbarrier
// (the box's innermost coordinate x must be 16-byte aligned).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tm, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// TMA tiled load of a 3D box (same alignment rule on x)
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tm, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, const uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint16_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.b16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// Load of data another CTA of the same launch may have written: L2, not L1.
__device__ __forceinline__ uint32_t ldcg32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.cg.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ldcg128(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Streaming global load that does not allocate in L1.
__device__ __forceinline__ uint4 ldg_stream128(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// Scalar format decoders
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) {
  float f;
  asm("{.reg .b16 t; mov.b16 t, %1; cvt.f32.f16 %0, t;}" : "=f"(f) : "h"(h));
  return f;
}

// 2^(e-127) for an E8M0 code (e = 255 is rejected upstream).
__device__ __forceinline__ float e8m0_to_f32(uint32_t e) {
  return e ? __uint_as_float(e << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ float fma_f16_lo_lo(uint32_t a, uint32_t b, float acc) {
  asm("{.reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;}"
      : "+f"(acc)
      : "r"(a), "r"(b));
  return acc;
}
__device__ __forceinline__ float fma_f16_hi_hi(uint32_t a, uint32_t b, float acc) {
  asm("{.reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, ah, bh, %0;}"
      : "+f"(acc)
      : "r"(a), "r"(b));
  return acc;
}

// Two E2M1 codes (one byte) -> f16x2 (element 2j low half, 2j+1 high half).
template <int BYTE>
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t word) {
  uint32_t r;
  if (BYTE == 0)
    asm("{.reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %1; cvt.rn.f16x2.e2m1x2 %0, b0;}" : "=r"(r) : "r"(word));
  else if (BYTE == 1)
    asm("{.reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %1; cvt.rn.f16x2.e2m1x2 %0, b1;}" : "=r"(r) : "r"(word));
  else if (BYTE == 2)
    asm("{.reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %1; cvt.rn.f16x2.e2m1x2 %0, b2;}" : "=r"(r) : "r"(word));
  else
    asm("{.reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %1; cvt.rn.f16x2.e2m1x2 %0, b3;}" : "=r"(r) : "r"(word));
  return r;
}

// Two fp32 lanes in one 64-bit register, for the paired fp32 FMA (fma.rn.f32x2).
__device__ __forceinline__ uint64_t pair2(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ void unpair2(uint64_t v, float& lo, float& hi) {
  uint32_t a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(a), "=r"(b) : "l"(v));
  lo = __uint_as_float(a);
  hi = __uint_as_float(b);
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Eight 4-bit codes (code i in bits 4i..4i+3) -> four f16x2 registers with one
// shift and four lop3s: o[0] = (1024 + q0, 1024 + q4), o[1] = (1024 + 16 q1,
// 1024 + 16 q5), o[2] = (1024 + q2, 1024 + q6), o[3] = (1024 + 16 q3,
// 1024 + 16 q7). 0x6400 is fp16 1024 (ulp 1): a code in mantissa bits 0-3 adds
// q, in bits 4-7 adds 16 q; all values are exact.
__device__ __forceinline__ void nib8_to_f16x2_offset(uint32_t w, uint32_t (&o)[4]) {
  constexpr uint32_t kLo = 0x000F000Fu, kHi = 0x00F000F0u, kMagic = 0x64006400u;
  const uint32_t t = w >> 8;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(o[0]) : "r"(w), "r"(kLo), "r"(kMagic));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(o[1]) : "r"(w), "r"(kHi), "r"(kMagic));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(o[2]) : "r"(t), "r"(kLo), "r"(kMagic));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(o[3]) : "r"(t), "r"(kHi), "r"(kMagic));
}

// Pack two bf16 bit patterns (low, high) into one register.
__device__ __forceinline__ uint32_t pack2(uint32_t lo16, uint32_t hi16) { return (lo16 & 0xFFFFu) | (hi16 << 16); }

// Sum R per-lane values over the 32 lanes of a warp with a transposed
// butterfly: at offsets 16, 8, ... each lane keeps half of its remaining values
// and adds its partner's copy of that half, so R values cost about
// R - 1 + log2(32 / R) shuffles instead of 5 R. Afterwards lane L holds the
// total of value transposed_row<R>(L).
template <int R, typename T>
__device__ __forceinline__ T transposed_warp_sum(T (&v)[R], int lane) {
  int cnt = R;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    if (cnt > 1) {
      const int half = cnt / 2;
      const bool upper = lane & o;
#pragma unroll
      for (int i = 0; i < R / 2; ++i) {
        if (i < half) {
          const T keep = upper ? v[i + half] : v[i];
          const T send = upper ? v[i] : v[i + half];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      cnt = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    }
  }
  return v[0];
}

template <int R>
__device__ __forceinline__ int transposed_row(int lane) {
  int row = 0, half = R / 2;
#pragma unroll
  for (int o = 16; o >= 1 && half >= 1; o >>= 1, half >>= 1)
    if (lane & o) row += half;
  return row;
}

// power-of-two exponent sigma such that max|v| * 2^-sigma lies in [2^14, 2^15):
// activations scaled by 2^-sigma fit fp16's range with the largest exponent
// (clamped at -126 so that 2^sigma and 2^-sigma are normal fp32 numbers)
__device__ __forceinline__ int fp16_prescale_exp(float amax) {
  if (!(amax > 0.f)) return 0;
  int e;
  frexpf(amax, &e);  // amax = f * 2^e, f in [0.5, 1)
  return max(e - 15, -126);
}

// 2^e as an fp32 for -126 <= e <= 127 (exact, two integer instructions)
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace qg
