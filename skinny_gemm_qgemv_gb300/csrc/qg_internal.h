// Host-side internals of libqgemv: kernel launchers shared between the
// translation units and the C entry points in api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace qg {

// Launch with cudaLaunchKernelEx; with pdl the launch carries the
// programmatic-stream-serialization attribute so the kernel may begin while the
// previous kernel on the stream drains (kernels call griddepcontrol.wait before
// touching activations or outputs).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

int device_sm_count();

// Device address of the library's sticky error word on the current device
// (looked up once per device), or null if it cannot be found.
uint32_t* err_word();

// Largest dynamic shared memory one CTA may opt into on the current device.
int device_max_smem_optin();

// Raise a kernel's dynamic shared-memory limit to the device maximum. The
// value is the same for every call, so launches captured into a CUDA graph
// (or replayed one by one by a profiler) never see a limit set for another
// shape.
template <typename... KArgs>
cudaError_t allow_max_smem(void (*kernel)(KArgs...)) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              device_max_smem_optin() - static_cast<int>(fa.sharedSizeBytes));
}

// W4A16 (w4a16_gemv.cu, w4a16_tc.cu)
struct GemvConfig {
  int kpl;            // consecutive k per lane (32 or 64)
  int rpw;            // rows per consumer warp per tile (2, 4, 8)
  int rg;             // row groups per CTA
  int ctas_per_sm;    // grid = min(tiles, ctas_per_sm * SMs)
  size_t smem_budget; // shared memory for the stage ring
};
bool gemv_fast_path_ok(int M, int N, int K);
GemvConfig gemv_pick_config(int M, int N, int K, int sms);
cudaError_t launch_w4a16_fast_cfg(const uint32_t* wq, const uint16_t* sc, const uint16_t* bi, const uint16_t* x,
                                  float* y, int M, int N, int K, const GemvConfig& cfg, uint32_t* err,
                                  cudaStream_t stream, bool pdl);
cudaError_t launch_w4a16_fast(const uint32_t* wq, const uint16_t* sc, const uint16_t* bi, const uint16_t* x,
                              float* y, int M, int N, int K, uint32_t* err, cudaStream_t stream, bool pdl);
bool tc_path_ok(int M, int N, int K);
size_t tc_workspace_size(int M, int N, int K);
cudaError_t launch_w4a16_tc(const uint32_t* wq, const uint16_t* sc, const uint16_t* bi, const uint16_t* x,
                            float* y, int M, int N, int K, void* ws, size_t ws_bytes, uint32_t* err,
                            cudaStream_t stream, bool pdl);
// Grouped skinny GEMM on tcgen05 (w4a16_tc.cu): one persistent launch over a
// list of independent projections Y_i = X_i W_i^T, all with 3 <= M <= 32 in one
// width class (M <= 16, or 17..32); full-K row tiles, no workspace.
struct TcGroupItem {
  const uint32_t* wq;
  const uint16_t* scales;
  const uint16_t* biases;
  const uint16_t* x;
  float* y;
  int M, N, K;
};
struct TcGroupPlan {
  void* d_gemvs;    // device descriptors (tensor maps + shapes)
  int* d_cta;       // [grid + 1] first unit of each CTA, then [grid] its projection
  void* d_scratch;  // M <= 16: every projection's B fragments and group table
  int ngemv, grid, NT, ST, mma, mma_nt, max_groups;
  uint32_t stage_bytes;
  size_t smem;
};
// 0: fine; 1: a shape outside the tcgen05 path; 2: mixed width classes
int tc_group_check(const TcGroupItem* list, int n);
cudaError_t tc_group_plan_build(const TcGroupItem* list, int n, int sms, TcGroupPlan* out);
void tc_group_plan_free(TcGroupPlan* p);
cudaError_t tc_group_launch(const TcGroupPlan& p, uint32_t* err, cudaStream_t stream, bool pdl);
// any M <= 32, group 32, 64 or 128 (one warp per row)
cudaError_t launch_w4a16_generic(const uint32_t* wq, const uint16_t* sc, const uint16_t* bi, const uint16_t* x,
                                 float* y, int M, int N, int K, int group, cudaStream_t stream, bool pdl);

// Hadamard + int8 (hadamard_i8.cu)
cudaError_t launch_hadamard32_quant_i8(const uint16_t* x, const uint32_t* sign_bits, int8_t* q, float* scale,
                                       int M, int K, cudaStream_t stream, bool pdl);

// W8A8 (w8a8_i32.cu)
cudaError_t launch_w8a8_i32(const int8_t* a, const int8_t* w, int32_t* c, int M, int N, int K, uint32_t* err,
                            cudaStream_t stream, bool pdl);
// W8A8 through exact fp16 operands on the tensor cores (w8a8_mma.cu): M <= 16,
// K a multiple of 512, N >= 128; clears C itself (split K adds into it)
bool w8a8_mma_ok(int M, int N, int K);
cudaError_t launch_w8a8_mma(const int8_t* a, const int8_t* w, int32_t* c, int M, int N, int K, uint32_t* err,
                            cudaStream_t stream, bool pdl);
// Hadamard + int8 + W8A8 + dequant in one cooperative launch (w8a8_mma.cu):
// M <= 16, K a multiple of 1024 and at most 4096
bool w8a8_fused_ok(int M, int N, int K);
size_t w8a8_fused_workspace_size(int M, int K);
cudaError_t launch_w8a8_fused(const uint16_t* x, const uint32_t* sign_bits, const int8_t* w, const float* sw,
                              float* y, int M, int N, int K, void* ws, uint32_t* err, cudaStream_t stream);

// Grouped M = 1 W4A16 GEMV (w4a16_group.cu): one persistent launch over a list
// of independent projections. The caller fills wq, scales, biases, x, y, N, K;
// group_plan_build fills the tiling fields and uploads the list.
struct GroupGemv {
  const uint32_t* wq;
  const uint16_t* scales;
  const uint16_t* biases;
  const uint16_t* x;
  float* y;
  int N, K;
  int S, RG, R;          // K-slices, row groups, rows per tile
  int tile0, tile_end;   // the projection's tiles in the group's tile list
  int pad;
};
struct GroupPlan {
  GroupGemv* d_gemvs;
  int* d_cta;  // [grid + 1] first tile of each CTA
  int ngemv, grid, ST;
  uint32_t stage_bytes;
  size_t smem;
};
bool group_gemv_ok(int N, int K);
cudaError_t group_plan_build(const GroupGemv* list, int n, int sms, GroupPlan* out);
void group_plan_free(GroupPlan* p);
cudaError_t group_launch(const GroupPlan& p, uint32_t* err, cudaStream_t stream, bool pdl);

// W4A16 GEMV chain (w4a16_chain.cu): the M = 1 projections of a decode step
// with dependency levels, one persistent launch; the weights are copied into
// a fragment-major layout at plan build.
constexpr int kChainXBf16 = 0;    // x given as bf16 [K]
constexpr int kChainXCopy = 1;    // x = bf16(alpha * src[k]), src fp32 [K]
constexpr int kChainXSwiglu = 2;  // x = bf16(silu(src[k]) * src[K + k] * alpha), src fp32 [2K]
constexpr int kChainMaxK = 16384;
struct ChainItem {
  const uint32_t* wq;
  const uint16_t* scales;
  const uint16_t* biases;
  int N, K, level, op;
  const void* xsrc;
  float alpha;
  float* y;
};
struct ChainProj {        // device copy of one projection
  const uint8_t* packed;  // fragment-major weights
  const void* xsrc;
  float* y;
  float alpha;
  int op, N, K, level;
};
struct ChainSeg {         // a run of row blocks of one projection for one CTA
  int proj, b0, b1, level;
};
struct ChainPlan {
  uint8_t* d_packed;
  ChainProj* d_proj;
  ChainSeg* d_seg;
  int* d_cta;       // [grid + 1] first segment of each CTA
  int* d_ltiles;    // [nlevels] row blocks per level
  unsigned* d_cnt;  // [nlevels + 1] level counters, CTAs finished
  unsigned long long* d_trace;  // null, or [grid][nlevels][4] timestamps
  int nproj, nlevels, grid, ST;
  uint32_t bfr_bytes;
  size_t smem, packed_bytes;
};
bool chain_proj_ok(int N, int K);
size_t chain_packed_bytes(int N, int K);
// items sorted by level (non-decreasing); the repack runs on the legacy
// stream and is complete when this returns
cudaError_t chain_plan_build(const ChainItem* items, int n, int sms, ChainPlan* out);
void chain_plan_free(ChainPlan* p);
cudaError_t chain_launch(const ChainPlan& p, uint32_t* err, cudaStream_t stream);
// allocate (zeroed) or free the per-(CTA, level) timestamp buffer
cudaError_t chain_set_trace(ChainPlan* p, bool enable);

// Failure-reporting self-test (selftest.cu): kind 0 waits on an mbarrier no
// one arrives at for `limit` polls, kind 1 on `flag` (which must stay 0) for
// `limit` microseconds; both record their code in err and return.
cudaError_t launch_selftest_wait(int kind, uint32_t limit, const unsigned* flag, uint32_t* err,
                                 cudaStream_t stream);

// TMA tensor maps (tmap.cu): 2D {inner, outer} with a row stride, 3D
// {inner, rows, chunks} with row and chunk strides; false if encoding fails.
bool tmap_2d(CUtensorMap* tm, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t outer,
             uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);
bool tmap_3d(CUtensorMap* tm, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t rows,
             uint64_t chunks, uint64_t row_bytes, uint64_t chunk_bytes, uint32_t box_inner, uint32_t box_rows,
             uint32_t box_chunks);

// affine codes at 2, 3, 4, 5, 6 or 8 bits, groups 32/64/128 (affine_gemv.cu):
// 1 <= M <= 4 on 32-code chunks (affine_fast_ok says which shapes), and the
// one-code-per-lane kernel for any M <= 32
bool affine_fast_ok(int bits, int M, int K, int group);
cudaError_t launch_affine_fast(const uint32_t* wq, int bits, const uint16_t* sc, const uint16_t* bi,
                               const uint16_t* x, float* y, int M, int N, int K, int group, cudaStream_t stream,
                               bool pdl);
cudaError_t launch_affine_generic(const uint32_t* wq, int bits, const uint16_t* sc, const uint16_t* bi,
                                  const uint16_t* x, float* y, int M, int N, int K, int group, cudaStream_t stream,
                                  bool pdl);

// W8A16 row-int8 GEMV (w8a16_gemv.cu)
cudaError_t launch_w8a16_gemv(const int8_t* wq, const float* scales, const uint16_t* x, float* y, int N, int K,
                              cudaStream_t stream, bool pdl);

// MXFP4 MoE (moe_mxfp4.cu, moe_mx_mma.cu)
constexpr int kMxTC = 8;                // pairs of one virtual expert: the N = 8 columns of one MMA
// upper bound of the virtual experts of a batch: every active expert once, plus
// one more for every further kMxTC pairs
inline int moe_nvirt_max(int T, int E, int top_k) {
  const int P = T * top_k;
  return (P < E ? P : E) + P / kMxTC;
}
// scratch of the tcgen05 block-scaled path (moe_mx_tc.cu), byte offsets in the workspace
struct MoeTcLayout {
  size_t elist, nexp, epair, gspan, dspan, ximg, xsf, dimg, dsf, gpart, dpart, gcnt, dcnt, end;
};
struct MoeLayout {
  size_t pair_expert, pair_weight, counts, offsets, active, order, nactive, xh, xexp, h, hh, hexp, partial;
  size_t hmax;
  bool has_tc;     // the tcgen05 path's scratch follows
  MoeTcLayout tc;
  size_t total;
};
MoeLayout moe_layout(int T, int H, int I, int E, int top_k);
bool moe_mx_mma_ok(int T, int H, int I, int E, int top_k);
bool moe_mx_tc_ok(int T, int H, int I, int E, int top_k);
MoeTcLayout moe_tc_layout(int T, int H, int I, int E, int top_k, size_t off);
cudaError_t launch_moe_mx_tc(const uint16_t* x, const float* logits, const uint8_t* gq, const uint8_t* gs,
                             const uint8_t* uq, const uint8_t* us, const uint8_t* dq, const uint8_t* ds, int T,
                             int H, int I, int E, int top_k, float* y, int32_t* idx, float* wts, uint8_t* ws,
                             const MoeTcLayout& L, float* h, uint32_t* err, cudaStream_t stream, bool pdl);
cudaError_t launch_moe_mx_mma(const uint16_t* x, const float* logits, const uint8_t* gq, const uint8_t* gs,
                              const uint8_t* uq, const uint8_t* us, const uint8_t* dq, const uint8_t* ds, int T,
                              int H, int I, int E, int top_k, float* y, int32_t* idx, float* wts, int32_t* xexp,
                              uint16_t* xh, uint32_t* hmax, float* h, uint16_t* hh, uint32_t* err,
                              cudaStream_t stream, bool pdl);
cudaError_t launch_moe_mxfp4(const uint16_t* x, const float* logits, const uint8_t* gq, const uint8_t* gs,
                             const uint8_t* uq, const uint8_t* us, const uint8_t* dq, const uint8_t* ds, int T,
                             int H, int I, int E, int top_k, float* y, int32_t* idx, float* wts, void* ws,
                             uint32_t* err, cudaStream_t stream, bool pdl);

}  // namespace qg
