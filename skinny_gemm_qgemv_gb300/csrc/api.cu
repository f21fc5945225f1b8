// C entry points of libqgemv (declared in include/qgemv.h): argument
// validation, variant selection and launch on the caller's stream.
//
// Validation happens entirely on the host before any launch, following the
// rule of "MLX Runner: An Inference Engine You Can Read", section "Untrusted
// input, verified output": malformed requests are rejected with a clear error
// and nothing reaches the GPU.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <new>
#include <vector>

#include "qg_common.cuh"
#include "qg_internal.h"
#include "qgemv.h"

namespace {

// Sticky device error word (one per device context, static device memory).
__device__ uint32_t g_qg_device_error;

constexpr int kMaxDevices = 64;
uint32_t* g_err_ptr[kMaxDevices] = {};
std::mutex g_err_mu;

}  // namespace

namespace qg {
// Device address of the error word for the current device (looked up once).
uint32_t* err_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_qg_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<uint32_t*>(p);
  }
  return g_err_ptr[dev];
}
}  // namespace qg

namespace {
using qg::err_word;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

thread_local cudaError_t t_last_cuda = cudaSuccess;  // behind the last QG_ERR_CUDA of this thread

qg_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return QG_OK;
  t_last_cuda = e;
  return QG_ERR_CUDA;
}

bool g_pdl = false;  // programmatic dependent launch for every kernel (see qg_set_pdl)

}  // namespace

namespace qg {
int device_max_smem_optin() {
  int dev = 0, v = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  return v;
}

int device_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess)
    sms = 0;
  return sms > 0 ? sms : 1;  // planners divide by it; without a device, size queries still answer
}
}  // namespace qg

extern "C" {

const char* qg_status_string(qg_status s) {
  switch (s) {
    case QG_OK: return "QG_OK";
    case QG_ERR_INVALID_ARG: return "QG_ERR_INVALID_ARG: null pointer, bad size or shape";
    case QG_ERR_MISALIGNED: return "QG_ERR_MISALIGNED: a pointer is not 16-byte aligned";
    case QG_ERR_UNSUPPORTED: return "QG_ERR_UNSUPPORTED: valid request this build does not handle";
    case QG_ERR_WORKSPACE: return "QG_ERR_WORKSPACE: workspace missing or too small";
    case QG_ERR_CUDA: return "QG_ERR_CUDA: a CUDA runtime call or kernel launch failed";
    case QG_ERR_DEVICE_TIMEOUT: return "QG_ERR_DEVICE_TIMEOUT: a kernel's bounded wait gave up";
  }
  return "QG_ERR_UNKNOWN";
}

int qg_version(void) { return 100; }

// Process-wide switch: launch kernels with programmatic dependent launch so a
// kernel's weight streaming may overlap the tail of the previous kernel on the
// stream. Activations and outputs are only touched after the dependency wait,
// but WEIGHTS may be read early: enable only when no kernel immediately before
// a call writes that call's weights. Off by default.
size_t qg_w8a8_hadamard_workspace_size(int M, int K) {
  if (M < 1 || M > 16 || K < 1) return 0;
  return qg::w8a8_fused_workspace_size(M, K);
}

qg_status gemm_w8a8_hadamard(const uint16_t* x_bf16, const uint32_t* sign_bits, const int8_t* w, const float* sw,
                             float* y, int M, int N, int K, void* workspace, size_t ws_bytes, void* stream) {
  if (!x_bf16 || !sign_bits || !w || !sw || !y || !workspace) return QG_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 32 || K % 32 != 0) return QG_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || !aligned16(sign_bits) || !aligned16(w) || !aligned16(sw) || !aligned16(y) ||
      !aligned16(workspace))
    return QG_ERR_MISALIGNED;
  if (!qg::w8a8_fused_ok(M, N, K)) return QG_ERR_UNSUPPORTED;
  if (ws_bytes < qg::w8a8_fused_workspace_size(M, K)) return QG_ERR_WORKSPACE;
  uint32_t* err = err_word();
  if (!err) return QG_ERR_CUDA;
  return from_cuda(qg::launch_w8a8_fused(x_bf16, sign_bits, w, sw, y, M, N, K, workspace, err,
                                         static_cast<cudaStream_t>(stream)));
}

void qg_set_pdl(int enable) { g_pdl = enable != 0; }

size_t qg_gemv_workspace_size(int N, int K, int group_size) {
  (void)N;
  (void)K;
  (void)group_size;
  return 0;
}

size_t qg_skinny_workspace_size(int M, int N, int K, int group_size) {
  if (group_size != 64 || M < 1 || M > 32 || N < 1 || K < 1) return 0;
  return qg::gemv_fast_path_ok(M, N, K) ? 0 : qg::tc_workspace_size(M, N, K);
}

static qg_status check_w4(const uint32_t* wq, const uint16_t* s, const uint16_t* b, const uint16_t* x,
                          const float* y, int M, int N, int K, int group) {
  if (!wq || !s || !b || !x || !y) return QG_ERR_INVALID_ARG;
  if (M < 1 || M > 32 || N < 1 || K < 1) return QG_ERR_INVALID_ARG;
  if (group != 32 && group != 64 && group != 128) return QG_ERR_INVALID_ARG;
  if (K % group != 0) return QG_ERR_INVALID_ARG;
  if ((long long)N * (K / 8) >= (1LL << 40)) return QG_ERR_INVALID_ARG;
  if (!aligned16(wq) || !aligned16(s) || !aligned16(b) || !aligned16(x) || !aligned16(y)) return QG_ERR_MISALIGNED;
  return QG_OK;
}

static qg_status run_w4(const uint32_t* wq, const uint16_t* s, const uint16_t* b, const uint16_t* x, float* y,
                        int M, int N, int K, int group, void* ws, size_t ws_bytes, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (group != 64) {
    // groups of 32 or 128 (the W4A16 fast paths fold per 64-code group): the
    // chunked affine kernel up to 4 rows, else the generic kernel
    e = qg::affine_fast_ok(4, M, K, group) ? qg::launch_affine_fast(wq, 4, s, b, x, y, M, N, K, group, st, g_pdl)
                                           : qg::launch_w4a16_generic(wq, s, b, x, y, M, N, K, group, st, g_pdl);
  } else if (qg::gemv_fast_path_ok(M, N, K)) {
    uint32_t* err = err_word();
    if (!err) return QG_ERR_CUDA;
    e = qg::launch_w4a16_fast(wq, s, b, x, y, M, N, K, err, st, g_pdl);
  } else if (qg::tc_path_ok(M, N, K)) {
    uint32_t* err = err_word();
    if (!err) return QG_ERR_CUDA;
    e = qg::launch_w4a16_tc(wq, s, b, x, y, M, N, K, ws, ws_bytes, err, st, g_pdl);
  } else if (qg::affine_fast_ok(4, M, K, 64)) {
    e = qg::launch_affine_fast(wq, 4, s, b, x, y, M, N, K, 64, st, g_pdl);
  } else {
    e = qg::launch_w4a16_generic(wq, s, b, x, y, M, N, K, 64, st, g_pdl);
  }
  return from_cuda(e);
}

qg_status qgemv_w4a16(const uint32_t* wq, const uint16_t* scales_f16, const uint16_t* biases_f16,
                      const uint16_t* x_bf16, float* y, int N, int K, int group_size, void* workspace,
                      size_t ws_bytes, void* stream) {
  qg_status st = check_w4(wq, scales_f16, biases_f16, x_bf16, y, 1, N, K, group_size);
  if (st != QG_OK) return st;
  if (ws_bytes < qg_gemv_workspace_size(N, K, group_size)) return QG_ERR_WORKSPACE;
  if (ws_bytes && !workspace) return QG_ERR_INVALID_ARG;
  return run_w4(wq, scales_f16, biases_f16, x_bf16, y, 1, N, K, group_size, workspace, ws_bytes, stream);
}

qg_status qgemm_affine(const uint32_t* wq, int bits, const uint16_t* scales_f16, const uint16_t* biases_f16,
                       const uint16_t* x_bf16, float* y, int M, int N, int K, int group_size, void* stream) {
  if (!wq || !scales_f16 || !biases_f16 || !x_bf16 || !y) return QG_ERR_INVALID_ARG;
  if (bits != 2 && bits != 3 && bits != 4 && bits != 5 && bits != 6 && bits != 8) return QG_ERR_INVALID_ARG;
  if (group_size != 32 && group_size != 64 && group_size != 128) return QG_ERR_INVALID_ARG;
  if (M < 1 || M > 32 || N < 1 || K < 32 || K % 32 || K % group_size || K > (1 << 20)) return QG_ERR_INVALID_ARG;
  if ((long long)N * (K / 32) * bits >= (1LL << 40)) return QG_ERR_INVALID_ARG;
  if (!aligned16(wq) || !aligned16(scales_f16) || !aligned16(biases_f16) || !aligned16(x_bf16) || !aligned16(y))
    return QG_ERR_MISALIGNED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (qg::affine_fast_ok(bits, M, K, group_size))
    return from_cuda(qg::launch_affine_fast(wq, bits, scales_f16, biases_f16, x_bf16, y, M, N, K, group_size, st,
                                            g_pdl));
  return from_cuda(qg::launch_affine_generic(wq, bits, scales_f16, biases_f16, x_bf16, y, M, N, K, group_size, st,
                                             g_pdl));
}

qg_status qgemv_w8a16(const int8_t* wq, const float* scales, const uint16_t* x_bf16, float* y, int N, int K,
                      void* stream) {
  if (!wq || !scales || !x_bf16 || !y) return QG_ERR_INVALID_ARG;
  if (N < 1 || K < 16 || K % 16 || K > 65536) return QG_ERR_INVALID_ARG;
  if (!aligned16(wq) || !aligned16(x_bf16)) return QG_ERR_MISALIGNED;
  return from_cuda(qg::launch_w8a16_gemv(wq, scales, x_bf16, y, N, K, static_cast<cudaStream_t>(stream), g_pdl));
}

struct qg_w4_group {
  qg::GroupPlan plan;
};

qg_status qgemv_w4a16_group_create(const qg_w4_gemv_desc* descs, int count, int group_size, qg_w4_group** group) {
  if (!descs || !group || count < 1) return QG_ERR_INVALID_ARG;
  std::vector<qg::GroupGemv> list(count);
  if (group_size == 32 || group_size == 128) return QG_ERR_UNSUPPORTED;  // grouped launches: g64 only
  for (int i = 0; i < count; ++i) {
    const qg_w4_gemv_desc& d = descs[i];
    qg_status st = check_w4(d.wq, d.scales_f16, d.biases_f16, d.x_bf16, d.y, 1, d.N, d.K, group_size);
    if (st != QG_OK) return st;
    if (!qg::group_gemv_ok(d.N, d.K)) return QG_ERR_UNSUPPORTED;
    qg::GroupGemv g{};
    g.wq = d.wq;
    g.scales = d.scales_f16;
    g.biases = d.biases_f16;
    g.x = d.x_bf16;
    g.y = d.y;
    g.N = d.N;
    g.K = d.K;
    list[i] = g;
  }
  auto* out = new (std::nothrow) qg_w4_group();
  if (!out) return QG_ERR_CUDA;
  if (qg::group_plan_build(list.data(), count, qg::device_sm_count(), &out->plan) != cudaSuccess) {
    delete out;
    return QG_ERR_CUDA;
  }
  *group = out;
  return QG_OK;
}

qg_status qgemv_w4a16_group_run(const qg_w4_group* group, void* stream) {
  if (!group) return QG_ERR_INVALID_ARG;
  uint32_t* err = err_word();
  if (!err) return QG_ERR_CUDA;
  return from_cuda(qg::group_launch(group->plan, err, static_cast<cudaStream_t>(stream), g_pdl));
}

void qgemv_w4a16_group_destroy(qg_w4_group* group) {
  if (!group) return;
  qg::group_plan_free(&group->plan);
  delete group;
}

struct qg_w4_chain {
  qg::ChainPlan plan;
};

qg_status qgemv_w4a16_chain_create(const qg_w4_chain_desc* descs, int count, int group_size, qg_w4_chain** chain) {
  if (!descs || !chain || count < 1) return QG_ERR_INVALID_ARG;
  if (group_size == 32 || group_size == 128) return QG_ERR_UNSUPPORTED;
  if (group_size != 64) return QG_ERR_INVALID_ARG;
  std::vector<qg::ChainItem> list(count);
  for (int i = 0; i < count; ++i) {
    const qg_w4_chain_desc& d = descs[i];
    if (!d.wq || !d.scales_f16 || !d.biases_f16 || !d.x_src || !d.y) return QG_ERR_INVALID_ARG;
    if (d.N < 1 || d.K < 64 || d.K % 64 != 0 || d.level < 0) return QG_ERR_INVALID_ARG;
    if (i > 0 && d.level < descs[i - 1].level) return QG_ERR_INVALID_ARG;
    if (d.x_op != QG_X_BF16 && d.x_op != QG_X_COPY && d.x_op != QG_X_SWIGLU) return QG_ERR_INVALID_ARG;
    if (!aligned16(d.wq) || !aligned16(d.scales_f16) || !aligned16(d.biases_f16) || !aligned16(d.x_src) ||
        !aligned16(d.y))
      return QG_ERR_MISALIGNED;
    if (!qg::chain_proj_ok(d.N, d.K)) return QG_ERR_UNSUPPORTED;
    list[i] = qg::ChainItem{d.wq, d.scales_f16, d.biases_f16, d.N, d.K, d.level, d.x_op, d.x_src, d.x_alpha, d.y};
  }
  auto* out = new (std::nothrow) qg_w4_chain();
  if (!out) return QG_ERR_CUDA;
  const cudaError_t e = qg::chain_plan_build(list.data(), count, qg::device_sm_count(), &out->plan);
  if (e != cudaSuccess) {
    delete out;
    return from_cuda(e);
  }
  *chain = out;
  return QG_OK;
}

qg_status qgemv_w4a16_chain_run(const qg_w4_chain* chain, void* stream) {
  if (!chain) return QG_ERR_INVALID_ARG;
  uint32_t* err = err_word();
  if (!err) return QG_ERR_CUDA;
  return from_cuda(qg::chain_launch(chain->plan, err, static_cast<cudaStream_t>(stream)));
}

void qgemv_w4a16_chain_destroy(qg_w4_chain* chain) {
  if (!chain) return;
  qg::chain_plan_free(&chain->plan);
  delete chain;
}

qg_status qgemv_w4a16_chain_trace_enable(qg_w4_chain* chain, int enable) {
  if (!chain) return QG_ERR_INVALID_ARG;
  return from_cuda(qg::chain_set_trace(&chain->plan, enable != 0));
}

qg_status qgemv_w4a16_chain_trace_read(const qg_w4_chain* chain, uint64_t* host, size_t count) {
  if (!chain || !host || !chain->plan.d_trace) return QG_ERR_INVALID_ARG;
  const size_t n = (size_t)chain->plan.grid * chain->plan.nlevels * 4;
  if (count > n) count = n;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(host, chain->plan.d_trace, count * sizeof(uint64_t), cudaMemcpyDeviceToHost);
  return from_cuda(e);
}

void qgemv_w4a16_chain_trace_shape(const qg_w4_chain* chain, int* grid, int* levels) {
  if (grid) *grid = chain ? chain->plan.grid : 0;
  if (levels) *levels = chain ? chain->plan.nlevels : 0;
}

size_t qgemv_w4a16_chain_bytes(const qg_w4_chain* chain) {
  if (!chain) return 0;
  const qg::ChainPlan& p = chain->plan;
  return p.packed_bytes + sizeof(qg::ChainProj) * p.nproj + sizeof(int) * (p.grid + 1 + p.nlevels) +
         sizeof(unsigned) * (p.nlevels + 1);
}

qg_status qgemm_w4a16_skinny(const uint32_t* wq, const uint16_t* scales_f16, const uint16_t* biases_f16,
                             const uint16_t* x_bf16, float* y, int M, int N, int K, int group_size,
                             void* workspace, size_t ws_bytes, void* stream) {
  qg_status st = check_w4(wq, scales_f16, biases_f16, x_bf16, y, M, N, K, group_size);
  if (st != QG_OK) return st;
  if (ws_bytes < qg_skinny_workspace_size(M, N, K, group_size)) return QG_ERR_WORKSPACE;
  if (ws_bytes && !workspace) return QG_ERR_INVALID_ARG;
  if (workspace && !aligned16(workspace)) return QG_ERR_MISALIGNED;
  return run_w4(wq, scales_f16, biases_f16, x_bf16, y, M, N, K, group_size, workspace, ws_bytes, stream);
}

struct qg_w4_skinny_group {
  qg::TcGroupPlan plan;
};

qg_status qgemm_w4a16_skinny_group_create(const qg_w4_gemm_desc* descs, int count, int group_size,
                                          qg_w4_skinny_group** group) {
  if (!descs || !group || count < 1) return QG_ERR_INVALID_ARG;
  if (group_size == 32 || group_size == 128) return QG_ERR_UNSUPPORTED;  // grouped launches: g64 only
  std::vector<qg::TcGroupItem> list(count);
  for (int i = 0; i < count; ++i) {
    const qg_w4_gemm_desc& d = descs[i];
    qg_status st = check_w4(d.wq, d.scales_f16, d.biases_f16, d.x_bf16, d.y, d.M, d.N, d.K, group_size);
    if (st != QG_OK) return st;
    list[i] = qg::TcGroupItem{d.wq, d.scales_f16, d.biases_f16, d.x_bf16, d.y, d.M, d.N, d.K};
  }
  if (qg::tc_group_check(list.data(), count) != 0) return QG_ERR_UNSUPPORTED;
  auto* out = new (std::nothrow) qg_w4_skinny_group();
  if (!out) return QG_ERR_CUDA;
  if (qg::tc_group_plan_build(list.data(), count, qg::device_sm_count(), &out->plan) != cudaSuccess) {
    delete out;
    return QG_ERR_CUDA;
  }
  *group = out;
  return QG_OK;
}

qg_status qgemm_w4a16_skinny_group_run(const qg_w4_skinny_group* group, void* stream) {
  if (!group) return QG_ERR_INVALID_ARG;
  uint32_t* err = err_word();
  if (!err) return QG_ERR_CUDA;
  return from_cuda(qg::tc_group_launch(group->plan, err, static_cast<cudaStream_t>(stream), g_pdl));
}

void qgemm_w4a16_skinny_group_destroy(qg_w4_skinny_group* group) {
  if (!group) return;
  qg::tc_group_plan_free(&group->plan);
  delete group;
}

size_t qg_moe_workspace_size(int T, int H, int I, int E, int top_k) {
  if (T < 1 || H < 1 || I < 1 || E < 1 || top_k < 1) return 0;
  return qg::moe_layout(T, H, I, E, top_k).total;
}

size_t qg_workspace_size(int op, int M, int N, int K, int T, int E, int top_k) {
  switch (op) {
    case QG_OP_GEMV_W4A16: return qg_gemv_workspace_size(N, K, 64);
    case QG_OP_SKINNY_W4A16: return qg_skinny_workspace_size(M, N, K, 64);
    case QG_OP_MOE_MXFP4: return qg_moe_workspace_size(T, N, K, E, top_k);
    case QG_OP_W8A8_HADAMARD: return qg_w8a8_hadamard_workspace_size(M, K);
    default: return 0;  // the Hadamard quantizer and the int32 W8A8 product need none
  }
}

size_t qg_moe_workspace_h_offset(int T, int H, int I, int E, int top_k) {
  if (T < 1 || H < 1 || I < 1 || E < 1 || top_k < 1) return 0;
  return qg::moe_layout(T, H, I, E, top_k).h;
}

qg_status moe_mxfp4_expert_forward(const uint16_t* x_bf16, const float* router_logits, const uint8_t* gate_q,
                                   const uint8_t* gate_e8m0, const uint8_t* up_q, const uint8_t* up_e8m0,
                                   const uint8_t* down_q, const uint8_t* down_e8m0, int T, int H, int I, int E,
                                   int top_k, float* y, int32_t* topk_idx, float* topk_w, void* workspace,
                                   size_t ws_bytes, void* stream) {
  if (!x_bf16 || !router_logits || !gate_q || !gate_e8m0 || !up_q || !up_e8m0 || !down_q || !down_e8m0 || !y ||
      !topk_idx || !topk_w)
    return QG_ERR_INVALID_ARG;
  if (T < 1 || H < 64 || I < 64 || E < 1 || top_k < 1) return QG_ERR_INVALID_ARG;
  if (H % 64 != 0 || I % 64 != 0 || top_k > E) return QG_ERR_INVALID_ARG;
  if (E > 1024 || top_k > 32 || (long long)T * top_k > 2048) return QG_ERR_UNSUPPORTED;
  const void* ptrs[] = {x_bf16, router_logits, gate_q, gate_e8m0, up_q, up_e8m0, down_q, down_e8m0,
                        y,      topk_idx,      topk_w};
  for (const void* p : ptrs)
    if (!aligned16(p)) return QG_ERR_MISALIGNED;
  if (!workspace || ws_bytes < qg_moe_workspace_size(T, H, I, E, top_k)) return QG_ERR_WORKSPACE;
  if (!aligned16(workspace)) return QG_ERR_MISALIGNED;
  uint32_t* err = err_word();
  if (!err) return QG_ERR_CUDA;
  return from_cuda(qg::launch_moe_mxfp4(x_bf16, router_logits, gate_q, gate_e8m0, up_q, up_e8m0, down_q,
                                        down_e8m0, T, H, I, E, top_k, y, topk_idx, topk_w, workspace, err,
                                        static_cast<cudaStream_t>(stream), g_pdl));
}

qg_status hadamard32_quant_i8(const uint16_t* x_bf16, const uint32_t* sign_bits, int8_t* q, float* scale, int M,
                              int K, void* stream) {
  if (!x_bf16 || !sign_bits || !q || !scale) return QG_ERR_INVALID_ARG;
  if (M < 1 || K < 32 || K % 32 != 0) return QG_ERR_INVALID_ARG;
  if (K > 49152) return QG_ERR_UNSUPPORTED;
  if (!aligned16(x_bf16) || !aligned16(sign_bits) || !aligned16(q) || !aligned16(scale)) return QG_ERR_MISALIGNED;
  return from_cuda(qg::launch_hadamard32_quant_i8(x_bf16, sign_bits, q, scale, M, K,
                                                  static_cast<cudaStream_t>(stream), g_pdl));
}

qg_status gemm_w8a8_i32(const int8_t* a, const int8_t* w, int32_t* c, int M, int N, int K, void* stream) {
  if (!a || !w || !c) return QG_ERR_INVALID_ARG;
  if (M < 1 || M > 32 || N < 1 || K < 64 || K % 64 != 0) return QG_ERR_INVALID_ARG;
  if ((long long)K * 127 * 128 >= (1LL << 31)) return QG_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(w) || !aligned16(c)) return QG_ERR_MISALIGNED;
  return from_cuda(qg::launch_w8a8_i32(a, w, c, M, N, K, err_word(), static_cast<cudaStream_t>(stream), g_pdl));
}

int qg_last_cuda_error(void) { return static_cast<int>(t_last_cuda); }

qg_status qg_selftest_wait_timeout(int kind, uint32_t limit, void* stream) {
  if (kind == 0 ? (limit < 1 || limit > (1u << 22)) : kind == 1 ? (limit < 1 || limit > 1000000u) : true)
    return QG_ERR_INVALID_ARG;
  uint32_t* err = err_word();
  if (!err) return QG_ERR_CUDA;
  // a zero counter that nothing writes: the library's own 4 bytes, per device
  static unsigned* zero[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QG_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!zero[dev]) {
      void* p = nullptr;
      cudaError_t e = cudaMalloc(&p, sizeof(unsigned));
      if (e == cudaSuccess) e = cudaMemset(p, 0, sizeof(unsigned));
      if (e != cudaSuccess) return from_cuda(e);
      zero[dev] = static_cast<unsigned*>(p);
    }
  }
  return from_cuda(qg::launch_selftest_wait(kind, limit, zero[dev], err, static_cast<cudaStream_t>(stream)));
}

const char* qg_last_cuda_error_string(void) { return cudaGetErrorString(t_last_cuda); }

qg_status qg_device_error(uint32_t* code, int clear) {
  uint32_t* p = err_word();
  if (!p) return QG_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return QG_ERR_CUDA;
  if (clear && v) {
    const uint32_t z = 0;
    if (cudaMemcpy(p, &z, sizeof z, cudaMemcpyHostToDevice) != cudaSuccess) return QG_ERR_CUDA;
  }
  if (code) *code = v;
  return v ? QG_ERR_DEVICE_TIMEOUT : QG_OK;
}

}  // extern "C"
