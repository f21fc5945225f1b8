// moe_mxfp4_expert_forward_noalloc: the MXFP4 MoE forward without a caller
// workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// layer: a plugin inside a host inference server that is handed only its input
// and output buffers, a runtime whose device memory is one pool reserved at
// start-up, or code running while a CUDA graph is being captured (cudaMalloc
// is not allowed during capture and can synchronize the device otherwise).
// This entry point serves them with scratch memory that lives inside the
// library: a statically sized device array, present on every GPU that loads
// the library until the process exits.
//
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "qg_internal.h"
#include "qgemv.h"

namespace {

constexpr size_t kNoallocBytes = QG_MOE_NOALLOC_MAX_BYTES;

// The scratch itself. In host code this name is only a host-side stand-in for
// the device symbol; its device address comes from cudaGetSymbolAddress.
__device__ __align__(256) uint8_t g_moe_scratch[kNoallocBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device, looked up once
// per device (the first call on a device does this; make that first call
// before any stream capture begins).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_moe_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

size_t qg_moe_noalloc_max_bytes(void) { return kNoallocBytes; }

qg_status moe_mxfp4_expert_forward_noalloc(const uint16_t* x_bf16, const float* router_logits,
                                           const uint8_t* gate_q, const uint8_t* gate_e8m0, const uint8_t* up_q,
                                           const uint8_t* up_e8m0, const uint8_t* down_q,
                                           const uint8_t* down_e8m0, int T, int H, int I, int E, int top_k,
                                           float* y, int32_t* topk_idx, float* topk_w, void* stream) {
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
  // the internal scratch has a fixed size: larger problems are refused
  if (qg::moe_layout(T, H, I, E, top_k).total > kNoallocBytes) return QG_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return QG_ERR_CUDA;
  // device-side timeouts go to the library's error word, read by qg_device_error
  uint32_t* err = qg::err_word();
  if (!err) return QG_ERR_CUDA;
  // Every MoE stage writes each scratch byte it later reads (routing lists,
  // operand images, h), and the counters that must start at zero are cleared
  // by the first kernel of every call, so stale contents from an earlier call
  // are harmless.
  const cudaError_t e = qg::launch_moe_mxfp4(x_bf16, router_logits, gate_q, gate_e8m0, up_q, up_e8m0, down_q,
                                             down_e8m0, T, H, I, E, top_k, y, topk_idx, topk_w, scratch, err,
                                             static_cast<cudaStream_t>(stream), false);
  return e == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // extern "C"
