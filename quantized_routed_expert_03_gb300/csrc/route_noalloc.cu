// route_noalloc.cu -- the router without a caller-supplied workspace.
//
// qre_route needs T * n_experts floats of scratch for the logits, which the
// caller normally passes as a workspace.  Some callers cannot allocate device
// memory at all: code running inside a host framework that owns every device
// allocation, real-time loops that must not allocate after start-up, and
// callers that only hold input and output buffers handed to them by someone
// else.  qre_route_noalloc serves them: its scratch is the fixed array below,
// which every GPU that loads this library keeps for the life of the process.
//
// The array is shared by every call.  Two calls whose kernels overlap on the
// GPU (for example on two streams without an ordering between them) race on it;
// calls on one stream, or otherwise ordered, are safe.  Nothing in it has to
// start at zero: every logit the selection reads is written first by the same
// call.  The array's device address is looked up once per device and kept; a
// device reset that destroys the primary context leaves it stale, so the entry
// point must not be called on that device again in the same process.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

// 65,536 floats (256 KiB): T * n_experts must not exceed this.
constexpr long long kRouteScratchFloats = 65536;
static __device__ __align__(256) float g_route_scratch[kRouteScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

extern "C" {

QRE_API qre_status qre_route_noalloc(const qre_layer_shape* shape, int32_t T, const uint16_t* x_bf16,
                                     const float* w_router, const float* bias, int32_t* topk_idx, float* topk_w,
                                     qre_stream_t stream) {
  size_t ws = 0;
  qre_status st = qre_workspace_size(shape, T, &ws);   // validates the shape and T (sets the message)
  if (st != QRE_OK) return st;
  if (T == 0) return QRE_OK;
  if ((long long)T * shape->n_experts > kRouteScratchFloats) {
    qre::set_error_message(
        "T * n_experts = %lld exceeds the fixed scratch of %lld floats; use qre_route with a workspace",
        (long long)T * shape->n_experts, kRouteScratchFloats);
    return QRE_ERR_UNSUPPORTED;
  }
  const void* ptrs[4] = {x_bf16, w_router, topk_idx, topk_w};
  const char* names[4] = {"x_bf16", "w_router", "topk_idx", "topk_w"};
  for (int i = 0; i < 4; ++i) {
    if (!ptrs[i]) {
      qre::set_error_message("%s is NULL", names[i]);
      return QRE_ERR_INVALID_ARG;
    }
    if (reinterpret_cast<uintptr_t>(ptrs[i]) & 15u) {
      qre::set_error_message("%s is not 16-byte aligned", names[i]);
      return QRE_ERR_MISALIGNED;
    }
  }
  if (bias && (reinterpret_cast<uintptr_t>(bias) & 15u)) {
    qre::set_error_message("bias is not 16-byte aligned");
    return QRE_ERR_MISALIGNED;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    qre::set_error_message("cudaGetDevice: %s", cudaGetErrorName(e));
    return QRE_ERR_CUDA;
  }
  float* scratch = nullptr;
  {
    // Set-up, once per device with that device current: the host name of the
    // array is only a stand-in, the kernels need its device address.
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_route_scratch);
      if (e != cudaSuccess || !p) {
        qre::set_error_message("cudaGetSymbolAddress: %s", cudaGetErrorName(e));
        return QRE_ERR_CUDA;
      }
      g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    scratch = g_scratch_ptr[dev];
  }
  e = qre::launch_route(*shape, T, x_bf16, w_router, bias, topk_idx, topk_w, scratch,
                        reinterpret_cast<cudaStream_t>(stream), /*allow_tc=*/false);   // the scratch holds logits only
  if (e != cudaSuccess) {
    qre::set_error_message("launch: %s (%s)", cudaGetErrorName(e), cudaGetErrorString(e));
    return QRE_ERR_CUDA;
  }
  qre::set_error_message("%s", "");
  return QRE_OK;
}

}  // extern "C"
