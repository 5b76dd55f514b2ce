// internal.h -- host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/qre.h"

namespace qre {

// Largest token count the bandwidth-bound decode FFN handles in one pass: the
// tokens (as E4M3 terms or fp16 parts) are the N side of its tcgen05 MMAs, at
// most 32 B-operand rows.
constexpr int kDecodeMaxTokens = 8;

// Bytes of each workspace region for a call with T tokens (each call uses its
// own region from offset 0; calls on one stream run one after the other).
size_t route_ws_bytes(const qre_layer_shape& s, int T);
size_t dispatch_ws_bytes(const qre_layer_shape& s, int T);
size_t ffn_ws_bytes(const qre_layer_shape& s, int T);
// The shared-expert-only FFN call keeps its own, smaller workspace.
size_t ffn_shared_ws_bytes(const qre_layer_shape& s, int T);
size_t ffn_prefill_shared_ws_bytes(const qre_layer_shape& s, int T);

// Which groups an expert-FFN launch computes.
enum FfnPart { kFfnAll = 0, kFfnRouted = 1, kFfnShared = 2 };

// Limit of the kernels' pipeline waits in ns (one second unless a test lowered
// it with qre_debug_wait_test), and the test hook's stall (0 = off).
uint64_t wait_limit_ns();
uint64_t test_stall_ns();
// Cost of a host-mapped unit in the decode kernels' range cut (<= 1: off).
int host_unit_cost();

// Sets the calling thread's qre_last_error() message (printf format).
void set_error_message(const char* fmt, ...);

// Device properties, cached per device.
int device_sm_count();
int device_max_smem_optin();
int* device_status_word();   // address of the current device's status word

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device (cached, so repeated launches and graph captures skip it).
cudaError_t ensure_smem_limit(const void* kernel, int bytes);

// Launches `kernel` as a programmatic dependent of the kernel before it in the
// stream (it may be scheduled while that kernel finishes).  Every kernel so
// launched executes griddepcontrol.wait before it reads or writes global
// memory that an earlier kernel touches, and lets its own dependent start
// (griddepcontrol.launch_dependents) only after that wait, so a dependent's
// early part never overlaps anything but its direct predecessor.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
  return err != cudaSuccess ? err : cudaGetLastError();
}

// Kernel launchers (return the launch error, cudaSuccess otherwise).
// w2 == nullptr: plain matrix of n_rows rows.  Otherwise the gate/up pair:
// n_rows = 2I output rows interleaved in blocks of 16 from w (gate) and w2 (up).
cudaError_t launch_quantize(int n_rows, int k_dim, int group, const float* w, const float* w2, uint8_t* packed,
                            uint16_t* scales, int* status, cudaStream_t stream);

// allow_tc: the workspace has route_ws_bytes (false: the logits only, the CUDA-core kernels).
cudaError_t launch_route(const qre_layer_shape& s, int T, const uint16_t* x, const float* w_router,
                         const float* bias, int32_t* topk_idx, float* topk_w, void* ws,
                         cudaStream_t stream, bool allow_tc = true);

// Router + dispatch in two launches (GEMV, then selection and dispatch in one
// CTA) when route_dispatch_fused(s, T) (one token); the outputs of launch_route
// followed by launch_dispatch.
bool route_dispatch_fused(const qre_layer_shape& s, int T);
cudaError_t launch_route_dispatch(const qre_layer_shape& s, int T, const uint16_t* x, const float* w_router,
                                  const float* bias, int32_t* topk_idx, float* topk_w, int32_t* counts,
                                  int32_t* offsets, int32_t* perm, int32_t* inv_perm, int32_t* active,
                                  int32_t* n_active, void* ws, cudaStream_t stream);

cudaError_t launch_dispatch(const qre_layer_shape& s, int T, const int32_t* topk_idx, int32_t* counts,
                            int32_t* offsets, int32_t* perm, int32_t* inv_perm, int32_t* active,
                            int32_t* n_active, void* ws, int* status, cudaStream_t stream);

// Returns cudaErrorInvalidValue when the shape has no decode kernel instance.
cudaError_t launch_ffn_decode(const qre_layer_shape& s, int T, const uint16_t* x, const qre_slot* slots,
                              const int32_t* offsets, const int32_t* perm, const int32_t* active,
                              const int32_t* n_active, float* expert_out, void* ws, int* status,
                              cudaStream_t stream, int part = kFfnAll);
bool ffn_decode_supported(const qre_layer_shape& s);

// Grouped-GEMM expert FFN for T > kDecodeMaxTokens (tcgen05, TMEM, TMA).
size_t ffn_prefill_ws_bytes(const qre_layer_shape& s, int T);
bool ffn_prefill_supported(const qre_layer_shape& s);
cudaError_t launch_ffn_prefill(const qre_layer_shape& s, int T, const uint16_t* x, const qre_slot* slots,
                               const int32_t* offsets, const int32_t* perm, const int32_t* active,
                               const int32_t* n_active, float* expert_out, void* ws, int* status,
                               cudaStream_t stream, int part = kFfnAll);

cudaError_t launch_cache_update(int E, int S, float decay, const int32_t* active, const int32_t* n_active,
                                float* scores, int32_t* slot_expert, int32_t* expert_slot, const qre_slot* home,
                                const qre_slot* slot_mem, qre_slot* table, int32_t* copy_list, int32_t* n_copies,
                                int max_copies, int* status, cudaStream_t stream);
cudaError_t launch_cache_copy(const qre_layer_shape& s, const qre_slot* home, const qre_slot* slot_mem,
                              const int32_t* copy_list, const int32_t* n_copies, int max_copies,
                              cudaStream_t stream);

// A streaming read of `bytes` bytes (device or host-mapped memory).
cudaError_t launch_read_probe(const void* src, size_t bytes, uint32_t* sink, cudaStream_t stream);

cudaError_t launch_combine(const qre_layer_shape& s, int T, const float* expert_out, const float* topk_w,
                           const int32_t* inv_perm, float* y_f32, uint16_t* y_bf16, cudaStream_t stream);

// 2-D bf16 row-major [rows][cols] tensor map: boxes of 64 columns x box_rows
// rows, 128-byte swizzle, zero fill outside.  False when the driver refuses it
// (e.g. a base that is not 16-byte aligned).
bool make_tmap_bf16(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows);

// Router logits on the tensor cores (long token batches): whether a call of T
// tokens takes them, the workspace they need beyond the logits (the router
// weights split into three bf16 parts), and the launch (split, then GEMM).
bool route_tc_wanted(const qre_layer_shape& s, int T);     // by shape (workspace sizing)
bool route_tc_eligible(const qre_layer_shape& s, int T);   // and shared memory of this device
size_t route_tc_split_bytes(const qre_layer_shape& s);
// Returns false when the tensor maps cannot be made (nothing launched then).
bool launch_route_logits_tc(const qre_layer_shape& s, int T, const uint16_t* x, const float* w_router,
                            float* logits, void* split_ws, cudaStream_t stream, cudaError_t* err);

}  // namespace qre
