// api.cu -- the C ABI: argument validation, workspace sizing, error reporting,
// the device status word, and dispatch to the kernel launchers.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "internal.h"

namespace {

thread_local char g_err[512] = "";

qre_status fail(qre_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

qre_status cuda_fail(cudaError_t e, const char* what) {
  return fail(QRE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

constexpr int kMaxDevices = 64;
constexpr uint64_t kMaxTestStallNs = 100000000ull;   // 100 ms

}  // namespace

// One status word per device; kernels OR QRE_DEV_* bits into it.
__device__ int g_qre_device_status;

namespace qre {

namespace {
std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};
std::atomic<uint64_t> g_test_stall_ns{0};
std::atomic<int> g_host_unit_cost{0};
}  // namespace

int host_unit_cost() { return g_host_unit_cost.load(std::memory_order_relaxed); }

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }
uint64_t test_stall_ns() { return g_test_stall_ns.load(std::memory_order_relaxed); }

void set_error_message(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

namespace {
struct DevCache {
  std::once_flag once;
  int sms = 0;
  int smem_optin = 0;
  int* status = nullptr;
};
DevCache g_dev[kMaxDevices];

DevCache& dev_cache() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) dev = 0;
  DevCache& c = g_dev[dev];
  std::call_once(c.once, [&c, dev]() {
    cudaDeviceGetAttribute(&c.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&c.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_qre_device_status) == cudaSuccess) c.status = static_cast<int*>(p);
  });
  return c;
}
}  // namespace

cudaError_t ensure_smem_limit(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> set;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_pair(dev, kernel);
  auto it = set.find(key);
  if (it != set.end() && it->second >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) set[key] = bytes;
  return e;
}

int device_sm_count() { return dev_cache().sms; }
int device_max_smem_optin() { return dev_cache().smem_optin; }
int* device_status_word() { return dev_cache().status; }

}  // namespace qre

namespace {

qre_status check_shape(const qre_layer_shape* s, int32_t T) {
  if (!s) return fail(QRE_ERR_INVALID_ARG, "shape is NULL");
  if (T < 0) return fail(QRE_ERR_INVALID_ARG, "T = %d is negative", T);
  if (s->hidden <= 0 || s->inter <= 0 || s->n_experts <= 0 || s->top_k <= 0 || s->group <= 0)
    return fail(QRE_ERR_INVALID_ARG, "shape fields must be positive (H=%d I=%d E=%d k=%d G=%d)", s->hidden,
                s->inter, s->n_experts, s->top_k, s->group);
  if (s->top_k > s->n_experts) return fail(QRE_ERR_INVALID_ARG, "top_k %d > n_experts %d", s->top_k, s->n_experts);
  if (s->group != 32 && s->group != 64 && s->group != 128)
    return fail(QRE_ERR_UNSUPPORTED, "group %d not in {32, 64, 128}", s->group);
  if (s->hidden % 128 || s->inter % 128 || s->hidden > 4096 || s->inter > 4096)
    return fail(QRE_ERR_UNSUPPORTED, "hidden %d and inter %d must be multiples of 128 and at most 4096", s->hidden,
                s->inter);
  if (s->n_experts > 1024) return fail(QRE_ERR_UNSUPPORTED, "n_experts %d > 1024", s->n_experts);
  if (s->top_k > 16) return fail(QRE_ERR_UNSUPPORTED, "top_k %d > 16", s->top_k);
  if ((long long)T * s->top_k > 65536) return fail(QRE_ERR_UNSUPPORTED, "T*top_k = %lld > 65536", (long long)T * s->top_k);
  return QRE_OK;
}

#define QRE_REQUIRE_PTR(p)                                                        \
  do {                                                                            \
    if (!(p)) return fail(QRE_ERR_INVALID_ARG, "%s is NULL", #p);                 \
    if (misaligned(p)) return fail(QRE_ERR_MISALIGNED, "%s is not 16-byte aligned", #p); \
  } while (0)

#define QRE_OPTIONAL_PTR(p)                                                        \
  do {                                                                             \
    if ((p) && misaligned(p)) return fail(QRE_ERR_MISALIGNED, "%s is not 16-byte aligned", #p); \
  } while (0)

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

qre_status check_workspace(const void* ws, size_t have, size_t need) {
  if (need == 0) return QRE_OK;
  if (!ws) return fail(QRE_ERR_INVALID_ARG, "workspace is NULL");
  if (misaligned(ws)) return fail(QRE_ERR_MISALIGNED, "workspace is not 16-byte aligned");
  if (have < need) return fail(QRE_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", have, need);
  return QRE_OK;
}

qre_status launched(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return cuda_fail(e, what);
  g_err[0] = '\0';
  return QRE_OK;
}

}  // namespace

extern "C" {

const char* qre_last_error(void) { return g_err; }

const char* qre_status_string(qre_status s) {
  switch (s) {
    case QRE_OK: return "QRE_OK";
    case QRE_ERR_INVALID_ARG: return "QRE_ERR_INVALID_ARG";
    case QRE_ERR_UNSUPPORTED: return "QRE_ERR_UNSUPPORTED";
    case QRE_ERR_MISALIGNED: return "QRE_ERR_MISALIGNED";
    case QRE_ERR_WORKSPACE: return "QRE_ERR_WORKSPACE";
    case QRE_ERR_CUDA: return "QRE_ERR_CUDA";
    case QRE_ERR_TIMEOUT: return "QRE_ERR_TIMEOUT";
    case QRE_ERR_DEVICE_CHECK: return "QRE_ERR_DEVICE_CHECK";
  }
  return "unknown";
}

int32_t qre_version(void) { return 100; }

qre_status qre_workspace_size(const qre_layer_shape* shape, int32_t T, size_t* bytes) {
  qre_status st = check_shape(shape, T);
  if (st != QRE_OK) return st;
  if (!bytes) return fail(QRE_ERR_INVALID_ARG, "bytes is NULL");
  size_t b = qre::route_ws_bytes(*shape, T);
  const size_t d = qre::dispatch_ws_bytes(*shape, T);
  const size_t f = T <= qre::kDecodeMaxTokens ? qre::ffn_ws_bytes(*shape, T) : qre::ffn_prefill_ws_bytes(*shape, T);
  if (d > b) b = d;
  if (f > b) b = f;
  *bytes = align256(b);
  g_err[0] = '\0';
  return QRE_OK;
}

qre_status qre_quantize(int32_t n_rows, int32_t k_dim, int32_t group, const float* w, uint8_t* packed,
                        uint16_t* scales, qre_stream_t stream) {
  if (group != 32 && group != 64 && group != 128) return fail(QRE_ERR_UNSUPPORTED, "group %d not in {32, 64, 128}", group);
  if (n_rows < 0 || n_rows % 128 || k_dim <= 0 || k_dim % group || k_dim % 64)
    return fail(QRE_ERR_INVALID_ARG,
                "need n_rows a multiple of 128 and k_dim a positive multiple of group and of 64 (got %d, %d)", n_rows,
                k_dim);
  if (n_rows == 0) return QRE_OK;
  QRE_REQUIRE_PTR(w);
  QRE_REQUIRE_PTR(packed);
  QRE_REQUIRE_PTR(scales);
  return launched(qre::launch_quantize(n_rows, k_dim, group, w, nullptr, packed, scales, qre::device_status_word(),
                                       reinterpret_cast<cudaStream_t>(stream)),
                  "qre_quantize launch");
}

qre_status qre_quantize_gate_up(int32_t inter, int32_t hidden, int32_t group, const float* w_gate, const float* w_up,
                                uint8_t* packed, uint16_t* scales, qre_stream_t stream) {
  if (group != 32 && group != 64 && group != 128) return fail(QRE_ERR_UNSUPPORTED, "group %d not in {32, 64, 128}", group);
  if (inter <= 0 || inter % 64 || hidden <= 0 || hidden % group || hidden % 64)
    return fail(QRE_ERR_INVALID_ARG, "need inter a positive multiple of 64 and hidden a positive multiple of group "
                "and of 64 (got %d, %d)", inter, hidden);
  QRE_REQUIRE_PTR(w_gate);
  QRE_REQUIRE_PTR(w_up);
  QRE_REQUIRE_PTR(packed);
  QRE_REQUIRE_PTR(scales);
  return launched(qre::launch_quantize(2 * inter, hidden, group, w_gate, w_up, packed, scales,
                                       qre::device_status_word(), reinterpret_cast<cudaStream_t>(stream)),
                  "qre_quantize_gate_up launch");
}

qre_status qre_route(const qre_layer_shape* shape, int32_t T, const uint16_t* x_bf16, const float* w_router,
                     const float* bias, int32_t* topk_idx, float* topk_w, void* workspace, size_t workspace_bytes,
                     qre_stream_t stream) {
  qre_status st = check_shape(shape, T);
  if (st != QRE_OK) return st;
  if (T == 0) return QRE_OK;
  QRE_REQUIRE_PTR(x_bf16);
  QRE_REQUIRE_PTR(w_router);
  QRE_OPTIONAL_PTR(bias);
  QRE_REQUIRE_PTR(topk_idx);
  QRE_REQUIRE_PTR(topk_w);
  st = check_workspace(workspace, workspace_bytes, qre::route_ws_bytes(*shape, T));
  if (st != QRE_OK) return st;
  return launched(qre::launch_route(*shape, T, x_bf16, w_router, bias, topk_idx, topk_w, workspace,
                                    reinterpret_cast<cudaStream_t>(stream)),
                  "qre_route launch");
}

qre_status qre_route_dispatch(const qre_layer_shape* shape, int32_t T, const uint16_t* x_bf16, const float* w_router,
                              const float* bias, int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                              int32_t* perm, int32_t* inv_perm, int32_t* active, int32_t* n_active, void* workspace,
                              size_t workspace_bytes, qre_stream_t stream) {
  qre_status st = check_shape(shape, T);
  if (st != QRE_OK) return st;
  if (T == 0) return QRE_OK;
  if (!qre::route_dispatch_fused(*shape, T)) {
    st = qre_route(shape, T, x_bf16, w_router, bias, topk_idx, topk_w, workspace, workspace_bytes, stream);
    if (st != QRE_OK) return st;
    return qre_dispatch(shape, T, topk_idx, counts, offsets, perm, inv_perm, active, n_active, workspace,
                        workspace_bytes, stream);
  }
  QRE_REQUIRE_PTR(x_bf16);
  QRE_REQUIRE_PTR(w_router);
  QRE_OPTIONAL_PTR(bias);
  QRE_REQUIRE_PTR(topk_idx);
  QRE_REQUIRE_PTR(topk_w);
  QRE_REQUIRE_PTR(counts);
  QRE_REQUIRE_PTR(offsets);
  QRE_REQUIRE_PTR(perm);
  QRE_REQUIRE_PTR(inv_perm);
  QRE_REQUIRE_PTR(active);
  QRE_REQUIRE_PTR(n_active);
  st = check_workspace(workspace, workspace_bytes, qre::route_ws_bytes(*shape, T));
  if (st != QRE_OK) return st;
  return launched(qre::launch_route_dispatch(*shape, T, x_bf16, w_router, bias, topk_idx, topk_w, counts, offsets,
                                             perm, inv_perm, active, n_active, workspace,
                                             reinterpret_cast<cudaStream_t>(stream)),
                  "qre_route_dispatch launch");
}

qre_status qre_dispatch(const qre_layer_shape* shape, int32_t T, const int32_t* topk_idx, int32_t* counts,
                        int32_t* offsets, int32_t* perm, int32_t* inv_perm, int32_t* active, int32_t* n_active,
                        void* workspace, size_t workspace_bytes, qre_stream_t stream) {
  qre_status st = check_shape(shape, T);
  if (st != QRE_OK) return st;
  if (T == 0) return QRE_OK;
  QRE_REQUIRE_PTR(topk_idx);
  QRE_REQUIRE_PTR(counts);
  QRE_REQUIRE_PTR(offsets);
  QRE_REQUIRE_PTR(perm);
  QRE_REQUIRE_PTR(inv_perm);
  QRE_REQUIRE_PTR(active);
  QRE_REQUIRE_PTR(n_active);
  st = check_workspace(workspace, workspace_bytes, qre::dispatch_ws_bytes(*shape, T));
  if (st != QRE_OK) return st;
  return launched(qre::launch_dispatch(*shape, T, topk_idx, counts, offsets, perm, inv_perm, active, n_active,
                                       workspace, qre::device_status_word(), reinterpret_cast<cudaStream_t>(stream)),
                  "qre_dispatch launch");
}

namespace {

// The expert FFN over the groups of `part` (qre::FfnPart); the routing
// arguments are only needed when routed groups are computed.
qre_status expert_ffn_part(const qre_layer_shape* shape, int32_t T, const uint16_t* x_bf16, const qre_slot* slots,
                           const int32_t* offsets, const int32_t* perm, const int32_t* active,
                           const int32_t* n_active, float* expert_out, void* workspace, size_t workspace_bytes,
                           qre_stream_t stream, int part, const char* name) {
  qre_status st = check_shape(shape, T);
  if (st != QRE_OK) return st;
  if (T == 0) return QRE_OK;
  QRE_REQUIRE_PTR(x_bf16);
  QRE_REQUIRE_PTR(slots);
  if (part != qre::kFfnShared) {
    QRE_REQUIRE_PTR(offsets);
    QRE_REQUIRE_PTR(perm);
    QRE_REQUIRE_PTR(active);
    QRE_REQUIRE_PTR(n_active);
  }
  QRE_REQUIRE_PTR(expert_out);
  cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
  const bool shared_only = part == qre::kFfnShared;
  if (T > qre::kDecodeMaxTokens) {
    if (!qre::ffn_prefill_supported(*shape))
      return fail(QRE_ERR_UNSUPPORTED, "no grouped-GEMM plan for hidden %d, inter %d, %d experts", shape->hidden,
                  shape->inter, shape->n_experts);
    st = check_workspace(workspace, workspace_bytes,
                         shared_only ? qre::ffn_prefill_shared_ws_bytes(*shape, T) : qre::ffn_prefill_ws_bytes(*shape, T));
    if (st != QRE_OK) return st;
    return launched(qre::launch_ffn_prefill(*shape, T, x_bf16, slots, offsets, perm, active, n_active, expert_out,
                                            workspace, qre::device_status_word(), st_, part),
                    name);
  }
  if (!qre::ffn_decode_supported(*shape))
    return fail(QRE_ERR_UNSUPPORTED, "no decode kernel plan for hidden %d, inter %d, group %d", shape->hidden,
                shape->inter, shape->group);
  st = check_workspace(workspace, workspace_bytes,
                       shared_only ? qre::ffn_shared_ws_bytes(*shape, T) : qre::ffn_ws_bytes(*shape, T));
  if (st != QRE_OK) return st;
  return launched(qre::launch_ffn_decode(*shape, T, x_bf16, slots, offsets, perm, active, n_active, expert_out,
                                         workspace, qre::device_status_word(), st_, part),
                  name);
}

}  // namespace

qre_status qre_expert_ffn(const qre_layer_shape* shape, int32_t T, const uint16_t* x_bf16, const qre_slot* slots,
                          const int32_t* offsets, const int32_t* perm, const int32_t* active,
                          const int32_t* n_active, float* expert_out, void* workspace, size_t workspace_bytes,
                          qre_stream_t stream) {
  return expert_ffn_part(shape, T, x_bf16, slots, offsets, perm, active, n_active, expert_out, workspace,
                         workspace_bytes, stream, qre::kFfnAll, "qre_expert_ffn launch");
}

qre_status qre_expert_ffn_routed(const qre_layer_shape* shape, int32_t T, const uint16_t* x_bf16,
                                 const qre_slot* slots, const int32_t* offsets, const int32_t* perm,
                                 const int32_t* active, const int32_t* n_active, float* expert_out, void* workspace,
                                 size_t workspace_bytes, qre_stream_t stream) {
  return expert_ffn_part(shape, T, x_bf16, slots, offsets, perm, active, n_active, expert_out, workspace,
                         workspace_bytes, stream, qre::kFfnRouted, "qre_expert_ffn_routed launch");
}

qre_status qre_expert_ffn_shared(const qre_layer_shape* shape, int32_t T, const uint16_t* x_bf16,
                                 const qre_slot* slots, float* expert_out, void* workspace, size_t workspace_bytes,
                                 qre_stream_t stream) {
  return expert_ffn_part(shape, T, x_bf16, slots, nullptr, nullptr, nullptr, nullptr, expert_out, workspace,
                         workspace_bytes, stream, qre::kFfnShared, "qre_expert_ffn_shared launch");
}

qre_status qre_shared_workspace_size(const qre_layer_shape* shape, int32_t T, size_t* bytes) {
  qre_status st = check_shape(shape, T);
  if (st != QRE_OK) return st;
  if (!bytes) return fail(QRE_ERR_INVALID_ARG, "bytes is NULL");
  const size_t b = T <= qre::kDecodeMaxTokens ? qre::ffn_shared_ws_bytes(*shape, T)
                                              : qre::ffn_prefill_shared_ws_bytes(*shape, T);
  *bytes = align256(b > 0 ? b : 1);
  g_err[0] = '\0';
  return QRE_OK;
}

qre_status qre_combine(const qre_layer_shape* shape, int32_t T, const float* expert_out, const float* topk_w,
                       const int32_t* inv_perm, float* y_f32, uint16_t* y_bf16, qre_stream_t stream) {
  qre_status st = check_shape(shape, T);
  if (st != QRE_OK) return st;
  if (T == 0) return QRE_OK;
  QRE_REQUIRE_PTR(expert_out);
  QRE_REQUIRE_PTR(topk_w);
  QRE_REQUIRE_PTR(inv_perm);
  QRE_REQUIRE_PTR(y_f32);
  QRE_OPTIONAL_PTR(y_bf16);
  return launched(qre::launch_combine(*shape, T, expert_out, topk_w, inv_perm, y_f32, y_bf16,
                                      reinterpret_cast<cudaStream_t>(stream)),
                  "qre_combine launch");
}

qre_status qre_cache_update(const qre_layer_shape* shape, int32_t n_slots, float decay, const int32_t* active,
                            const int32_t* n_active, float* scores, int32_t* expert_slot, int32_t* slot_expert,
                            const qre_slot* home, const qre_slot* slot_mem, qre_slot* table, int32_t* copy_list,
                            int32_t* n_copies, int32_t max_copies, qre_stream_t stream) {
  qre_status st = check_shape(shape, 0);
  if (st != QRE_OK) return st;
  if (n_slots < 1 || n_slots > 1024) return fail(QRE_ERR_UNSUPPORTED, "n_slots %d not in [1, 1024]", n_slots);
  if (max_copies < 1) return fail(QRE_ERR_INVALID_ARG, "max_copies %d < 1", max_copies);
  if (!(decay >= 0.0f && decay <= 1.0f)) return fail(QRE_ERR_INVALID_ARG, "decay must be in [0, 1]");
  QRE_REQUIRE_PTR(active);
  QRE_REQUIRE_PTR(n_active);
  QRE_REQUIRE_PTR(scores);
  QRE_REQUIRE_PTR(expert_slot);
  QRE_REQUIRE_PTR(slot_expert);
  QRE_REQUIRE_PTR(home);
  QRE_REQUIRE_PTR(slot_mem);
  QRE_REQUIRE_PTR(table);
  QRE_REQUIRE_PTR(copy_list);
  QRE_REQUIRE_PTR(n_copies);
  return launched(qre::launch_cache_update(shape->n_experts, n_slots, decay, active, n_active, scores, slot_expert,
                                           expert_slot, home, slot_mem, table, copy_list, n_copies, max_copies,
                                           qre::device_status_word(), reinterpret_cast<cudaStream_t>(stream)),
                  "qre_cache_update launch");
}

qre_status qre_cache_copy(const qre_layer_shape* shape, const qre_slot* home, const qre_slot* slot_mem,
                          const int32_t* copy_list, const int32_t* n_copies, int32_t max_copies, qre_stream_t stream) {
  qre_status st = check_shape(shape, 0);
  if (st != QRE_OK) return st;
  if (max_copies < 1) return fail(QRE_ERR_INVALID_ARG, "max_copies %d < 1", max_copies);
  QRE_REQUIRE_PTR(home);
  QRE_REQUIRE_PTR(slot_mem);
  QRE_REQUIRE_PTR(copy_list);
  QRE_REQUIRE_PTR(n_copies);
  return launched(qre::launch_cache_copy(*shape, home, slot_mem, copy_list, n_copies, max_copies,
                                         reinterpret_cast<cudaStream_t>(stream)),
                  "qre_cache_copy launch");
}

qre_status qre_stage_experts(const qre_layer_shape* shape, const qre_slot* host_table, const qre_slot* host_staging,
                             int32_t n_staging, qre_slot* host_out, qre_slot* table_out, int32_t* n_staged,
                             qre_stream_t stream) {
  qre_status st = check_shape(shape, 0);
  if (st != QRE_OK) return st;
  if (!host_table || !host_out || !n_staged) return fail(QRE_ERR_INVALID_ARG, "host_table, host_out and n_staged must be non-NULL");
  if (n_staging < 0 || (n_staging > 0 && !host_staging))
    return fail(QRE_ERR_INVALID_ARG, "n_staging %d with host_staging %p", n_staging, (const void*)host_staging);
  QRE_REQUIRE_PTR(table_out);
  const char* names[4] = {"w_gate_up", "s_gate_up", "w_down", "s_down"};
  const size_t H = shape->hidden, I = shape->inter, G = shape->group;
  const size_t bytes[4] = {I * H, 2 * I * (H / G) * 2, H * I / 2, H * (I / G) * 2};
  for (int j = 0; j < n_staging; ++j) {
    const qre_slot& s = host_staging[j];
    const void* ptrs[4] = {s.w_gate_up, s.s_gate_up, s.w_down, s.s_down};
    if (s.tier != 0 || s.reserved != 0) return fail(QRE_ERR_INVALID_ARG, "staging slot %d: tier must be 0", j);
    for (int i = 0; i < 4; ++i) {
      if (!ptrs[i]) return fail(QRE_ERR_INVALID_ARG, "staging slot %d: %s is NULL", j, names[i]);
      if (misaligned(ptrs[i])) return fail(QRE_ERR_MISALIGNED, "staging slot %d: %s is not 16-byte aligned", j, names[i]);
    }
  }
  for (int e = 0; e <= shape->n_experts; ++e) {
    const qre_slot& s = host_table[e];
    if (s.tier > 1 || s.reserved != 0) return fail(QRE_ERR_INVALID_ARG, "slot %d: tier %u / reserved %u", e, s.tier, s.reserved);
    if (s.tier == 1) {
      const void* ptrs[4] = {s.w_gate_up, s.s_gate_up, s.w_down, s.s_down};
      for (int i = 0; i < 4; ++i)
        if (!ptrs[i] || misaligned(ptrs[i]))
          return fail(QRE_ERR_INVALID_ARG, "slot %d: %s is NULL or not 16-byte aligned", e, names[i]);
    }
  }
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  int j = 0;
  for (int e = 0; e <= shape->n_experts; ++e) {
    const qre_slot& s = host_table[e];
    host_out[e] = s;
    if (s.tier != 1 || j >= n_staging) continue;
    const qre_slot& d = host_staging[j];
    const void* src[4] = {s.w_gate_up, s.s_gate_up, s.w_down, s.s_down};
    const void* dst[4] = {d.w_gate_up, d.s_gate_up, d.w_down, d.s_down};
    for (int i = 0; i < 4; ++i) {
      const cudaError_t err = cudaMemcpyAsync(const_cast<void*>(dst[i]), src[i], bytes[i], cudaMemcpyDefault, cs);
      if (err != cudaSuccess) return cuda_fail(err, "qre_stage_experts: copy");
    }
    host_out[e] = d;
    ++j;
  }
  const cudaError_t err =
      cudaMemcpyAsync(table_out, host_out, (size_t)(shape->n_experts + 1) * sizeof(qre_slot), cudaMemcpyHostToDevice, cs);
  if (err != cudaSuccess) return cuda_fail(err, "qre_stage_experts: table upload");
  *n_staged = j;
  g_err[0] = '\0';
  return QRE_OK;
}

qre_status qre_read_probe(const void* src, size_t bytes, uint32_t* sink, qre_stream_t stream) {
  QRE_REQUIRE_PTR(src);
  QRE_REQUIRE_PTR(sink);
  if (bytes == 0 || bytes % 16) return fail(QRE_ERR_INVALID_ARG, "bytes %zu must be a positive multiple of 16", bytes);
  return launched(qre::launch_read_probe(src, bytes, sink, reinterpret_cast<cudaStream_t>(stream)),
                  "qre_read_probe launch");
}

qre_status qre_validate_slots(const qre_layer_shape* shape, const qre_slot* host_slots) {
  qre_status st = check_shape(shape, 0);
  if (st != QRE_OK) return st;
  if (!host_slots) return fail(QRE_ERR_INVALID_ARG, "host_slots is NULL");
  const char* names[4] = {"w_gate_up", "s_gate_up", "w_down", "s_down"};
  // pass 1: structure (no CUDA calls)
  for (int e = 0; e <= shape->n_experts; ++e) {
    const qre_slot& s = host_slots[e];
    const void* ptrs[4] = {s.w_gate_up, s.s_gate_up, s.w_down, s.s_down};
    if (s.reserved != 0) return fail(QRE_ERR_INVALID_ARG, "slot %d: reserved field is %u, must be 0", e, s.reserved);
    if (s.tier > 1) return fail(QRE_ERR_INVALID_ARG, "slot %d: tier %u not in {0, 1}", e, s.tier);
    for (int i = 0; i < 4; ++i) {
      if (!ptrs[i]) return fail(QRE_ERR_INVALID_ARG, "slot %d: %s is NULL", e, names[i]);
      if (misaligned(ptrs[i])) return fail(QRE_ERR_MISALIGNED, "slot %d: %s is not 16-byte aligned", e, names[i]);
    }
  }
  // pass 2: each pointer is memory of the kind its tier says
  for (int e = 0; e <= shape->n_experts; ++e) {
    const qre_slot& s = host_slots[e];
    const void* ptrs[4] = {s.w_gate_up, s.s_gate_up, s.w_down, s.s_down};
    for (int i = 0; i < 4; ++i) {
      cudaPointerAttributes attr;
      const cudaError_t err = cudaPointerGetAttributes(&attr, ptrs[i]);
      if (err != cudaSuccess) {
        cudaGetLastError();
        return fail(QRE_ERR_INVALID_ARG, "slot %d: %s is not a CUDA pointer (%s)", e, names[i], cudaGetErrorName(err));
      }
      if (s.tier == 0 && attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return fail(QRE_ERR_INVALID_ARG, "slot %d: %s has tier 0 but is not device memory", e, names[i]);
      if (s.tier == 1 && (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr))
        return fail(QRE_ERR_INVALID_ARG, "slot %d: %s has tier 1 but is not device-mapped host memory", e, names[i]);
    }
  }
  g_err[0] = '\0';
  return QRE_OK;
}

qre_status qre_debug_wait_test(uint64_t wait_limit_ns, uint64_t stall_ns) {
  if (wait_limit_ns > qre::kWaitLimitNs)
    return fail(QRE_ERR_INVALID_ARG, "wait_limit_ns %llu is above the default of %llu",
                (unsigned long long)wait_limit_ns, (unsigned long long)qre::kWaitLimitNs);
  if (stall_ns > kMaxTestStallNs)
    return fail(QRE_ERR_INVALID_ARG, "stall_ns %llu is above %llu", (unsigned long long)stall_ns,
                (unsigned long long)kMaxTestStallNs);
  qre::g_wait_limit_ns.store(wait_limit_ns ? wait_limit_ns : qre::kWaitLimitNs, std::memory_order_relaxed);
  qre::g_test_stall_ns.store(stall_ns, std::memory_order_relaxed);
  g_err[0] = '\0';
  return QRE_OK;
}

qre_status qre_set_host_unit_cost(int32_t cost) {
  if (cost < 0 || cost > 64) return fail(QRE_ERR_INVALID_ARG, "host unit cost %d not in [0, 64]", cost);
  qre::g_host_unit_cost.store(cost, std::memory_order_relaxed);
  g_err[0] = '\0';
  return QRE_OK;
}

qre_status qre_read_device_status(qre_stream_t stream, int32_t* status) {
  if (!status) return fail(QRE_ERR_INVALID_ARG, "status is NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "qre_read_device_status: stream synchronize");
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_qre_device_status, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "qre_read_device_status: read");
  *status = v;
  g_err[0] = '\0';
  return QRE_OK;
}

qre_status qre_clear_device_status(qre_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "qre_clear_device_status: stream synchronize");
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_qre_device_status, &zero, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "qre_clear_device_status: write");
  g_err[0] = '\0';
  return QRE_OK;
}

}  // extern "C"
