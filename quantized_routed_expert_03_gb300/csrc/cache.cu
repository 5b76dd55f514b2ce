// cache.cu -- device-side LFU expert cache: manager and miss copy.
//
// The RTX PRO 6000 recipe (config.expert_cache.mechanism) runs, per MoE layer
// and decode step, one CUDA block right after routing: the LFU scores decay by
// 0.995, every miss takes the lowest-scoring slot that the current call does not
// use, the expert pointer tables are rewritten in place, and a copy kernel then
// streams the missed experts from host memory into their slots; both kernels
// read the miss count on the device, so decode never synchronizes with the host.
//
// Here the pointer table is the qre_slot table the expert FFN reads.  State per
// layer (device memory, owned by the caller):
//   scores[E]        fp32 LFU scores
//   expert_slot[E]   cache slot of each expert, -1 = not cached, -2 = static
//   slot_expert[S]   expert held by each slot, -1 = empty
// Rules (the same as the policy replay the tests compare against):
//   * scores[e] = fp32(fp32(scores[e] * decay) + [e used by this call]);
//   * misses (used, not static, not cached) in ascending expert id; each takes
//     the slot whose expert is not used by this call and has the lowest score
//     (empty slots first), ties to the lowest slot index; with no such slot the
//     miss stays host-resident for this call;
//   * the admitted expert's table entry points at its slot (tier 0), the evicted
//     expert's entry at its home copy (tier 1), and (expert, slot) is appended
//     to the copy list;
//   * a call admits at most max_copies experts (the copy list's capacity): a
//     later miss of the same call stays host-resident, its table entry unchanged.
#include "common.cuh"
#include "internal.h"

namespace qre {
namespace {

constexpr int kCacheThreads = 1024;

struct KeySlot {
  float key;
  int slot;
};

__device__ __forceinline__ bool key_less(const KeySlot& a, const KeySlot& b) {
  return a.key < b.key || (a.key == b.key && a.slot < b.slot);
}

__global__ void __launch_bounds__(kCacheThreads) cache_update_kernel(
    int E, int S, float decay, const int32_t* __restrict__ active, const int32_t* __restrict__ n_active,
    float* scores, int32_t* slot_expert, int32_t* expert_slot, const qre_slot* __restrict__ home,
    const qre_slot* __restrict__ slot_mem, qre_slot* table, int32_t* copy_list, int32_t* n_copies, int max_copies,
    int* status) {
  __shared__ unsigned char used[1024];
  __shared__ KeySlot wbest[32];
  __shared__ int n_adm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  int na = *n_active;
  na = na < 0 ? 0 : (na > E ? E : na);
  for (int e = tid; e < E; e += blockDim.x) used[e] = 0;
  if (tid == 0) n_adm = 0;
  __syncthreads();
  for (int i = tid; i < na; i += blockDim.x) {
    const int e = active[i];
    if (e >= 0 && e < E) used[e] = 1;
    else set_status(status, QRE_DEV_BAD_INDEX);
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    float s = __fmul_rn(scores[e], decay);
    if (used[e]) s = __fadd_rn(s, 1.0f);
    scores[e] = s;
  }
  __syncthreads();
  // misses in ascending expert id (active is ascending), until the copy list is full
  for (int i = 0; i < na; ++i) {
    if (n_adm >= max_copies) break;   // shared, written by thread 0 before the last barrier
    const int e = active[i];
    if (e < 0 || e >= E || expert_slot[e] != -1) continue;  // hit, static or bad id
    KeySlot best{INFINITY, 0x7fffffff};
    for (int s = tid; s < S; s += blockDim.x) {
      const int cur = slot_expert[s];
      if (cur >= 0 && cur < E && used[cur]) continue;
      const KeySlot c{cur < 0 ? -INFINITY : scores[cur], s};
      if (key_less(c, best)) best = c;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const KeySlot other{__shfl_xor_sync(0xffffffffu, best.key, o), __shfl_xor_sync(0xffffffffu, best.slot, o)};
      if (key_less(other, best)) best = other;
    }
    if (lane == 0) wbest[warp] = best;
    __syncthreads();
    if (tid == 0) {
      KeySlot b = wbest[0];
      for (int w = 1; w < nw; ++w)
        if (key_less(wbest[w], b)) b = wbest[w];
      if (b.slot < S) {
        const int s = b.slot, old = slot_expert[s];
        if (old >= 0 && old < E) {
          expert_slot[old] = -1;
          table[old] = home[old];
        }
        slot_expert[s] = e;
        expert_slot[e] = s;
        table[e] = slot_mem[s];
        copy_list[2 * n_adm] = e;
        copy_list[2 * n_adm + 1] = s;
        ++n_adm;
      }
    }
    __syncthreads();
  }
  if (tid == 0) *n_copies = n_adm;
}

// Copies the admitted experts' four arrays from their home copies (pinned host
// memory read over the host link) into their slots.  Work item = one 16-byte
// vector of one array of one copy; the grid strides over all of them, each
// thread with kCopyUnroll loads in flight before it stores (the host link's
// latency is long: one load at a time left it at a third of its read rate).
constexpr int kCopyUnroll = 8;

__device__ __forceinline__ void copy_vector(const qre_slot* home, const qre_slot* slot_mem, const int32_t* copy_list,
                                            long long per, long long n_wgu, long long n_sgu, long long n_wd,
                                            long long i, const uint4*& from, uint4*& to) {
  const int c = (int)(i / per);
  long long v = i - (long long)c * per;
  const int e = copy_list[2 * c], s = copy_list[2 * c + 1];
  const qre_slot& src = home[e];
  const qre_slot& dst = slot_mem[s];
  if (v < n_wgu) {
    from = reinterpret_cast<const uint4*>(src.w_gate_up);
    to = reinterpret_cast<uint4*>(const_cast<uint8_t*>(dst.w_gate_up));
  } else if ((v -= n_wgu) < n_sgu) {
    from = reinterpret_cast<const uint4*>(src.s_gate_up);
    to = reinterpret_cast<uint4*>(const_cast<uint16_t*>(dst.s_gate_up));
  } else if ((v -= n_sgu) < n_wd) {
    from = reinterpret_cast<const uint4*>(src.w_down);
    to = reinterpret_cast<uint4*>(const_cast<uint8_t*>(dst.w_down));
  } else {
    v -= n_wd;
    from = reinterpret_cast<const uint4*>(src.s_down);
    to = reinterpret_cast<uint4*>(const_cast<uint16_t*>(dst.s_down));
  }
  from += v;
  to += v;
}

__global__ void __launch_bounds__(256) cache_copy_kernel(const qre_slot* __restrict__ home,
                                                         const qre_slot* __restrict__ slot_mem,
                                                         const int32_t* __restrict__ copy_list,
                                                         const int32_t* __restrict__ n_copies, int max_copies,
                                                         long long n_wgu, long long n_sgu, long long n_wd,
                                                         long long n_sd) {
  int nc = *n_copies;
  nc = nc < 0 ? 0 : (nc > max_copies ? max_copies : nc);
  const long long per = n_wgu + n_sgu + n_wd + n_sd;   // 16-byte vectors per expert
  const long long total = per * nc;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i0 = (long long)blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += kCopyUnroll * stride) {
    uint4 val[kCopyUnroll];
    uint4* to[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const long long i = i0 + u * stride;
      if (i < total) {
        const uint4* from;
        copy_vector(home, slot_mem, copy_list, per, n_wgu, n_sgu, n_wd, i, from, to[u]);
        val[u] = __ldcs(from);
      }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u)
      if (i0 + u * stride < total) *to[u] = val[u];
  }
}

}  // namespace

cudaError_t launch_cache_update(int E, int S, float decay, const int32_t* active, const int32_t* n_active,
                                float* scores, int32_t* slot_expert, int32_t* expert_slot, const qre_slot* home,
                                const qre_slot* slot_mem, qre_slot* table, int32_t* copy_list, int32_t* n_copies,
                                int max_copies, int* status, cudaStream_t stream) {
  cache_update_kernel<<<1, kCacheThreads, 0, stream>>>(E, S, decay, active, n_active, scores, slot_expert, expert_slot,
                                                       home, slot_mem, table, copy_list, n_copies, max_copies, status);
  return cudaGetLastError();
}

cudaError_t launch_cache_copy(const qre_layer_shape& s, const qre_slot* home, const qre_slot* slot_mem,
                              const int32_t* copy_list, const int32_t* n_copies, int max_copies,
                              cudaStream_t stream) {
  const long long H = s.hidden, I = s.inter, G = s.group;
  const long long n_wgu = 2 * I * H / 2 / 16, n_sgu = 2 * I * (H / G) * 2 / 16;
  const long long n_wd = H * I / 2 / 16, n_sd = H * (I / G) * 2 / 16;
  const int grid = device_sm_count() * 4;
  cache_copy_kernel<<<grid > 0 ? grid : 1, 256, 0, stream>>>(home, slot_mem, copy_list, n_copies, max_copies, n_wgu,
                                                             n_sgu, n_wd, n_sd);
  return cudaGetLastError();
}

}  // namespace qre
