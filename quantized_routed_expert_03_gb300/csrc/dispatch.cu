// dispatch.cu -- per-expert histogram, offsets, stable permutation, active list.
//
// The glm53-flash-offload README ("Elastic CLOCK expert cache") dedups the
// router picks of a layer in one block; batched streams share the resulting
// expert union ("Batched decode").  Here the T*k picks p = t*k + j are ordered
// stably by (expert, p): perm[q] is the pick at sorted position q, inv_perm its
// inverse, offsets the exclusive prefix sum of the per-expert counts, and
// active the ascending list of experts with at least one pick.
//
// Every step is integer-exact and order-fixed, so the result is deterministic.
// Picks are cut into chunks of kChunk; each expert's thread walks a chunk in
// pick order, which makes the placement stable without any sort:
//   * one chunk (decode): a single CTA does count, scan and placement;
//   * several chunks (prefill): count per chunk, one scan CTA over (chunk,
//     expert), then placement per chunk from the chunk's base offsets.
#include "common.cuh"
#include "internal.h"
#include "routing.cuh"

namespace qre {
namespace {

constexpr int kChunk = 1024;

__device__ __forceinline__ int load_pick(const int32_t* idx, int p, int E, int* status) {
  const int e = idx[p];
  if (e < 0 || e >= E) {
    set_status(status, QRE_DEV_BAD_INDEX);
    return -1;
  }
  return e;
}

// Single CTA: the whole pick list is one chunk.  blockDim.x = max(E, 32) rounded up to a warp.
__global__ void __launch_bounds__(1024) dispatch_single(int P, int E, const int32_t* __restrict__ idx,
                                                         int32_t* counts, int32_t* offsets, int32_t* perm,
                                                         int32_t* inv_perm, int32_t* active, int32_t* n_active,
                                                         int* status) {
  grid_dependency_wait();
  grid_dependents_launch();
  __shared__ int s_idx[kChunk];
  __shared__ int s_cnt[1024];
  __shared__ int warp_tot[32];
  __shared__ int total;
  for (int p = threadIdx.x; p < P; p += blockDim.x) s_idx[p] = load_pick(idx, p, E, status);
  __syncthreads();
  dispatch_block(P, E, s_idx, counts, offsets, perm, inv_perm, active, n_active, s_cnt, warp_tot, &total);
}

// Multi-chunk, step 1: per-chunk counts -> ccount[chunk][E].
__global__ void __launch_bounds__(1024) dispatch_count(int P, int E, const int32_t* __restrict__ idx, int* ccount,
                                                        int* status) {
  grid_dependency_wait();
  grid_dependents_launch();
  __shared__ int s_cnt[1024];
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * kChunk;
  const int n = min(kChunk, P - p0);
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int e = load_pick(idx, p0 + i, E, status);
    if (e >= 0) atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) ccount[(size_t)blockIdx.x * E + e] = s_cnt[e];
}

// Multi-chunk, step 2 (one CTA): totals, offsets, active list; ccount becomes
// each chunk's base position per expert.
__global__ void __launch_bounds__(1024) dispatch_scan(int nchunk, int E, int* ccount, int32_t* counts,
                                                       int32_t* offsets, int32_t* active, int32_t* n_active) {
  grid_dependency_wait();
  grid_dependents_launch();
  __shared__ int warp_tot[32];
  __shared__ int total;
  const int e = threadIdx.x;
  int run = 0;
  if (e < E)
    for (int c = 0; c < nchunk; ++c) {
      const int v = ccount[(size_t)c * E + e];
      ccount[(size_t)c * E + e] = run;
      run += v;
    }
  const int off = block_exclusive_scan(run, warp_tot, &total);
  const int flag = run > 0 ? 1 : 0;
  const int apos = block_exclusive_scan(flag, warp_tot, &total);
  if (e < E) {
    counts[e] = run;
    offsets[e] = off;
    if (flag) active[apos] = e;
    for (int c = 0; c < nchunk; ++c) ccount[(size_t)c * E + e] += off;
  }
  if (threadIdx.x == 0) n_active[0] = total;
  if (e == E - 1) offsets[E] = off + run;
}

// Multi-chunk, step 3: placement per chunk.
__global__ void __launch_bounds__(1024) dispatch_place(int P, int E, const int32_t* __restrict__ idx,
                                                        const int* ccount, int32_t* perm, int32_t* inv_perm) {
  grid_dependency_wait();
  grid_dependents_launch();
  __shared__ int s_idx[kChunk];
  const int p0 = blockIdx.x * kChunk;
  const int n = min(kChunk, P - p0);
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int e = idx[p0 + i];
    s_idx[i] = (e >= 0 && e < E) ? e : -1;
  }
  __syncthreads();
  const int e = threadIdx.x;
  const int base = e < E ? ccount[(size_t)blockIdx.x * E + e] : 0;
  place_chunk(s_idx, p0, n, E, base, perm, inv_perm);
}

}  // namespace

size_t dispatch_ws_bytes(const qre_layer_shape& s, int T) {
  const long long P = (long long)T * s.top_k;
  const long long nchunk = (P + kChunk - 1) / kChunk;
  return nchunk > 1 ? (size_t)nchunk * s.n_experts * sizeof(int) : 0;
}

cudaError_t launch_dispatch(const qre_layer_shape& s, int T, const int32_t* topk_idx, int32_t* counts,
                            int32_t* offsets, int32_t* perm, int32_t* inv_perm, int32_t* active,
                            int32_t* n_active, void* ws, int* status, cudaStream_t stream) {
  const int P = T * s.top_k, E = s.n_experts;
  const int threads = ((E + 31) / 32) * 32;
  if (P <= kChunk) {
    return launch_dependent(dispatch_single, dim3(1), dim3(threads), 0, stream, P, E, topk_idx, counts, offsets, perm,
                            inv_perm, active, n_active, status);
  }
  const int nchunk = (P + kChunk - 1) / kChunk;
  int* ccount = static_cast<int*>(ws);
  cudaError_t err = launch_dependent(dispatch_count, dim3(nchunk), dim3(1024), 0, stream, P, E, topk_idx, ccount, status);
  if (err != cudaSuccess) return err;
  err = launch_dependent(dispatch_scan, dim3(1), dim3(threads), 0, stream, nchunk, E, ccount, counts, offsets, active,
                         n_active);
  if (err != cudaSuccess) return err;
  return launch_dependent(dispatch_place, dim3(nchunk), dim3(threads), 0, stream, P, E, topk_idx, ccount, perm,
                          inv_perm);
}

}  // namespace qre
