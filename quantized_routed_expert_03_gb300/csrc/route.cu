// route.cu -- router: fp32 logits, sigmoid scores, top-k, renormalised weights.
//
// Each token picks top_k of n_experts (8 of 288 in the GLM-5.3-Flash recipes:
// the RTX 3090 recipe's summary).  The scoring function is not on the pages;
// this library reads it as sigmoid scores with an optional selection-only bias,
// ties to the lower expert id, and weights s / sum(s) over the selection.
//
// Three logits kernels:
//   * T <= 16 (decode): a GEMV that streams W_r once; each CTA owns two expert
//     rows and keeps all T tokens' partial sums in registers.
//   * 16 < T < 1024: a tiled fp32 GEMM (64 tokens x 96 experts per CTA).
//   * T >= 1024: the tensor cores with W_r split into three exact bf16 parts
//     (route_tc.cu).
// Each accumulates in a fixed order, so results are deterministic.  Selection:
// for T <= 64 one CTA per token (block_topk: warp bitonic sorts, then ranks
// among the warps' offers); for larger T one warp per token runs k rounds of
// arg-max.  Both give the same bits (same fp32 scores, same exact order, same
// summation).
#include "common.cuh"
#include "internal.h"
#include "routing.cuh"

namespace qre {
namespace {

constexpr int kGemvTMax = 16;

template <int TMAX>
__global__ void __launch_bounds__(256) route_logits_gemv(int T, int H, int E, const uint16_t* __restrict__ x,
                                                         const float* __restrict__ W, float* __restrict__ logits,
                                                         int stage) {
  __shared__ float part[2][4][TMAX];
  extern __shared__ uint4 xs_dyn[];   // T * H bf16 when staged (dynamic size > 0)
  // While the kernel before finishes: start this CTA's two weight rows on their
  // way into L2 (a prefetch only warms the cache; the loads after the wait read
  // whatever is current).
  {
    const int e0 = blockIdx.x * 2, rows = E - e0 < 2 ? E - e0 : 2;
    const char* w0 = reinterpret_cast<const char*>(W + (size_t)e0 * H);
    for (int l = threadIdx.x; l < rows * H / 32; l += blockDim.x)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(w0 + 128 * l));
  }
  grid_dependency_wait();
  grid_dependents_launch();
  logits_gemv_pair<TMAX>(blockIdx.x * 2, T, H, E, x, W, logits, part, stage ? xs_dyn : nullptr);
}

// logits[T][E] = X[T][H] (bf16) * W[E][H]^T (fp32), fp32 CUDA-core GEMM for
// T > 16.  A CTA computes 64 tokens x 96 experts, each thread 4 x 6 outputs
// from 16-deep k slices held in shared memory (double-buffered: the next
// slice's global loads are in flight while the current one is consumed).  Every
// output is one fp32 FMA chain over k in ascending order, so the result does
// not depend on the tiling.
constexpr int TM = 4, TN = 6;   // outputs per thread: tokens x experts
constexpr int BM = 16 * TM, BN = 16 * TN, BK = 16;
__global__ void __launch_bounds__(256) route_logits_gemm(int T, int H, int E, const uint16_t* __restrict__ x,
                                                         const float* __restrict__ W, float* __restrict__ logits) {
  __shared__ __align__(16) float xs[2][BK][BM + 4];
  __shared__ __align__(16) float ws[2][BK][BN + 4];
  grid_dependency_wait();
  grid_dependents_launch();
  const int tm = blockIdx.y * BM, en = blockIdx.x * BN;
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;   // 16 x 16 threads: experts tx*TN.., tokens ty*TM..
  // global -> register staging of one k slice: X BM rows x 16 (one uint4 of 8
  // bf16 per thread, threads below 2 BM), W 96 rows x 16 (384 float4: threads
  // 0..255, then 0..127)
  const bool xl = tid < 2 * BM;
  const int xr = xl ? tid >> 1 : 0, xk = (tid & 1) * 8;
  uint4 xv;
  float4 wv[2];
  auto load_slice = [&](int k0) {
    const int tok = tm + xr;
    xv = (xl && tok < T) ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)tok * H + k0 + xk))
                         : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int f = tid + 256 * i;   // float4 index in the 96 x 4 slice
      const int er = f >> 2, kq = (f & 3) * 4;
      wv[i] = (f < BN * BK / 4 && en + er < E)
                  ? __ldg(reinterpret_cast<const float4*>(W + (size_t)(en + er) * H + k0 + kq))
                  : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto store_slice = [&](int buf) {
    const uint32_t v[4] = {xv.x, xv.y, xv.z, xv.w};
    if (xl) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        xs[buf][xk + 2 * j][xr] = bf16_bits_to_float(v[j] & 0xFFFFu);
        xs[buf][xk + 2 * j + 1][xr] = bf16_bits_to_float(v[j] >> 16);
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int f = tid + 256 * i;
      if (f < BN * BK / 4) {
        const int er = f >> 2, kq = (f & 3) * 4;
        ws[buf][kq + 0][er] = wv[i].x;
        ws[buf][kq + 1][er] = wv[i].y;
        ws[buf][kq + 2][er] = wv[i].z;
        ws[buf][kq + 3][er] = wv[i].w;
      }
    }
  };
  float acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
  load_slice(0);
  store_slice(0);
  __syncthreads();
  const int nk = H / BK;
  for (int ks = 0; ks < nk; ++ks) {
    const int buf = ks & 1;
    if (ks + 1 < nk) load_slice((ks + 1) * BK);
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[TM];
#pragma unroll
      for (int i = 0; i < TM; i += 4) {
        const float4 a4 = *reinterpret_cast<const float4*>(&xs[buf][kk][ty * TM + i]);
        a[i] = a4.x;
        a[i + 1] = a4.y;
        a[i + 2] = a4.z;
        a[i + 3] = a4.w;
      }
      float bv[TN];
#pragma unroll
      for (int j = 0; j < TN; j += 2) {
        const float2 b2 = *reinterpret_cast<const float2*>(&ws[buf][kk][tx * TN + j]);
        bv[j] = b2.x;
        bv[j + 1] = b2.y;
      }
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], bv[j], acc[i][j]);
    }
    if (ks + 1 < nk) store_slice(buf ^ 1);
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int tok = tm + ty * TM + i;
    if (tok >= T) continue;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int ex = en + tx * TN + j;
      if (ex < E) logits[(size_t)tok * E + ex] = acc[i][j];
    }
  }
}

// One warp per token (select_token_warp).
constexpr int kSelWarps = 8;
__global__ void __launch_bounds__(kSelWarps * 32) route_select(int T, int E, int k, const float* __restrict__ logits,
                                                               const float* __restrict__ bias, int32_t* __restrict__ idx,
                                                               float* __restrict__ wout) {
  __shared__ int sid[kSelWarps][16];
  __shared__ float ssc[kSelWarps][16];
  grid_dependency_wait();
  grid_dependents_launch();
  const int warp = threadIdx.x >> 5;
  const int t = blockIdx.x * kSelWarps + warp;
  if (t >= T) return;
  if (E <= 320)
    select_token_warp<10>(t, E, k, logits + (size_t)t * E, bias, idx, wout, sid[warp], ssc[warp], nullptr);
  else
    select_token_warp<32>(t, E, k, logits + (size_t)t * E, bias, idx, wout, sid[warp], ssc[warp], nullptr);
}

// One CTA per token (small T): block_topk picks the k experts (order:
// selection score descending, id ascending), which are then compacted in
// ascending id with a block-wide prefix count; each pick's thread writes its
// index and its weight s / sum(s), the sum taken in ascending id.
__global__ void __launch_bounds__(1024) route_select_rank(int T, int E, int k, const float* __restrict__ logits,
                                                          const float* __restrict__ bias, int32_t* __restrict__ idx,
                                                          float* __restrict__ wout) {
  __shared__ unsigned long long offers[32 * 16];
  __shared__ int flag[1024];
  __shared__ int wcount[32];
  __shared__ float chosen_s[16];
  grid_dependency_wait();
  grid_dependents_launch();
  const int t = blockIdx.x, e = threadIdx.x, lane = e & 31, warp = e >> 5;
  float sc = 0.f;
  unsigned long long key = 0ull;
  if (e < E) {
    sc = 1.0f / (1.0f + expf(-logits[(size_t)t * E + e]));
    key = selection_key(bias ? sc + bias[e] : sc, e);
  }
  const bool pick = block_topk(key, k, offers, flag);
  const unsigned bal = __ballot_sync(0xffffffffu, pick);
  if (lane == 0) wcount[warp] = __popc(bal);
  __syncthreads();
  int pos = __popc(bal & ((1u << lane) - 1u));
  for (int w = 0; w < warp; ++w) pos += wcount[w];
  if (pick) chosen_s[pos] = sc;   // exactly k picks: pos < k
  __syncthreads();
  if (pick) {
    float tot = 0.f;
    for (int j = 0; j < k; ++j) tot += chosen_s[j];
    idx[(size_t)t * k + pos] = e;
    wout[(size_t)t * k + pos] = sc / tot;
  }
}

// One token: selection and dispatch in one CTA, one dependent launch less
// between the router and the expert FFN.  The picks are those of
// route_select_rank, and for one token the dispatch is direct: the picks are
// distinct and already in ascending id, so pick j sits at position j (perm and
// inv_perm are the identity on 0..k-1), expert e's count is whether it was
// picked and its offset the number of picks below e -- the prefix count that
// places the picks.  The same bits as route_select_rank then dispatch_single.
// (For several tokens, a version whose last CTA dispatched all picks measured
// slower than the two kernels.)
__global__ void __launch_bounds__(1024) route_select_dispatch1(int E, int k, const float* __restrict__ logits,
                                                               const float* __restrict__ bias, int32_t* idx,
                                                               float* __restrict__ wout, int32_t* counts,
                                                               int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                                                               int32_t* active, int32_t* n_active) {
  __shared__ unsigned long long offers[32 * 16];
  __shared__ int flag[1024];
  __shared__ int wcount[32];
  __shared__ float chosen_s[16];
  grid_dependency_wait();
  grid_dependents_launch();
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  float sc = 0.f;
  unsigned long long key = 0ull;
  if (e < E) {
    sc = 1.0f / (1.0f + expf(-logits[e]));
    key = selection_key(bias ? sc + bias[e] : sc, e);
  }
  const bool pick = block_topk(key, k, offers, flag);
  const unsigned bal = __ballot_sync(0xffffffffu, pick);
  if (lane == 0) wcount[warp] = __popc(bal);
  __syncthreads();
  int pos = __popc(bal & ((1u << lane) - 1u));   // picks below e
  for (int w = 0; w < warp; ++w) pos += wcount[w];
  if (e < E) {
    counts[e] = pick ? 1 : 0;
    offsets[e] = pos;
    if (e == E - 1) offsets[E] = pos + (pick ? 1 : 0);
  }
  if (pick) {
    chosen_s[pos] = sc;   // exactly k picks: pos < k
    idx[pos] = e;
    active[pos] = e;
  }
  if (e < k) {
    perm[e] = e;
    inv_perm[e] = e;
  }
  if (e == 0) n_active[0] = k;
  __syncthreads();
  if (pick) {
    float tot = 0.f;
    for (int j = 0; j < k; ++j) tot += chosen_s[j];
    wout[pos] = sc / tot;
  }
}

}  // namespace

// The logits, and for long batches the router weights split into three bf16
// parts after them (route_tc.cu).
size_t route_logits_bytes(const qre_layer_shape& s, int T) {
  return ((size_t)T * s.n_experts * sizeof(float) + 255) & ~(size_t)255;
}

size_t route_ws_bytes(const qre_layer_shape& s, int T) {
  return route_tc_wanted(s, T) ? route_logits_bytes(s, T) + route_tc_split_bytes(s)
                               : (size_t)T * s.n_experts * sizeof(float);
}

bool route_dispatch_fused(const qre_layer_shape&, int T) { return T == 1; }

cudaError_t launch_route_dispatch(const qre_layer_shape& s, int T, const uint16_t* x, const float* w_router,
                                  const float* bias, int32_t* topk_idx, float* topk_w, int32_t* counts,
                                  int32_t* offsets, int32_t* perm, int32_t* inv_perm, int32_t* active,
                                  int32_t* n_active, void* ws, cudaStream_t stream) {
  float* logits = static_cast<float*>(ws);
  const int H = s.hidden, E = s.n_experts;
  const size_t xs_bytes = (size_t)T * H * 2;
  const int stage = xs_bytes <= 64 * 1024 ? 1 : 0;
  const size_t dyn = stage ? xs_bytes : 0;
  auto kernel = route_logits_gemv<8>;
  cudaError_t err;
  if (stage) {
    err = ensure_smem_limit(reinterpret_cast<const void*>(kernel), (int)dyn);
    if (err != cudaSuccess) return err;
  }
  err = launch_dependent(kernel, dim3((E + 1) / 2), dim3(256), dyn, stream, T, H, E, x, w_router, logits, stage);
  if (err != cudaSuccess) return err;
  return launch_dependent(route_select_dispatch1, dim3(1), dim3(((E + 31) / 32) * 32), 0, stream, E, s.top_k,
                          (const float*)logits, bias, topk_idx, topk_w, counts, offsets, perm, inv_perm, active,
                          n_active);
}

cudaError_t launch_route(const qre_layer_shape& s, int T, const uint16_t* x, const float* w_router,
                         const float* bias, int32_t* topk_idx, float* topk_w, void* ws, cudaStream_t stream,
                         bool allow_tc) {
  float* logits = static_cast<float*>(ws);
  const int H = s.hidden, E = s.n_experts;
  cudaError_t err;
  // the tokens go through shared memory when they fit (64 KB)
  const size_t xs_bytes = (size_t)T * H * 2;
  const int stage = xs_bytes <= 64 * 1024 ? 1 : 0;
  const size_t dyn = stage ? xs_bytes : 0;
  if (T <= kGemvTMax) {
    auto kernel = T <= 8 ? route_logits_gemv<8> : route_logits_gemv<kGemvTMax>;
    if (stage) {
      err = ensure_smem_limit(reinterpret_cast<const void*>(kernel), (int)dyn);
      if (err != cudaSuccess) return err;
    }
    err = launch_dependent(kernel, dim3((E + 1) / 2), dim3(256), dyn, stream, T, H, E, x, w_router, logits, stage);
  } else if (allow_tc && route_tc_eligible(s, T) &&
             launch_route_logits_tc(s, T, x, w_router, logits, static_cast<char*>(ws) + route_logits_bytes(s, T),
                                    stream, &err)) {
    // tensor cores (long batches; the CUDA-core GEMM below when the tensor maps cannot be made)
  } else {
    dim3 grid((E + BN - 1) / BN, (T + BM - 1) / BM);
    err = launch_dependent(route_logits_gemm, grid, dim3(256), 0, stream, T, H, E, x, w_router, logits);
  }
  if (err != cudaSuccess) return err;
  if (T <= 64)
    return launch_dependent(route_select_rank, dim3(T), dim3(((E + 31) / 32) * 32), 0, stream, T, E, s.top_k,
                            (const float*)logits, bias, topk_idx, topk_w);
  return launch_dependent(route_select, dim3((T + kSelWarps - 1) / kSelWarps), dim3(kSelWarps * 32), 0, stream, T, E,
                          s.top_k, (const float*)logits, bias, topk_idx, topk_w);
}

}  // namespace qre
