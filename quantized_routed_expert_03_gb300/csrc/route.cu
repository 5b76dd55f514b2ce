// route.cu -- router: fp32 logits, sigmoid scores, top-k, renormalised weights.
//
// Each token picks top_k of n_experts (8 of 288 in the GLM-5.3-Flash recipes:
// the RTX 3090 recipe's summary).  The scoring function is not on the pages;
// this library reads it as sigmoid scores with an optional selection-only bias,
// ties to the lower expert id, and weights s / sum(s) over the selection.
//
// Two logits kernels:
//   * T <= 16 (decode): a GEMV that streams W_r once; each CTA owns two expert
//     rows and keeps all T tokens' partial sums in registers.
//   * T > 16 (prefill): a tiled fp32 GEMM (64 tokens x 64 experts per CTA).
// Both accumulate in a fixed order, so results are deterministic.  Selection:
// for T <= 64 one CTA per token ranks every expert against all others in
// parallel; for larger T one warp per token runs k rounds of arg-max.  Both
// give the same bits (same fp32 scores, same exact order, same summation).
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
  grid_dependency_wait();
  grid_dependents_launch();
  logits_gemv_pair<TMAX>(blockIdx.x * 2, T, H, E, x, W, logits, part, stage ? xs_dyn : nullptr);
}

// logits[T][E] = X[T][H] (bf16) * W[E][H]^T (fp32), fp32 CUDA-core GEMM.
constexpr int BM = 64, BN = 64, BK = 32;
__global__ void __launch_bounds__(256) route_logits_gemm(int T, int H, int E, const uint16_t* __restrict__ x,
                                                         const float* __restrict__ W, float* __restrict__ logits) {
  __shared__ float xs[BK][BM + 4];
  __shared__ float ws[BK][BN + 4];
  grid_dependency_wait();
  grid_dependents_launch();
  const int tm = blockIdx.y * BM, en = blockIdx.x * BN;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;   // 16 x 16 threads, 4 x 4 outputs each
  float acc[4][4] = {};
  for (int k0 = 0; k0 < H; k0 += BK) {
    // load 64 x 32 of X and of W; 256 threads, 8 elements each
    for (int i = threadIdx.x; i < BM * BK / 4; i += 256) {
      const int r = i / (BK / 4), cc = (i % (BK / 4)) * 4;
      const int tok = tm + r;
      if (tok < T) {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(x + (size_t)tok * H + k0 + cc));
        xs[cc + 0][r] = bf16_bits_to_float(v.x & 0xFFFFu);
        xs[cc + 1][r] = bf16_bits_to_float(v.x >> 16);
        xs[cc + 2][r] = bf16_bits_to_float(v.y & 0xFFFFu);
        xs[cc + 3][r] = bf16_bits_to_float(v.y >> 16);
      } else {
        xs[cc + 0][r] = xs[cc + 1][r] = xs[cc + 2][r] = xs[cc + 3][r] = 0.f;
      }
      const int ex = en + r;
      if (ex < E) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(W + (size_t)ex * H + k0 + cc));
        ws[cc + 0][r] = v.x;
        ws[cc + 1][r] = v.y;
        ws[cc + 2][r] = v.z;
        ws[cc + 3][r] = v.w;
      } else {
        ws[cc + 0][r] = ws[cc + 1][r] = ws[cc + 2][r] = ws[cc + 3][r] = 0.f;
      }
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int tok = tm + ty * 4 + i;
    if (tok >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int ex = en + tx * 4 + j;
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

// One CTA per token (small T): every expert computes its rank in the order
// (selection score descending, id ascending) against all others; the k experts
// of rank < k are compacted in ascending id with a block-wide prefix count.
__global__ void __launch_bounds__(1024) route_select_rank(int T, int E, int k, const float* __restrict__ logits,
                                                          const float* __restrict__ bias, int32_t* __restrict__ idx,
                                                          float* __restrict__ wout) {
  __shared__ float sel_s[1024];
  __shared__ int wcount[32];
  __shared__ int chosen[16];
  __shared__ float chosen_s[16];
  grid_dependency_wait();
  grid_dependents_launch();
  const int t = blockIdx.x, e = threadIdx.x, lane = e & 31, warp = e >> 5;
  float sc = 0.f, my = -INFINITY;
  if (e < E) {
    sc = 1.0f / (1.0f + expf(-logits[(size_t)t * E + e]));
    my = bias ? sc + bias[e] : sc;
    sel_s[e] = my;
  }
  __syncthreads();
  int rank = 0;
  if (e < E) {
    for (int j = 0; j < E; ++j) {
      const float v = sel_s[j];
      rank += (v > my || (v == my && j < e)) ? 1 : 0;
    }
  }
  const bool pick = e < E && rank < k;
  const unsigned bal = __ballot_sync(0xffffffffu, pick);
  if (lane == 0) wcount[warp] = __popc(bal);
  __syncthreads();
  if (pick) {
    int pos = __popc(bal & ((1u << lane) - 1u));
    for (int w = 0; w < warp; ++w) pos += wcount[w];
    if (pos < 16) {
      chosen[pos] = e;
      chosen_s[pos] = sc;
    }
  }
  __syncthreads();
  if (e == 0) {
    float tot = 0.f;
    for (int j = 0; j < k; ++j) tot += chosen_s[j];
    for (int j = 0; j < k; ++j) {
      idx[(size_t)t * k + j] = chosen[j];
      wout[(size_t)t * k + j] = chosen_s[j] / tot;
    }
  }
}

}  // namespace

size_t route_ws_bytes(const qre_layer_shape& s, int T) { return (size_t)T * s.n_experts * sizeof(float); }

cudaError_t launch_route(const qre_layer_shape& s, int T, const uint16_t* x, const float* w_router,
                         const float* bias, int32_t* topk_idx, float* topk_w, void* ws, cudaStream_t stream) {
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
