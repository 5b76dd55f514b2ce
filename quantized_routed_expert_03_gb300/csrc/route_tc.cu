// route_tc.cu -- router logits for long token batches on the tensor cores.
//
// logits[T][E] = X[T][H] (bf16) * W[E][H]^T (fp32), the same function as the
// CUDA-core kernels of route.cu, computed exactly in its products: W is first
// split into three bf16 parts, W = W0 + W1 + W2 with Wi = bf16_rn(the rest),
// which holds W exactly (each rest is a multiple of W's last fp32 unit, and
// after two roundings to 8 significant bits at most 8 remain), and every
// product of a bf16 x with a bf16 part is exact in fp32.  A tcgen05 MMA
// (kind::f16, bf16 A and B, fp32 accumulator in tensor memory) then sums
// x * W0 + x * W1 + x * W2 over H; only the order and rounding of the fp32
// accumulation differ from the CUDA-core chain (both deterministic).  The
// prefill recipes route thousands of tokens per call; there the fp32 GEMM on
// CUDA cores was the third-largest kernel of the layer.
//
// One CTA per 128 tokens x NT experts (NT <= 256, a multiple of 16): warp 0
// TMA-loads each 64-wide K step (the token tile and the three part tiles,
// 128-byte swizzled) into a ring of stages, warp 1 issues the 12 MMAs of a
// step (3 parts x 4 K-slices of 16) and releases the stage by tcgen05.commit,
// warps 2-5 read the accumulator back (one token row per thread) and store it.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace qre {
namespace {

constexpr int kTcM = 128;          // tokens per CTA (UMMA M)
constexpr int kTcK = 64;           // reduction elements per stage: one 128-byte swizzled bf16 row
constexpr int kTcParts = 3;        // W = W0 + W1 + W2
constexpr int kTcThreads = 192;    // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kTcMinTokens = 1024;
constexpr uint32_t kTcCols = 256;  // tensor-memory columns (the fp32 accumulator, NT <= 256)

// Experts per CTA: E in ceil(E / 256) equal tiles, rounded up to 16 (UMMA N).
int tc_ntile(int E) {
  const int nn = (E + 255) / 256;
  const int nt = (E + nn - 1) / nn;
  return (nt + 15) / 16 * 16;
}

size_t tc_stage_bytes(int NT) { return (size_t)kTcM * 128 + (size_t)kTcParts * NT * 128; }

// Ring stages that fit (at least 2), or 0.
int tc_stages(int NT) {
  const long long budget = (long long)device_max_smem_optin() - 1024 - 256;
  const long long n = budget / (long long)tc_stage_bytes(NT);
  return n >= 2 ? (int)(n > 4 ? 4 : n) : 0;
}

// parts[p][i] = bf16 part p of w[i] (bf16 bits), n = E * H.
__global__ void __launch_bounds__(256) split_router_kernel(long long n, const float* __restrict__ w,
                                                           uint16_t* __restrict__ parts) {
  grid_dependency_wait();   // the workspace may still be read by the kernel before
  grid_dependents_launch();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const float v = w[i];
    const __nv_bfloat16 p0 = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(p0);   // exact
    const __nv_bfloat16 p1 = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(p1);  // exact, at most 8 significant bits
    parts[i] = __bfloat16_as_ushort(p0);
    parts[n + i] = __bfloat16_as_ushort(p1);
    parts[2 * n + i] = __bfloat16_as_ushort(__float2bfloat16_rn(r2));
  }
}

__global__ void __launch_bounds__(kTcThreads, 1)
    route_logits_tc(int T, int E, int H, int NT, int S, const __grid_constant__ CUtensorMap tx,
                    const __grid_constant__ CUtensorMap tw, float* __restrict__ logits, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t a_bytes = kTcM * 128, b_bytes = (uint32_t)NT * 128;
  const uint32_t stage_bytes = a_bytes + kTcParts * b_bytes;   // multiple of 1024
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * stage_bytes);
  uint64_t* empty = full + S;
  uint64_t* done = empty + S;
  uint64_t* drain = done + 1;
  uint32_t* tmem_p = reinterpret_cast<uint32_t*>(drain + 1);
  int* misc = reinterpret_cast<int*>(tmem_p + 1);
  volatile int* abort_flag = misc;   // a wait gave up
  int* issued = misc + 1;            // K steps whose loads the producer issued

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kTcM, n0 = blockIdx.y * NT;
  const int nk = H / kTcK;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    *issued = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_p, kTcCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dependency_wait();   // the split weights, and the tokens
  grid_dependents_launch();
  const uint32_t tmem = *tmem_p;

  if (warp == 0) {
    if (lane == 0) {
      int s = 0;
      for (; s < nk; ++s) {
        const int st = s % S;
        if (s >= S && !mbar_wait_bounded(&empty[st], ((s / S) - 1) & 1, abort_flag, status, kWaitLimitNs)) break;
        uint8_t* sb = smem + (size_t)st * stage_bytes;
        mbar_arrive_expect_tx(&full[st], stage_bytes);
        tma_load_2d(sb, &tx, s * kTcK, m0, &full[st]);
        for (int p = 0; p < kTcParts; ++p) tma_load_2d(sb + a_bytes + p * b_bytes, &tw, s * kTcK, p * E + n0, &full[st]);
      }
      *issued = s;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(kTcM, NT);
      for (int s = 0; s < nk; ++s) {
        const int st = s % S;
        if (!mbar_wait_bounded(&full[st], (s / S) & 1, abort_flag, status, kWaitLimitNs)) break;
        tc_fence_after();
        const uint32_t sa = smem_addr(smem + (size_t)st * stage_bytes);
#pragma unroll
        for (int p = 0; p < kTcParts; ++p)
#pragma unroll
          for (int kk = 0; kk < kTcK / 16; ++kk)
            umma_f16(tmem, umma_desc_sw128(sa + 32 * kk), umma_desc_sw128(sa + a_bytes + p * b_bytes + 32 * kk), idesc,
                     (s | p | kk) ? 1u : 0u);
        umma_commit(&empty[st]);
      }
      umma_commit(done);
    }
  } else {
    // epilogue: warp w reads tensor-memory lanes 32 (w mod 4) .. + 31, one token row per thread
    const int q = warp & 3;
    const int row = m0 + 32 * q + lane;
    // the tensor-memory loads below are warp-collective: the whole warp reads or none
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(done, 0, abort_flag, status, kWaitLimitNs) ? 1 : 0);
    tc_fence_after();
    if (ok) {
      float* out = logits + (size_t)row * E + n0;
      const bool vec = (E & 3) == 0;
      for (int c = 0; c < NT; c += 16) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c, v);
        tmem_ld_wait();
        if (row >= T) continue;
        if (vec && n0 + c + 16 <= E) {
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<float4*>(out + c + j) = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                                                   __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (n0 + c + j < E) out[c + j] = __uint_as_float(v[j]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    // a wait gave up: every tensor-core operation and every TMA load already
    // issued completes before the CTA frees tensor memory and exits
    const int n_iss = *issued;
    for (int s = n_iss - S > 0 ? n_iss - S : 0; s < n_iss; ++s) mbar_wait_drain(&full[s % S], (s / S) & 1, status);
  }
  if (*abort_flag && warp == 1 && lane == 0) {
    umma_commit(drain);
    mbar_wait_drain(drain, 0, status);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcCols);
  }
}

}  // namespace

bool route_tc_wanted(const qre_layer_shape& s, int T) {
  return T >= kTcMinTokens && s.hidden % kTcK == 0 && tc_ntile(s.n_experts) <= 256;
}

bool route_tc_eligible(const qre_layer_shape& s, int T) {
  return route_tc_wanted(s, T) && tc_stages(tc_ntile(s.n_experts)) >= 2;
}

size_t route_tc_split_bytes(const qre_layer_shape& s) {
  return (size_t)kTcParts * s.n_experts * s.hidden * sizeof(uint16_t);
}

bool launch_route_logits_tc(const qre_layer_shape& s, int T, const uint16_t* x, const float* w_router,
                            float* logits, void* split_ws, cudaStream_t stream, cudaError_t* err) {
  const int H = s.hidden, E = s.n_experts, NT = tc_ntile(E), S = tc_stages(NT);
  uint16_t* parts = static_cast<uint16_t*>(split_ws);
  CUtensorMap tx, tw;
  if (!make_tmap_bf16(&tx, x, T, H, kTcM) || !make_tmap_bf16(&tw, parts, (long long)kTcParts * E, H, NT)) return false;
  const long long n = (long long)E * H;
  const int sms = device_sm_count();
  const long long blocks = (n + 255) / 256;
  *err = launch_dependent(split_router_kernel, dim3((unsigned)(blocks < 4LL * sms ? blocks : 4LL * sms)), dim3(256), 0,
                          stream, n, w_router, parts);
  if (*err != cudaSuccess) return true;
  const int smem = (int)((size_t)S * tc_stage_bytes(NT) + 1024 + 256);
  *err = ensure_smem_limit(reinterpret_cast<const void*>(route_logits_tc), smem);
  if (*err != cudaSuccess) return true;
  dim3 grid((T + kTcM - 1) / kTcM, (E + NT - 1) / NT);
  *err = launch_dependent(route_logits_tc, grid, dim3(kTcThreads), (size_t)smem, stream, T, E, H, NT, S, tx, tw, logits,
                          device_status_word());
  return true;
}

}  // namespace qre
