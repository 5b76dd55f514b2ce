// combine_quant.cu -- the routing-weighted combine, and the weight quantizer.
#include "common.cuh"
#include "internal.h"

namespace qre {
namespace {

// y[t] = sum_j w[t][j] * eo[inv_perm[t*k + j]] + eo[T*k + t] in fp32, j ascending
// (ascending expert id), the shared term last.  Summing the expert partials in
// fp32 after the experts follows the glm53-flash-offload README ("CPU tier"
// bullet).  y_bf16 (optional) is round-to-nearest-even of y.
// KMAX > 0: top_k <= KMAX, and every weight, row index and expert row of the
// thread is loaded before the first sum (one round of memory latency instead
// of k dependent ones); KMAX == 0: any top_k, one pick at a time.  Same sums,
// same order, same bits either way.  A pick whose row index is out of range
// (one a dispatch that met a bad expert id left unset) adds nothing.
template <int KMAX>
__global__ void __launch_bounds__(256) combine_kernel(int T, int H, int k, const float* __restrict__ eo,
                                                      const float* __restrict__ w, const int32_t* __restrict__ inv_perm,
                                                      float* __restrict__ y, uint16_t* __restrict__ ybf) {
  grid_dependency_wait();
  grid_dependents_launch();
  const int t = blockIdx.y;
  const int h = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (t >= T || h >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  auto add = [&](float wj, const float4 v) {
    acc.x = fmaf(wj, v.x, acc.x);
    acc.y = fmaf(wj, v.y, acc.y);
    acc.z = fmaf(wj, v.z, acc.z);
    acc.w = fmaf(wj, v.w, acc.w);
  };
  const float4 sh = __ldg(reinterpret_cast<const float4*>(eo + ((size_t)T * k + t) * H + h));
  if constexpr (KMAX > 0) {
    float wj[KMAX];
    int qj[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k) {
        wj[j] = __ldg(w + (size_t)t * k + j);
        qj[j] = __ldg(inv_perm + (size_t)t * k + j);
      }
    // an out-of-range row index reads row 0 (the loads stay unconditional and in
    // bounds, all k in flight together) and its term is skipped in the sums
    float4 v[KMAX];
    uint32_t okm = 0;
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k) {
        const bool ok = (unsigned)qj[j] < (unsigned)(T * k);
        okm |= (ok ? 1u : 0u) << j;
        v[j] = __ldg(reinterpret_cast<const float4*>(eo + (size_t)(ok ? qj[j] : 0) * H + h));
      }
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k && ((okm >> j) & 1u)) add(wj[j], v[j]);
  } else {
    for (int j = 0; j < k; ++j) {
      const float wj = __ldg(w + (size_t)t * k + j);
      const int q = __ldg(inv_perm + (size_t)t * k + j);
      add(wj, (unsigned)q < (unsigned)(T * k) ? __ldg(reinterpret_cast<const float4*>(eo + (size_t)q * H + h))
                                              : make_float4(0.f, 0.f, 0.f, 0.f));
    }
  }
  acc.x += sh.x;
  acc.y += sh.y;
  acc.z += sh.z;
  acc.w += sh.w;
  *reinterpret_cast<float4*>(y + (size_t)t * H + h) = acc;
  if (ybf) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 out;
    out.x = *reinterpret_cast<const uint32_t*>(&lo);
    out.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(ybf + (size_t)t * H + h) = out;
  }
}

// Quantizer: each thread owns 8 consecutive elements of a row; G/8 threads form
// a group and share the group's max |w| through shuffles.
//   s = fp16_RNE(max|w| / 7), the quotient in fp64;
//   q = clamp(rint(w / s), -8, 7) in fp64 (0 when s == 0); nibble q + 8, even
//   element in the low nibble.
// With w2 != NULL the output is the gate/up pair stored row-interleaved in
// blocks of 16: output row r takes row 16*(r/32) + r%16 of w (r%32 < 16) or of
// w2 (otherwise).
__global__ void __launch_bounds__(256) quantize_kernel(long long n_threads, int K, int G, const float* __restrict__ w,
                                                       const float* __restrict__ w2, uint8_t* __restrict__ packed,
                                                       uint16_t* __restrict__ scales, int* status) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int tpg = G / 8;                      // threads per group: 4, 8 or 16
  const bool valid = i < n_threads;
  float v[8];
  float amax = 0.f;
  if (valid) {
    const long long orow = (i * 8) / K;
    const long long col8 = (i * 8 - orow * K) / 8;
    const float* src = w;
    long long srow = orow;
    if (w2) {
      const long long b = orow / 32, o = orow % 32;
      src = o < 16 ? w : w2;
      srow = 16 * b + (o % 16);
    }
    const float4* base = reinterpret_cast<const float4*>(src + srow * K) + 2 * col8;
    const float4 a = __ldg(base);
    const float4 b = __ldg(base + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
    // fmaxf drops NaN; keep it visible so the scale comes out non-finite
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (v[j] != v[j]) amax = v[j];
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = 0.f;
  }
  // group max over tpg consecutive lanes (groups never straddle a warp: tpg | 32)
  for (int o = 1; o < tpg; o <<= 1) {
    const float other = __shfl_xor_sync(0xffffffffu, amax, o);
    amax = (other != other || amax != amax) ? __int_as_float(0x7fc00000) : fmaxf(amax, other);
  }
  if (!valid) return;
  const __half s16 = __double2half((double)amax / 7.0);
  const double s = (double)__half2float(s16);
  const bool finite = isfinite(s);
  uint32_t word = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    int q = 0;
    if (finite && s > 0.0) {
      double r = rint((double)v[j] / s);
      r = r < -8.0 ? -8.0 : (r > 7.0 ? 7.0 : r);
      q = (int)r;
    }
    word |= (uint32_t)(q + 8) << (4 * j);
  }
  // tiled storage: 4 KB chunks of 128 rows x 64 elements; inside a chunk the
  // first 32 elements of every row (16 bytes each, rows in order), then the last 32
  const long long elem = i * 8;
  const long long row = elem / K;
  const int col = (int)(elem - row * K);
  const long long chunk = (row >> 7) * (K >> 6) + (col >> 6);
  const long long byte = chunk * 4096 + ((col >> 5) & 1) * 2048 + (row & 127) * 16 + ((col & 31) >> 1);
  reinterpret_cast<uint32_t*>(packed)[byte >> 2] = word;
  if (col % G == 0) {
    scales[((row >> 7) * (K / G) + col / G) * 128 + (row & 127)] = __half_as_ushort(s16);
    if (!finite) set_status(status, QRE_DEV_BAD_SCALE);
  }
}

}  // namespace

cudaError_t launch_combine(const qre_layer_shape& s, int T, const float* expert_out, const float* topk_w,
                           const int32_t* inv_perm, float* y_f32, uint16_t* y_bf16, cudaStream_t stream) {
  const int H = s.hidden;
  const int threads = T <= 8 ? 64 : 256;   // small batches: spread over more SMs
  dim3 grid((H / 4 + threads - 1) / threads, T);
  auto kernel = s.top_k <= 8 ? combine_kernel<8> : (s.top_k <= 16 ? combine_kernel<16> : combine_kernel<0>);
  return launch_dependent(kernel, grid, dim3(threads), 0, stream, T, H, s.top_k, expert_out, topk_w, inv_perm, y_f32,
                          y_bf16);
}

cudaError_t launch_quantize(int n_rows, int k_dim, int group, const float* w, const float* w2, uint8_t* packed,
                            uint16_t* scales, int* status, cudaStream_t stream) {
  const long long n_threads = (long long)n_rows * k_dim / 8;
  const long long blocks = (n_threads + 255) / 256;
  quantize_kernel<<<(unsigned)blocks, 256, 0, stream>>>(n_threads, k_dim, group, w, w2, packed, scales, status);
  return cudaGetLastError();
}

}  // namespace qre
