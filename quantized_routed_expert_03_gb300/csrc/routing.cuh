// routing.cuh -- device building blocks of the router (route.cu) and the
// dispatch (dispatch.cu): the logits GEMV, the per-token warp selection and the
// one-block dispatch.
#pragma once
#include "common.cuh"

namespace qre {

// ---------------------------------------------------------------- logits

// Router logits of expert rows e0 and e0 + 1 for T <= TMAX tokens: threads
// 0..255 of the CTA, 128 per row, keep all tokens' partial sums in registers
// while W streams once; further threads only take part in the barrier.  The
// reduction order is fixed (deterministic).  xs (shared, T * H bf16, or null):
// the CTA first copies the tokens there with one round of loads issued
// together with the weight loads, instead of one dependent round per column
// block.
template <int TMAX>
__device__ __forceinline__ void logits_gemv_pair(int e0, int T, int H, int E, const uint16_t* __restrict__ x,
                                                 const float* __restrict__ W, float* __restrict__ logits,
                                                 float (*part)[4][TMAX], uint4* xs = nullptr) {
  const bool in_gemv = threadIdx.x < 256;
  const int row = (threadIdx.x >> 7) & 1;   // expert row within the pair
  const int c = threadIdx.x & 127;          // column slot
  const int warp_in_row = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
  const int e = e0 + row;
  float acc[TMAX];
#pragma unroll
  for (int t = 0; t < TMAX; ++t) acc[t] = 0.f;
  float4 wbuf[8];
  if (in_gemv && e < E) {
    const float* w = W + (size_t)e * H;
#pragma unroll
    for (int m = 0; m < 8; ++m) {   // all of this thread's weights in flight at once
      const int j = c * 4 + m * 512;
      wbuf[m] = j < H ? __ldg(reinterpret_cast<const float4*>(w + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  const uint16_t* xsrc = x;
  if (xs) {
    const int n16 = T * H / 8;
#pragma unroll 4
    for (int i = threadIdx.x; i < n16; i += blockDim.x) xs[i] = __ldg(reinterpret_cast<const uint4*>(x) + i);
    __syncthreads();
    xsrc = reinterpret_cast<const uint16_t*>(xs);
  }
  if (in_gemv && e < E) {
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int j = c * 4 + m * 512;
      if (j >= H) break;
      const float4 wv = wbuf[m];
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
          const uint2 xv = *reinterpret_cast<const uint2*>(xsrc + (size_t)t * H + j);
          float a = acc[t];
          a = fmaf(bf16_bits_to_float(xv.x & 0xFFFFu), wv.x, a);
          a = fmaf(bf16_bits_to_float(xv.x >> 16), wv.y, a);
          a = fmaf(bf16_bits_to_float(xv.y & 0xFFFFu), wv.z, a);
          a = fmaf(bf16_bits_to_float(xv.y >> 16), wv.w, a);
          acc[t] = a;
        }
      }
    }
  }
  if (in_gemv) {
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      float v = acc[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) part[row][warp_in_row][t] = v;
    }
  }
  __syncthreads();
  if (threadIdx.x < 2 * TMAX) {
    const int r = threadIdx.x / TMAX, t = threadIdx.x % TMAX;
    const int ee = e0 + r;
    if (ee < E && t < T) {
      const float v = ((part[r][0][t] + part[r][1][t]) + part[r][2][t]) + part[r][3][t];
      logits[(size_t)t * E + ee] = v;
    }
  }
}

// ---------------------------------------------------------------- selection

struct Cand {
  float v;
  int id;
};
__device__ __forceinline__ bool better(const Cand& a, const Cand& b) {
  return a.v > b.v || (a.v == b.v && a.id < b.id);
}

// One warp selects token t's experts from its logits row lg (E <= 32 * NSLOT,
// NSLOT <= 32: the expert slots each lane scans):
// sigmoid scores, selection score = score + bias, k rounds of warp arg-max
// (ties to the lower id), output in ascending id with weights s / sum(s)
// summed in ascending id order.  Writes idx/wout rows t and, if s_pick is not
// null, the k ids to s_pick.  sid/ssc: 16 shared entries of this warp.  The
// logits are read through L2 (they may come from other CTAs of the launch).
template <int NSLOT>
__device__ __forceinline__ void select_token_warp(int t, int E, int k, const float* lg, const float* bias,
                                                  int32_t* idx, float* wout, int* sid, float* ssc, int* s_pick) {
  const int lane = threadIdx.x & 31;
  float s[NSLOT], sel[NSLOT];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < NSLOT; ++i) {
    const int e = i * 32 + lane;
    if (e < E) {
      const float sc = 1.0f / (1.0f + expf(-__ldcg(lg + e)));
      s[i] = sc;
      sel[i] = bias ? sc + bias[e] : sc;
    } else {
      s[i] = 0.f;
      sel[i] = -INFINITY;
      taken |= 1u << i;
    }
  }
  int my_id = -1;
  float my_s = 0.f;
  for (int r = 0; r < k; ++r) {
    Cand best{-INFINITY, 0x7fffffff};
    int best_i = -1;
#pragma unroll
    for (int i = 0; i < NSLOT; ++i) {
      if (!(taken >> i & 1u)) {
        const Cand c{sel[i], i * 32 + lane};
        if (best_i < 0 || better(c, best)) {
          best = c;
          best_i = i;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Cand other{__shfl_xor_sync(0xffffffffu, best.v, o), __shfl_xor_sync(0xffffffffu, best.id, o)};
      if (better(other, best)) best = other;
    }
    const int owner = best.id & 31, slot = best.id >> 5;
    float sw = 0.f;
    if (lane == owner) {
#pragma unroll
      for (int i = 0; i < NSLOT; ++i)
        if (i == slot) {
          taken |= 1u << i;
          sw = s[i];
        }
    }
    sw = __shfl_sync(0xffffffffu, sw, owner);
    if (lane == r) {
      my_id = best.id;
      my_s = sw;
    }
  }
  // rank = number of picks with a smaller id
  int rank = 0;
  for (int j = 0; j < k; ++j) {
    const int other = __shfl_sync(0xffffffffu, my_id, j);
    if (lane < k && other < my_id) ++rank;
  }
  if (lane < k) {
    sid[rank] = my_id;
    ssc[rank] = my_s;
  }
  __syncwarp();
  if (lane == 0) {
    float tot = 0.f;
    for (int j = 0; j < k; ++j) tot += ssc[j];
    for (int j = 0; j < k; ++j) {
      idx[(size_t)t * k + j] = sid[j];
      wout[(size_t)t * k + j] = ssc[j] / tot;
      if (s_pick) s_pick[j] = sid[j];
    }
  }
  __syncwarp();
}

// ---------------------------------------------------------------- one-block top-k

// Selection key of expert e with selection score v: a larger key comes earlier
// in the selection order (score descending, id ascending).  The score's bits
// are mapped so that unsigned order is float order; no selection score is -0
// (a sigmoid in (0, 1] plus a bias rounds to +0 at most), so on finite scores
// this is exactly the comparison `v > w || (v == w && e < f)`.  Every key of
// an expert is above 0, the key of an empty thread.
__device__ __forceinline__ unsigned long long selection_key(float v, int e) {
  uint32_t b = __float_as_uint(v);
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)b << 32) | (0xFFFFFFFFu - (uint32_t)e);
}

// Top k (k <= 16) of one token's experts, one expert per thread: key from
// selection_key, or 0 for a thread without an expert.  Each warp sorts its 32
// keys (bitonic, descending) and offers its first k; every expert of the top k
// is offered (all experts before it are in the top k - 1, so no warp holds k
// of them ahead of it), and its rank among the offers is its rank among all
// experts.  The keys are distinct, so exactly k offers have rank < k.  Returns
// whether the thread's expert is picked.  All threads of the block call it
// (two barriers).  offers: shared, >= 32 * k keys; flag: shared, >= blockDim.x.
__device__ __forceinline__ bool block_topk(unsigned long long key, int k, unsigned long long* offers, int* flag) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  unsigned long long v = key;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
      v = keep_max ? (o > v ? o : v) : (o < v ? o : v);
    }
  }
  if (lane < k) offers[warp * k + lane] = v;
  flag[threadIdx.x] = 0;
  __syncthreads();
  const int n_off = nw * k;
  if ((int)threadIdx.x < n_off) {
    const unsigned long long mine = offers[threadIdx.x];
    int rank = 0;
    for (int j = 0; j < n_off; ++j) rank += offers[j] > mine ? 1 : 0;
    const uint32_t id = 0xFFFFFFFFu - (uint32_t)(mine & 0xFFFFFFFFu);
    if (rank < k && mine != 0ull && id < blockDim.x) flag[id] = 1;
  }
  __syncthreads();
  return flag[threadIdx.x] != 0;
}

// ---------------------------------------------------------------- dispatch

// Block-wide exclusive scan of one value per thread (blockDim.x <= 1024).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < nw) warp_tot[lane] = wi - w;
    if (lane == nw - 1) *total = wi;
  }
  __syncthreads();
  const int r = warp_tot[warp] + inc - v;
  __syncthreads();
  return r;
}

// Places the picks of one chunk for expert e: its picks in pick order from
// position base_e.
__device__ __forceinline__ void place_expert(const int* s_idx, int p0, int n, int e, int base_e, int32_t* perm,
                                             int32_t* inv_perm) {
  int pos = base_e;
  for (int i = 0; i < n; ++i) {
    if (s_idx[i] == e) {
      perm[pos] = p0 + i;
      inv_perm[p0 + i] = pos;
      ++pos;
    }
  }
}

// Places the picks of one chunk: thread e walks the chunk in pick order.
__device__ __forceinline__ void place_chunk(const int* s_idx, int p0, int n, int E, int base_e, int32_t* perm,
                                            int32_t* inv_perm) {
  if ((int)threadIdx.x < E) place_expert(s_idx, p0, n, threadIdx.x, base_e, perm, inv_perm);
}

// One CTA (E <= 4 * blockDim.x, blockDim.x <= 1024) dispatches the P picks in
// s_idx (shared; ids in [0, E), or -1 for a dropped pick): counts, offsets,
// the ascending active list and n_active, and the stable permutation.  Thread
// i owns the ceil(E / blockDim.x) consecutive experts from i * that, so one
// block scan over the threads' totals orders everything by expert id.
// s_cnt: 1024 shared ints; warp_tot: 32; total: 1.
__device__ __forceinline__ void dispatch_block(int P, int E, const int* s_idx, int32_t* counts, int32_t* offsets,
                                               int32_t* perm, int32_t* inv_perm, int32_t* active, int32_t* n_active,
                                               int* s_cnt, int* warp_tot, int* total) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += blockDim.x)
    if (s_idx[p] >= 0) atomicAdd(&s_cnt[s_idx[p]], 1);
  __syncthreads();
  const int ept = (E + blockDim.x - 1) / blockDim.x;   // <= 4
  const int e0 = threadIdx.x * ept;
  int c[4], csum = 0, fsum = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    c[i] = (i < ept && e0 + i < E) ? s_cnt[e0 + i] : 0;
    csum += c[i];
    fsum += c[i] > 0 ? 1 : 0;
  }
  int off = block_exclusive_scan(csum, warp_tot, total);
  int apos = block_exclusive_scan(fsum, warp_tot, total);
  if (threadIdx.x == 0) n_active[0] = *total;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = e0 + i;
    if (i < ept && e < E) {
      counts[e] = c[i];
      offsets[e] = off;
      if (c[i] > 0) active[apos++] = e;
      if (e == E - 1) offsets[E] = off + c[i];
      place_expert(s_idx, 0, P, e, off, perm, inv_perm);
      off += c[i];
    }
  }
}

}  // namespace qre
