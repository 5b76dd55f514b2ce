// ffn_decode.cu -- bandwidth-bound fused dequant + SwiGLU expert FFN for T <= 8.
//
// The decode step of a routed MoE layer reads every byte of the union of the
// experts its tokens picked, plus the shared expert, once (glm53-flash-offload
// README, "Batched decode": streams share the per-layer expert union).  The
// work is a matrix-vector product per expert over 4-bit weights; the bound is
// HBM bandwidth, so the design goal is to stream packed weights at full rate
// and keep every other cost under it.
//
// Layout of the work
//   * A unit is 16 consecutive output rows of one expert's matrix over the full
//     reduction length K (16 x K/2 bytes of packed weights plus their scales).
//     Units of all active experts and the shared expert are split into equal
//     contiguous ranges, one per CTA; one CTA per SM (persistent).
//   * A producer warp streams each unit from HBM into a ring of shared-memory
//     stages with one 1-D bulk (TMA) copy per row, completing on an mbarrier.
//     Rows land at a pitch of 16 mod 128 bytes so the consumers' 32-bit loads are
//     free of bank conflicts.  Units of host-resident experts (slot tier 1) skip
//     the ring: the consumers read them with direct loads over the host link,
//     as the README's "Zero-copy home" does.
//   * 16 consumer warps split K; each warp owns a fixed K range, so the
//     activation operand for that range is loaded once into registers (gate/up)
//     or once per expert (down).  The tokens are the N = 8 side of the
//     m16n8k16 tensor-core MMA: rows of weights are M, T <= 8 tokens are N.  A
//     32-bit word of 8 nibbles decodes to four fp16 pairs of exact integer codes;
//     the MMA multiplies them by fp16 activations exactly and accumulates in
//     fp32 per quantization group, and the group's fp16 scale is applied in fp32.
//     The K order inside a 32-element chunk is permuted identically in weights
//     and activations, which leaves every dot product unchanged.
//   * Per unit, the 16 warps' partial sums are added in fixed warp order
//     (deterministic), and the result goes to the gate/up workspace (gate/up
//     kernel) or to the expert's output rows (down kernel).
// The down kernel computes h = silu(g) * u from the gate/up workspace while it
// loads its activation operand, and splits h into an fp16 high part and an fp16
// remainder so that its products stay accurate to about fp32.
#include "common.cuh"
#include "internal.h"

namespace qre {
namespace {

constexpr int kNW = 16;                    // consumer warps
constexpr int kThreads = (kNW + 1) * 32;   // + one producer warp
constexpr int kRows = 16;                  // output rows per unit (MMA M)
constexpr int kTok = kDecodeMaxTokens;     // MMA N
constexpr int kRedStride = 20;             // floats between token columns of a partial
constexpr int kRedWarp = kTok * kRedStride;

struct FfnParams {
  int H, I, E, k, G, T;
  int K;            // reduction length: H (gate/up) or I (down)
  int n_out;        // rows per expert: 2I (gate/up) or H (down)
  int gc;           // 32-element chunks per quantization group
  int aw;           // working consumer warps
  int pitch;        // shared-memory row pitch in bytes
  int stage_bytes;  // rows + scales of one unit
  int nstage;
  int amax;         // largest possible number of active experts, min(E, T*k)
  const uint16_t* x;
  const qre_slot* slots;
  const int32_t* offsets;
  const int32_t* perm;
  const int32_t* active;
  const int32_t* n_active;
  float* gu;          // [(max active + 1)][8][2I] fp32: gate/up outputs
  float* expert_out;  // [T*k + T][H]
  int* status;
};

struct Unit {
  const uint8_t* w;
  const uint16_t* s;
  int a;      // index in the active list; n_active = shared expert
  int e;      // expert id (E = shared)
  int r0;     // first output row
  bool host;  // read over the host link
  bool ok;
};

template <int MODE>
__device__ __forceinline__ Unit resolve_unit(const FfnParams& p, int u, int n_act, int units_per_exp) {
  Unit un;
  un.a = u / units_per_exp;
  un.r0 = (u - un.a * units_per_exp) * kRows;
  un.e = (un.a < n_act) ? __ldg(p.active + un.a) : p.E;
  un.ok = (un.e >= 0 && un.e <= p.E);
  if (!un.ok) {
    un.w = nullptr;
    un.s = nullptr;
    un.host = false;
    return un;
  }
  const qre_slot* sl = p.slots + un.e;
  const uint8_t* w = MODE == 0 ? sl->w_gate_up : sl->w_down;
  const uint16_t* s = MODE == 0 ? sl->s_gate_up : sl->s_down;
  un.host = sl->tier != 0;
  un.ok = w != nullptr && s != nullptr && ((reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(s)) & 15) == 0;
  un.w = w + (size_t)un.r0 * (p.K / 2);
  un.s = s + (size_t)un.r0 * (p.K / p.G);
  return un;
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float lds_half_as_float(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return __half2float(__ushort_as_half(v));
}
__device__ __forceinline__ uint32_t ldg_u32(const void* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}
__device__ __forceinline__ float ldg_half_as_float(const uint16_t* p) {
  return __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(p))));
}

// Dot products of one unit's 16 rows with the warp's K range.  SMEM selects
// shared-memory stage reads (wbase/sbase are shared addresses) or direct global
// reads (host-resident experts).  NB = 4 (one fp16 operand) or 8 (high + low).
template <int CPW, int NB, bool SMEM>
__device__ __forceinline__ void unit_dot(uintptr_t wbase, int wpitch, uintptr_t sbase, int s_stride, int c0,
                                         int gc, int g, int t, const uint32_t (&bfr)[CPW][NB], float (&acc)[4]) {
  float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int cl = 0; cl < CPW; ++cl) {
    const int c = c0 + cl;
    const uintptr_t off_lo = (uintptr_t)g * wpitch + c * 16 + t * 4;
    const uintptr_t off_hi = off_lo + (uintptr_t)8 * wpitch;
    uint32_t wlo, whi;
    if constexpr (SMEM) {
      wlo = lds_u32((uint32_t)(wbase + off_lo));
      whi = lds_u32((uint32_t)(wbase + off_hi));
    } else {
      wlo = ldg_u32(reinterpret_cast<const void*>(wbase + off_lo));
      whi = ldg_u32(reinterpret_cast<const void*>(wbase + off_hi));
    }
    uint32_t pl[4], ph[4];
    decode_nibbles(wlo, pl);
    decode_nibbles(whi, ph);
    mma_f16_16816(d, pl[0], ph[0], pl[1], ph[1], bfr[cl][0], bfr[cl][1]);
    if constexpr (NB == 8) mma_f16_16816(d, pl[0], ph[0], pl[1], ph[1], bfr[cl][4], bfr[cl][5]);
    mma_f16_16816(d, pl[2], ph[2], pl[3], ph[3], bfr[cl][2], bfr[cl][3]);
    if constexpr (NB == 8) mma_f16_16816(d, pl[2], ph[2], pl[3], ph[3], bfr[cl][6], bfr[cl][7]);
    if (((cl + 1) & (gc - 1)) == 0) {  // end of a quantization group
      const int grp = c / gc;
      float slo, shi;
      if constexpr (SMEM) {
        slo = lds_half_as_float((uint32_t)(sbase + ((uintptr_t)g * s_stride + grp) * 2));
        shi = lds_half_as_float((uint32_t)(sbase + ((uintptr_t)(g + 8) * s_stride + grp) * 2));
      } else {
        slo = ldg_half_as_float(reinterpret_cast<const uint16_t*>(sbase) + (size_t)g * s_stride + grp);
        shi = ldg_half_as_float(reinterpret_cast<const uint16_t*>(sbase) + (size_t)(g + 8) * s_stride + grp);
      }
      acc[0] = fmaf(slo, d[0], acc[0]);
      acc[1] = fmaf(slo, d[1], acc[1]);
      acc[2] = fmaf(shi, d[2], acc[2]);
      acc[3] = fmaf(shi, d[3], acc[3]);
      d[0] = d[1] = d[2] = d[3] = 0.f;
    }
  }
}

// Activation operand for gate/up: x[token g][32c + 8t .. +7] as fp16 pairs
// (x0,x4) (x1,x5) (x2,x6) (x3,x7), matching decode_nibbles' pair order.
template <int CPW>
__device__ __forceinline__ void load_x_frags(const FfnParams& p, int c0, int g, int t, uint32_t (&bfr)[CPW][4]) {
#pragma unroll
  for (int cl = 0; cl < CPW; ++cl) {
    if (g < p.T) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)g * p.H + (c0 + cl) * 32 + t * 8));
      const float f0 = bf16_bits_to_float(v.x & 0xFFFFu), f1 = bf16_bits_to_float(v.x >> 16);
      const float f2 = bf16_bits_to_float(v.y & 0xFFFFu), f3 = bf16_bits_to_float(v.y >> 16);
      const float f4 = bf16_bits_to_float(v.z & 0xFFFFu), f5 = bf16_bits_to_float(v.z >> 16);
      const float f6 = bf16_bits_to_float(v.w & 0xFFFFu), f7 = bf16_bits_to_float(v.w >> 16);
      bfr[cl][0] = pack_half2(f0, f4);
      bfr[cl][1] = pack_half2(f1, f5);
      bfr[cl][2] = pack_half2(f2, f6);
      bfr[cl][3] = pack_half2(f3, f7);
    } else {
      bfr[cl][0] = bfr[cl][1] = bfr[cl][2] = bfr[cl][3] = 0u;
    }
  }
}

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

// Activation operand for down: h = silu(g) * u for intermediate features
// 32c + 8t .. +7 of token column g, from the gate/up workspace of active
// index a, split into fp16 high parts (slots 0..3) and remainders (4..7).
template <int CPW>
__device__ __forceinline__ void load_h_frags(const FfnParams& p, int a, int c0, int g, int t, uint32_t (&bfr)[CPW][8]) {
  const float* gb = p.gu + ((size_t)a * kTok + g) * (2 * p.I);
#pragma unroll
  for (int cl = 0; cl < CPW; ++cl) {
    const int f0 = (c0 + cl) * 32 + t * 8;
    const int gate_row = 32 * (f0 / 16) + (f0 % 16);
    const float4 ga = *reinterpret_cast<const float4*>(gb + gate_row);
    const float4 gb4 = *reinterpret_cast<const float4*>(gb + gate_row + 4);
    const float4 ua = *reinterpret_cast<const float4*>(gb + gate_row + 16);
    const float4 ub4 = *reinterpret_cast<const float4*>(gb + gate_row + 20);
    const float gv[8] = {ga.x, ga.y, ga.z, ga.w, gb4.x, gb4.y, gb4.z, gb4.w};
    const float uv[8] = {ua.x, ua.y, ua.z, ua.w, ub4.x, ub4.y, ub4.z, ub4.w};
    float hi[8], lo[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float h = silu_f32(gv[i]) * uv[i];
      const __half hh = __float2half_rn(h);
      hi[i] = __half2float(hh);
      lo[i] = h - hi[i];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      bfr[cl][j] = pack_half2(hi[j], hi[j + 4]);
      bfr[cl][4 + j] = pack_half2(lo[j], lo[j + 4]);
    }
  }
}

// Output row of expert_out for token n of the unit's expert, or -1.
__device__ __forceinline__ int output_row(const FfnParams& p, const Unit& un, int n_act, int n) {
  if (n >= p.T) return -1;
  if (un.a >= n_act) return p.T * p.k + n;  // shared expert
  const int lo = __ldg(p.offsets + un.e), hi = __ldg(p.offsets + un.e + 1);
  for (int q = lo; q < hi; ++q)
    if (__ldg(p.perm + q) / p.k == n) return q;
  return -1;
}

template <int MODE, int CPW>
__global__ void __launch_bounds__(kThreads, 1) ffn_decode_kernel(const FfnParams p) {
  constexpr int NB = MODE == 0 ? 4 : 8;
  extern __shared__ __align__(128) uint8_t smem[];
  int n_act = *p.n_active;
  n_act = n_act < 0 ? 0 : (n_act > p.amax ? p.amax : n_act);
  const int units_per_exp = p.n_out / kRows;
  const int U = (n_act + 1) * units_per_exp;
  const int ub = (int)((long long)blockIdx.x * U / gridDim.x);
  const int ue = (int)((long long)(blockIdx.x + 1) * U / gridDim.x);
  if (ub >= ue) return;

  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)p.nstage * p.stage_bytes);
  uint64_t* empty = full + p.nstage;
  float* red = reinterpret_cast<float*>(empty + p.nstage);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 2 * kNW * kRedWarp);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.nstage; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], p.aw);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kNW) {
    // ---------------- producer: one thread issues the bulk copies
    if (lane == 0) {
      const uint32_t row_bytes = p.K / 2;
      const uint32_t scale_bytes = kRows * (p.K / p.G) * 2;
      int it = 0;
      for (int u = ub; u < ue; ++u) {
        const Unit un = resolve_unit<MODE>(p, u, n_act, units_per_exp);
        if (!un.ok || un.host) continue;
        const int s = it % p.nstage;
        const uint32_t par = ((it / p.nstage) & 1) ^ 1;
        if (!mbar_wait_bounded(&empty[s], par, abort_flag, p.status)) break;
        uint8_t* dst = stages + (size_t)s * p.stage_bytes;
        mbar_arrive_expect_tx(&full[s], kRows * row_bytes + scale_bytes);
        for (int r = 0; r < kRows; ++r) bulk_copy_g2s(dst + r * p.pitch, un.w + (size_t)r * row_bytes, row_bytes, &full[s]);
        bulk_copy_g2s(dst + kRows * p.pitch, un.s, scale_bytes, &full[s]);
        ++it;
      }
      // Every issued copy must land before the CTA exits (also after an abort).
      const int first = it > p.nstage ? it - p.nstage : 0;
      for (int j = first; j < it; ++j)
        mbar_wait_bounded(&full[j % p.nstage], (j / p.nstage) & 1, nullptr, p.status);
    }
    return;
  }

  // ---------------- consumers
  const int g = lane >> 2, t = lane & 3;
  const int tid = threadIdx.x;
  const bool working = warp < p.aw;
  const int c0 = warp * CPW;
  uint32_t bfr[CPW][NB];
  if constexpr (MODE == 0) {
    if (working) load_x_frags<CPW>(p, c0, g, t, bfr);
  }
  int cur_a = -1, myq = -1, it = 0, buf = 0;
  for (int u = ub; u < ue; ++u) {
    const Unit un = resolve_unit<MODE>(p, u, n_act, units_per_exp);
    if (!un.ok) {
      if (tid == 0) set_status(p.status, QRE_DEV_NULL_SLOT);
      continue;
    }
    if (un.a != cur_a) {
      cur_a = un.a;
      if constexpr (MODE == 1) {
        if (working) load_h_frags<CPW>(p, un.a, c0, g, t, bfr);
        if (tid < kRows * kTok) myq = output_row(p, un, n_act, tid / kRows);
      }
    }
    if (working) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (!un.host) {
        const int s = it % p.nstage;
        const bool have = mbar_wait_bounded(&full[s], (it / p.nstage) & 1, abort_flag, p.status);
        const uint32_t wb = smem_addr(stages + (size_t)s * p.stage_bytes);
        if (have) unit_dot<CPW, NB, true>(wb, p.pitch, wb + kRows * p.pitch, p.K / p.G, c0, p.gc, g, t, bfr, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      } else {
        unit_dot<CPW, NB, false>(reinterpret_cast<uintptr_t>(un.w), p.K / 2, reinterpret_cast<uintptr_t>(un.s),
                                 p.K / p.G, c0, p.gc, g, t, bfr, acc);
      }
      float* rw = red + (size_t)(buf * kNW + warp) * kRedWarp;
      rw[(2 * t) * kRedStride + g] = acc[0];
      rw[(2 * t + 1) * kRedStride + g] = acc[1];
      rw[(2 * t) * kRedStride + g + 8] = acc[2];
      rw[(2 * t + 1) * kRedStride + g + 8] = acc[3];
    }
    if (!un.host) ++it;
    named_barrier_sync(1, kNW * 32);
    if (tid < kRows * kTok) {
      const int n = tid / kRows, r = tid % kRows;
      float v = 0.f;
      for (int w = 0; w < p.aw; ++w) v += red[(size_t)(buf * kNW + w) * kRedWarp + n * kRedStride + r];
      if (MODE == 0) {
        p.gu[((size_t)un.a * kTok + n) * (2 * p.I) + un.r0 + r] = v;
      } else if (myq >= 0) {
        p.expert_out[(size_t)myq * p.H + un.r0 + r] = v;
      }
    }
    buf ^= 1;
  }
}

struct Plan {
  int cpw = 0, aw = 0, gc = 0, pitch = 0, stage_bytes = 0, nstage = 0;
  size_t smem = 0;
  bool ok = false;
};

Plan make_plan(int K, int G, int smem_budget) {
  Plan pl;
  const int nchunks = K / 32;
  pl.gc = G / 32;
  for (int c : {1, 2, 4, 8}) {
    if (c < pl.gc || c % pl.gc || nchunks % c || nchunks / c > kNW) continue;
    pl.cpw = c;
    break;
  }
  if (!pl.cpw) return pl;
  pl.aw = nchunks / pl.cpw;
  pl.pitch = ((K / 2 + 127) / 128) * 128 + 16;
  pl.stage_bytes = kRows * pl.pitch + kRows * (K / G) * 2;
  pl.stage_bytes = (pl.stage_bytes + 127) / 128 * 128;
  const int fixed = 2 * kNW * kRedWarp * 4 + 16;
  int ns = (smem_budget - fixed) / (pl.stage_bytes + 16);
  if (ns > 8) ns = 8;
  if (ns < 2) return pl;
  pl.nstage = ns;
  pl.smem = (size_t)ns * pl.stage_bytes + (size_t)ns * 16 + fixed;
  pl.ok = true;
  return pl;
}

template <int MODE>
cudaError_t launch_mode(const FfnParams& base, const Plan& pl, int grid, cudaStream_t stream) {
  FfnParams p = base;
  p.gc = pl.gc;
  p.aw = pl.aw;
  p.pitch = pl.pitch;
  p.stage_bytes = pl.stage_bytes;
  p.nstage = pl.nstage;
  void (*kern)(const FfnParams) = nullptr;
  switch (pl.cpw) {
    case 1: kern = ffn_decode_kernel<MODE, 1>; break;
    case 2: kern = ffn_decode_kernel<MODE, 2>; break;
    case 4: kern = ffn_decode_kernel<MODE, 4>; break;
    case 8: kern = ffn_decode_kernel<MODE, 8>; break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(kern), (int)pl.smem);
  if (err != cudaSuccess) return err;
  kern<<<grid, kThreads, pl.smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool ffn_decode_supported(const qre_layer_shape& s) {
  const int budget = device_max_smem_optin();
  return make_plan(s.hidden, s.group, budget).ok && make_plan(s.inter, s.group, budget).ok;
}

size_t ffn_ws_bytes(const qre_layer_shape& s, int T) {
  const long long pk = (long long)T * s.top_k;
  const long long amax = pk < s.n_experts ? pk : s.n_experts;
  return (size_t)(amax + 1) * kTok * 2 * s.inter * sizeof(float);
}

cudaError_t launch_ffn_decode(const qre_layer_shape& s, int T, const uint16_t* x, const qre_slot* slots,
                              const int32_t* offsets, const int32_t* perm, const int32_t* active,
                              const int32_t* n_active, float* expert_out, void* ws, int* status,
                              cudaStream_t stream) {
  const int budget = device_max_smem_optin();
  const Plan gu_plan = make_plan(s.hidden, s.group, budget);
  const Plan dn_plan = make_plan(s.inter, s.group, budget);
  if (!gu_plan.ok || !dn_plan.ok) return cudaErrorInvalidValue;
  FfnParams p{};
  p.H = s.hidden;
  p.I = s.inter;
  p.E = s.n_experts;
  p.k = s.top_k;
  p.G = s.group;
  p.T = T;
  p.x = x;
  p.slots = slots;
  p.offsets = offsets;
  p.perm = perm;
  p.active = active;
  p.n_active = n_active;
  p.gu = static_cast<float*>(ws);
  p.expert_out = expert_out;
  p.status = status;
  const long long pk = (long long)T * s.top_k;
  const int amax = (int)(pk < s.n_experts ? pk : s.n_experts);
  p.amax = amax;
  const int sms = device_sm_count();

  p.K = s.hidden;
  p.n_out = 2 * s.inter;
  long long units = (long long)(amax + 1) * (p.n_out / kRows);
  int grid = (int)(units < sms ? units : sms);
  cudaError_t err = launch_mode<0>(p, gu_plan, grid, stream);
  if (err != cudaSuccess) return err;

  p.K = s.inter;
  p.n_out = s.hidden;
  units = (long long)(amax + 1) * (p.n_out / kRows);
  grid = (int)(units < sms ? units : sms);
  return launch_mode<1>(p, dn_plan, grid, stream);
}

}  // namespace qre
