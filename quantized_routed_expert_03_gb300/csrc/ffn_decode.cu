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
//   * A unit is 32 consecutive output rows of one expert's matrix (for gate/up,
//     one block of 16 gate rows and the matching 16 up rows) over the full
//     reduction length K, staged in two K halves ("parts").
//     Units of all active experts and the shared expert are split into equal
//     contiguous ranges, one per CTA; one CTA per SM (persistent).
//   * A producer warp streams each unit from HBM into a ring of shared-memory
//     stages with 1-D bulk (TMA) copies, one row per lane, so a stage's copies
//     leave in one warp-wide instruction (one thread issuing them one by one was
//     measured to cap the stream near 2 TB/s), completing on an mbarrier.  Rows land at a pitch of 16 mod 128 bytes so
//     the consumers' 32-bit loads are free of bank conflicts.  Units of host-resident experts (slot tier 1) skip
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
//   * Per unit, the 16 warps' partial sums go to one of two shared buffers and a
//     reducer warp adds them in fixed warp order (deterministic) while the
//     consumers continue with the next unit; the result goes to the gate/up
//     workspace (gate/up kernel) or to the expert's output rows (down kernel).
// The down kernel computes h = silu(g) * u from the gate/up workspace while it
// loads its activation operand, and splits h into an fp16 high part and an fp16
// remainder so that its products stay accurate to about fp32.
#include "common.cuh"
#include "internal.h"

namespace qre {
namespace {

constexpr int kNW = 16;                    // consumer warps
constexpr int kProducerWarp = kNW;
constexpr int kReducerWarp = kNW + 1;
constexpr int kThreads = (kNW + 2) * 32;   // + one producer warp + one reducer warp
constexpr int kTiles = 2;                  // MMA M tiles (16 rows each) per unit
constexpr int kRows = 16 * kTiles;         // rows per unit: one gate block + one up block
static_assert(kRows == 32, "the producer issues one row copy per lane");
constexpr int kTok = kDecodeMaxTokens;     // MMA N
constexpr int kRedStride = 20;             // floats between token columns of a partial
constexpr int kRedTile = kTok * kRedStride;
constexpr int kRedWarp = kTiles * kRedTile;
constexpr int kMaxGroups = kDecodeMaxTokens * 16 + 1;   // T*k active experts + the shared one

// One active expert (or the shared expert) as this kernel sees it; built once
// per CTA in shared memory so that no unit waits on dependent global loads.
struct Group {
  const uint8_t* w;    // packed matrix of this kernel (gate/up or down)
  const uint16_t* s;   // its scales
  int e;               // expert id (E = shared)
  int flags;           // bit 0: usable, bit 1: host-resident (read with direct loads)
  int outq[kTok];      // down kernel: expert_out row of token n, or -1
};

struct FfnParams {
  int H, I, E, k, G, T;
  int K;            // reduction length: H (gate/up) or I (down)
  int n_out;        // rows per expert: 2I (gate/up) or H (down)
  int gc;           // 32-element chunks per quantization group
  int aw;           // working consumer warps
  int nparts;       // K is staged in this many parts; warp w reads part w / (aw / nparts)
  int pitch;        // shared-memory row pitch in bytes (16 mod 128)
  int part_bytes;   // bytes of one row in one part
  int stage_bytes;  // rows of one part + the unit's scales
  int nstage;
  int amax;         // largest possible number of active experts, min(E, T*k)
  const uint16_t* x;
  const qre_slot* slots;
  const int32_t* offsets;
  const int32_t* perm;
  const int32_t* active;
  const int32_t* n_active;
  uint16_t* hfrag;    // [(amax+1)][I/32][32 lanes][16 halves]: h as MMA B fragments
  float* expert_out;  // [T*k + T][H]
  int* status;
};

__device__ __forceinline__ uint32_t ldg_u32(const void* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}
__device__ __forceinline__ float ldg_half_as_float(const uint16_t* p) {
  return __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(p))));
}

// Dot products of one unit's 32 rows (two 16-row MMA tiles) with the warp's K
// range.  SMEM: wbase/sbase point into the shared-memory stage (the staged part
// and the unit's scales); otherwise global addresses of row 0 and its scales.
// cbase is subtracted from the global chunk index to address the staged part.
// Each tile accumulates into kAcc independent fragments (chunk cl goes to
// cl % kAcc) so consecutive MMAs do not wait on each other; they are summed
// when a quantization group ends.
constexpr int kAcc = 2;
template <int CPW, int NB, bool SMEM>
__device__ __forceinline__ void unit_dot(const uint8_t* wbase, uint32_t wbase_s, int wpitch, const uint16_t* sbase,
                                         uint32_t sbase_s, int s_stride, int c0, int cbase, int gc, int g, int t,
                                         const uint32_t (&bfr)[CPW][NB], float (&acc)[kTiles][4]) {
  float d[kTiles][kAcc][4];
#pragma unroll
  for (int i = 0; i < kTiles; ++i)
#pragma unroll
    for (int j = 0; j < kAcc; ++j) d[i][j][0] = d[i][j][1] = d[i][j][2] = d[i][j][3] = 0.f;
  // Loads are issued one quantization group (GCMAX chunks at most) ahead of
  // their use, so they overlap the previous group's MMAs.
  constexpr int GCMAX = CPW < 4 ? CPW : 4;
  uint32_t wv[GCMAX][kTiles][2];
#pragma unroll
  for (int cl = 0; cl < CPW; ++cl) {
    const int c = c0 + cl;
    const int j = cl % kAcc;
    if (cl % GCMAX == 0) {
#pragma unroll
      for (int u = 0; u < GCMAX; ++u) {
        const int col = (c + u - cbase) * 16 + t * 4;
#pragma unroll
        for (int i = 0; i < kTiles; ++i) {
          if constexpr (SMEM) {
            const uint32_t a_lo = wbase_s + (uint32_t)((16 * i + g) * wpitch + col);
            wv[u][i][0] = lds32(a_lo);
            wv[u][i][1] = lds32(a_lo + 8 * wpitch);
          } else {
            const uint8_t* r_lo = wbase + (size_t)(16 * i + g) * wpitch + col;
            wv[u][i][0] = ldg_u32(r_lo);
            wv[u][i][1] = ldg_u32(r_lo + (size_t)8 * wpitch);
          }
        }
      }
    }
    const int u = cl % GCMAX;
#pragma unroll
    for (int i = 0; i < kTiles; ++i) {
      uint32_t pl[4], ph[4];
      decode_nibbles(wv[u][i][0], pl);
      decode_nibbles(wv[u][i][1], ph);
      mma_f16_16816(d[i][j], pl[0], ph[0], pl[1], ph[1], bfr[cl][0], bfr[cl][1]);
      if constexpr (NB == 8) mma_f16_16816(d[i][j], pl[0], ph[0], pl[1], ph[1], bfr[cl][4], bfr[cl][5]);
      mma_f16_16816(d[i][j], pl[2], ph[2], pl[3], ph[3], bfr[cl][2], bfr[cl][3]);
      if constexpr (NB == 8) mma_f16_16816(d[i][j], pl[2], ph[2], pl[3], ph[3], bfr[cl][6], bfr[cl][7]);
    }
    if (((cl + 1) & (gc - 1)) == 0) {  // end of a quantization group
      const int grp = c / gc;
#pragma unroll
      for (int i = 0; i < kTiles; ++i) {
        const size_t e_lo = (size_t)(16 * i + g) * s_stride + grp;
        const size_t e_hi = e_lo + (size_t)8 * s_stride;
        float slo, shi;
        if constexpr (SMEM) {
          slo = __half2float(__ushort_as_half(lds16(sbase_s + (uint32_t)(e_lo * 2))));
          shi = __half2float(__ushort_as_half(lds16(sbase_s + (uint32_t)(e_hi * 2))));
        } else {
          slo = ldg_half_as_float(sbase + e_lo);
          shi = ldg_half_as_float(sbase + e_hi);
        }
        float v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          v[q] = d[i][0][q];
#pragma unroll
          for (int jj = 1; jj < kAcc; ++jj) v[q] += d[i][jj][q];
        }
        acc[i][0] = fmaf(slo, v[0], acc[i][0]);
        acc[i][1] = fmaf(slo, v[1], acc[i][1]);
        acc[i][2] = fmaf(shi, v[2], acc[i][2]);
        acc[i][3] = fmaf(shi, v[3], acc[i][3]);
#pragma unroll
        for (int jj = 0; jj < kAcc; ++jj) d[i][jj][0] = d[i][jj][1] = d[i][jj][2] = d[i][jj][3] = 0.f;
      }
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

// Activation operand for down: the fragments the gate/up kernel stored.
template <int CPW>
__device__ __forceinline__ void load_h_frags(const FfnParams& p, int a, int c0, int lane, uint32_t (&bfr)[CPW][8]) {
  const int nch = p.I / 32;
#pragma unroll
  for (int cl = 0; cl < CPW; ++cl) {
    const uint4* src = reinterpret_cast<const uint4*>(p.hfrag + (((size_t)a * nch + c0 + cl) * 32 + lane) * 16);
    const uint4 v0 = src[0], v1 = src[1];
    bfr[cl][0] = v0.x; bfr[cl][1] = v0.y; bfr[cl][2] = v0.z; bfr[cl][3] = v0.w;
    bfr[cl][4] = v1.x; bfr[cl][5] = v1.y; bfr[cl][6] = v1.z; bfr[cl][7] = v1.w;
  }
}

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

template <int MODE, int CPW>
__global__ void __launch_bounds__(kThreads, 1) ffn_decode_kernel(const FfnParams p) {
  constexpr int NB = MODE == 0 ? 4 : 8;
  extern __shared__ __align__(128) uint8_t smem[];
  int n_act = *p.n_active;
  n_act = n_act < 0 ? 0 : (n_act > p.amax ? p.amax : n_act);
  const int ngroups = n_act + 1;
  const int upe = p.n_out / kRows;                 // units per expert
  const int U = ngroups * upe;
  const int ub = (int)((long long)blockIdx.x * U / gridDim.x);
  const int ue = (int)((long long)(blockIdx.x + 1) * U / gridDim.x);
  if (ub >= ue) return;

  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)p.nstage * p.stage_bytes);
  uint64_t* empty = full + p.nstage;
  uint64_t* red_full = empty + p.nstage;    // [2] partials of a unit written by the consumer warps
  uint64_t* red_empty = red_full + 2;       // [2] the reducer has read them
  float* red = reinterpret_cast<float*>(red_empty + 2);
  Group* groups = reinterpret_cast<Group*>(red + 2 * kNW * kRedWarp);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(groups + kMaxGroups);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  // Only the groups this CTA's units touch are needed; filling all is cheap.
  for (int a = tid; a < ngroups; a += blockDim.x) {
    Group gr;
    gr.e = a < n_act ? __ldg(p.active + a) : p.E;
    gr.w = nullptr;
    gr.s = nullptr;
    gr.flags = 0;
    if (gr.e >= 0 && gr.e <= p.E) {
      const qre_slot* sl = p.slots + gr.e;
      gr.w = MODE == 0 ? sl->w_gate_up : sl->w_down;
      gr.s = MODE == 0 ? sl->s_gate_up : sl->s_down;
      const bool ok = gr.w && gr.s &&
                      ((reinterpret_cast<uintptr_t>(gr.w) | reinterpret_cast<uintptr_t>(gr.s)) & 15) == 0;
      gr.flags = (ok ? 1 : 0) | (sl->tier != 0 ? 2 : 0);
    }
    Group& dst = groups[a];
    dst.w = gr.w;
    dst.s = gr.s;
    dst.e = gr.e;
    dst.flags = gr.flags;
#pragma unroll
    for (int n = 0; n < kTok; ++n) dst.outq[n] = (MODE == 1 && a == n_act && n < p.T) ? p.T * p.k + n : -1;
    if (MODE == 1 && a < n_act && (gr.flags & 1)) {
      const int lo = __ldg(p.offsets + gr.e), hi = __ldg(p.offsets + gr.e + 1);
      for (int q = lo; q < hi && q < lo + kTok; ++q) {
        const int tk = __ldg(p.perm + q) / p.k;
        if (tk >= 0 && tk < kTok) dst.outq[tk] = q;
      }
    }
  }
  if (tid == 0) {
    for (int s = 0; s < p.nstage; ++s) {
      mbar_init(&full[s], 1);                  // the producer's expect_tx arrival
      mbar_init(&empty[s], p.aw / p.nparts);   // one arrival per consumer warp of the part
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&red_full[b], p.aw);
      mbar_init(&red_empty[b], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const int part_chunks = (p.K / 32) / p.nparts;
  const uint32_t scale_bytes = kRows * (p.K / p.G) * 2;

  if (warp == kProducerWarp) {
    // ---------------- producer: per part-stage, lane r issues the 1-D bulk (TMA)
    // copy of row r and lane 0 the scales, so the 33 copies of a stage leave in
    // one warp-wide instruction instead of 33 serial ones from a single thread.
    const size_t row_bytes = p.K / 2;
    int it = 0;
    for (int u = ub; u < ue; ++u) {
      const int a = u / upe, r0 = (u - a * upe) * kRows;
      const Group& gr = groups[a];
      if ((gr.flags & 3) != 1) continue;   // skipped or host-resident
      bool stop = false;
      for (int part = 0; part < p.nparts; ++part, ++it) {
        const int s = it % p.nstage;
        int ok = 1;
        if (lane == 0) {
          ok = mbar_wait_bounded(&empty[s], ((it / p.nstage) & 1) ^ 1, abort_flag, p.status) ? 1 : 0;
          if (ok) mbar_arrive_expect_tx(&full[s], kRows * p.part_bytes + scale_bytes);
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {   // warp-uniform
          stop = true;
          break;
        }
        uint8_t* dst = stages + (size_t)s * p.stage_bytes;
        const uint8_t* src = gr.w + (size_t)r0 * row_bytes + (size_t)part * p.part_bytes;
        bulk_copy_g2s(dst + lane * p.pitch, src + lane * row_bytes, p.part_bytes, &full[s]);   // kRows == 32
        if (lane == 0)
          bulk_copy_g2s(dst + kRows * p.pitch, gr.s + (size_t)r0 * (p.K / p.G), scale_bytes, &full[s]);
      }
      if (stop) break;
    }
    // Every issued copy must land before the CTA exits (also after an abort).
    if (lane == 0) {
      const int first = it > p.nstage ? it - p.nstage : 0;
      for (int j = first; j < it; ++j)
        mbar_wait_bounded(&full[j % p.nstage], (j / p.nstage) & 1, nullptr, p.status);
    }
    return;
  }

  if (warp == kReducerWarp) {
    // ---------------- reducer: adds the consumer warps' partials of each unit in
    // fixed warp order (deterministic) while the consumers go on with the next
    // unit; two partial buffers.
    int ru = 0;
    for (int u = ub; u < ue; ++u) {
      const int a = u / upe, r0 = (u - a * upe) * kRows;
      const Group& gr = groups[a];
      if (!(gr.flags & 1)) continue;
      const int buf = ru & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(&red_full[buf], (ru >> 1) & 1, abort_flag, p.status) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      const float* rb = red + (size_t)buf * kNW * kRedWarp;
      if (ok) {
        if constexpr (MODE == 0) {
          // gate row r and up row r of token n -> h = silu(g) * u, stored as the
          // down kernel's B fragment: feature f = r0/2 + r of chunk f/32, lane
          // 4n + (f%32)/8, pair (f%8)%4, half (f%8)/4; high part then remainder.
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int o = lane + 32 * j, n = o >> 4, r = o & 15;
            float gs = 0.f, us = 0.f;
#pragma unroll
            for (int w = 0; w < kNW; ++w) {
              if (w < p.aw) {
                gs += rb[w * kRedWarp + n * kRedStride + r];
                us += rb[w * kRedWarp + kRedTile + n * kRedStride + r];
              }
            }
            const float h = silu_f32(gs) * us;
            const __half hh = __float2half_rn(h);
            const __half hl = __float2half_rn(h - __half2float(hh));
            const int f = r0 / 2 + r;
            const int c = f >> 5, tt = (f & 31) >> 3, i8 = f & 7;
            const size_t base = (((size_t)a * (p.I / 32) + c) * 32 + (4 * n + tt)) * 16;
            p.hfrag[base + (i8 & 3) * 2 + (i8 >> 2)] = __half_as_ushort(hh);
            p.hfrag[base + (4 + (i8 & 3)) * 2 + (i8 >> 2)] = __half_as_ushort(hl);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int o = lane + 32 * j, i = o >> 7, n = (o >> 4) & 7, r = o & 15;
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < kNW; ++w)
              if (w < p.aw) v += rb[w * kRedWarp + i * kRedTile + n * kRedStride + r];
            const int q = gr.outq[n];
            if (q >= 0) p.expert_out[(size_t)q * p.H + r0 + 16 * i + r] = v;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_empty[buf]);
      ++ru;
    }
    return;
  }

  // ---------------- consumers
  const int g = lane >> 2, t = lane & 3;
  if (warp >= p.aw) return;                 // no K range for this warp (small shapes)
  const int c0 = warp * CPW;
  const int wpart = warp / (p.aw / p.nparts);
  uint32_t bfr[CPW][NB];
  if constexpr (MODE == 0) load_x_frags<CPW>(p, c0, g, t, bfr);
  int cur_a = -1, units0 = 0, ru = 0;
  for (int u = ub; u < ue; ++u) {
    const int a = u / upe, r0 = (u - a * upe) * kRows;
    const Group& gr = groups[a];
    if (!(gr.flags & 1)) {
      if (threadIdx.x == 0) set_status(p.status, QRE_DEV_NULL_SLOT);
      continue;
    }
    const bool host = gr.flags & 2;
    if constexpr (MODE == 1) {
      if (a != cur_a) load_h_frags<CPW>(p, a, c0, lane, bfr);
    }
    cur_a = a;
    float acc[kTiles][4];
#pragma unroll
    for (int i = 0; i < kTiles; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    if (!host) {
      const int it = units0 * p.nparts + wpart;
      const int s = it % p.nstage;
      const bool have = mbar_wait_bounded(&full[s], (it / p.nstage) & 1, abort_flag, p.status);
      const uint32_t wb = after_wait(smem_addr(stages + (size_t)s * p.stage_bytes));
      if (have)
        unit_dot<CPW, NB, true>(nullptr, wb, p.pitch, nullptr, wb + kRows * p.pitch, p.K / p.G, c0,
                                wpart * part_chunks, p.gc, g, t, bfr, acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      ++units0;
    } else {
      unit_dot<CPW, NB, false>(gr.w + (size_t)r0 * (p.K / 2), 0, p.K / 2, gr.s + (size_t)r0 * (p.K / p.G), 0,
                               p.K / p.G, c0, 0, p.gc, g, t, bfr, acc);
    }
    const int buf = ru & 1;
    int ok = 1;
    if (lane == 0) ok = mbar_wait_bounded(&red_empty[buf], ((ru >> 1) & 1) ^ 1, abort_flag, p.status) ? 1 : 0;
    __syncwarp();
    (void)ok;
    float* rw = red + (size_t)(buf * kNW + warp) * kRedWarp;
#pragma unroll
    for (int i = 0; i < kTiles; ++i) {
      rw[i * kRedTile + (2 * t) * kRedStride + g] = acc[i][0];
      rw[i * kRedTile + (2 * t + 1) * kRedStride + g] = acc[i][1];
      rw[i * kRedTile + (2 * t) * kRedStride + g + 8] = acc[i][2];
      rw[i * kRedTile + (2 * t + 1) * kRedStride + g + 8] = acc[i][3];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&red_full[buf]);
    ++ru;
  }
}

struct Plan {
  int cpw = 0, aw = 0, gc = 0, nparts = 1, pitch = 0, part_bytes = 0, stage_bytes = 0, nstage = 0;
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
  pl.nparts = (pl.aw % 2 == 0) ? 2 : 1;
  pl.part_bytes = K / 2 / pl.nparts;
  pl.pitch = ((pl.part_bytes + 127) / 128) * 128 + 16;
  pl.stage_bytes = kRows * pl.pitch + kRows * (K / G) * 2;
  pl.stage_bytes = (pl.stage_bytes + 127) / 128 * 128;
  const int fixed = 4 * 8 + 2 * kNW * kRedWarp * 4 + kMaxGroups * (int)sizeof(Group) + 16;
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
  p.nparts = pl.nparts;
  p.pitch = pl.pitch;
  p.part_bytes = pl.part_bytes;
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
  return (size_t)(amax + 1) * (s.inter / 32) * 32 * 16 * sizeof(uint16_t);
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
  p.hfrag = static_cast<uint16_t*>(ws);
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
