// ffn_decode.cu -- bandwidth-bound fused dequant + SwiGLU expert FFN for T <= 8.
//
// The decode step of a routed MoE layer reads every byte of the union of the
// experts its tokens picked, plus the shared expert, once (glm53-flash-offload
// README, "Batched decode": streams share the per-layer expert union).  The work
// is a matrix-vector product per expert over 4-bit weights and the bound is HBM
// bandwidth, so the packed weights must stream at full rate while everything
// else stays under that.
//
// Two kernels share the structure below: ffn_e4m3_kernel for group 128 (every
// full-size configuration: weights as FP8 E4M3 codes, 128-element stages, see
// the comment above it) and ffn_decode_kernel for groups 32 and 64 (weights as
// fp16 codes, 64-element stages).  Both launch as programmatic dependents
// (launch_dependent): gate/up waits for the dispatch, down's CTAs take the SMs
// gate/up CTAs leave and wait for the gate/up grid only before reading h.
//
// Layout of the work (5th-generation tensor cores, weights in tensor memory)
//   * A unit is 128 consecutive rows of one expert's matrix (UMMA M = 128; for
//     gate/up four blocks of 16 gate rows, each followed by its 16 up rows).
//     Units of all active experts and the shared expert are split into equal
//     contiguous ranges, one per CTA; one CTA per SM.
//   * The four warpgroups of a CTA split the reduction length K.  Thread r of a
//     warpgroup owns weight row r of the unit and tensor-memory lane r.  The
//     packed weights are stored in 4 KB chunks of 128 rows x 64 reduction
//     elements, so each warp's 16-byte loads cover 512 contiguous bytes; they
//     run a few stages ahead, across unit boundaries (FP8 kernel: through a
//     cp.async ring in shared memory; host-resident experts are read the same
//     way with direct loads, zero-copy).  Each thread decodes its nibbles into
//     exact codes and writes them into its lane with tcgen05.st.
//   * One tcgen05.mma (A from tensor memory, B from shared memory) is cheap for
//     the tensor core but takes a warp on the order of a hundred cycles to
//     issue, while issues from different warps overlap.  So every warp issues:
//     the stages of a warpgroup are issued in turn by its four warps, one stage
//     late, once all four warps have arrived on the stage's mbarrier, and
//     complete on one commit per stage.
//   * B holds the tokens (T <= 8) in shared memory, 128-byte swizzled: fp16
//     kernel, row 2n the fp16 high part of token n and row 2n + 1 the remainder
//     (x - high); FP8 kernel, E4M3 terms per token and group.  The weights are
//     exact codes, so the only rounding is that of the activations' split and
//     the fp32 accumulation.
//   * Every quantization group accumulates into its own buffer; a few stages
//     later the owning threads read it back (tcgen05.ld), combine the columns
//     of each token and apply the group's fp16 scale in fp32.
//   * The warpgroups' partial rows are added in fixed order (deterministic), one
//     unit after they were handed over: gate/up pairs each gate row with its up
//     row (16 lanes apart, a shuffle) and stores h for the down kernel; down
//     writes the expert's output rows.
//   * fp16 kernel: inside every group of 8 reduction elements the tokens and h
//     are stored in the order the nibble decode yields weight pairs
//     (0,4,1,5,2,6,3,7), which leaves every dot product unchanged.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

#include <cuda_fp8.h>

namespace qre {
namespace {

constexpr int kWG = 4;                    // warpgroups (K splits) per CTA
constexpr int kThreads = kWG * 128;
constexpr int BM = 128;                   // weight rows per unit (UMMA M, one TMEM lane each)
constexpr int BN = 16;                    // UMMA N: token high parts, then remainders
constexpr int SK = 64;                    // reduction elements per stage (32 TMEM columns)
constexpr int kTok = kDecodeMaxTokens;    // tokens
constexpr int kColsPerWG = 128;           // TMEM columns per warpgroup: NA A buffers of 32, then the D buffers
constexpr int kMaxGroups = kDecodeMaxTokens * 16 + 1;   // T*k active experts + the shared one
constexpr int kChunk = BM * SK / 2;       // bytes of one packed 128 x 64 chunk

struct Group {
  const uint8_t* w;    // packed matrix of this kernel (gate/up or down)
  const uint16_t* s;   // its scales
  int e;               // expert id (E = shared)
  int flags;           // bit 0: usable
  int outq[kTok];      // down kernel: expert_out row of token n, or -1
};

struct FfnParams {
  int H, I, E, k, G, T;
  int K;            // reduction length: H (gate/up) or I (down)
  int n_out;        // rows per expert: 2I (gate/up) or H (down)
  int kq;           // warpgroups sharing K (1, 2 or 4)
  int lgG;          // log2 G
  int nB;           // B buffers in shared memory (down kernel: experts resident at once)
  int amax;         // largest possible number of active experts, min(E, T*k)
  int part;         // groups of this launch: 0 routed + shared, 1 routed only, 2 shared only
  int host_cost;    // > 1: the cost-cut instance, a host-mapped unit counted as this many (qre_set_host_unit_cost)
  const uint16_t* x;
  const qre_slot* slots;
  const int32_t* offsets;
  const int32_t* perm;
  const int32_t* active;
  const int32_t* n_active;
  __half* hbuf;       // [(amax+1)][2*kTok][I]: row 2n = h high part of token n, 2n+1 its remainder
  float* expert_out;  // [T*k + T][H]
  int* status;
  uint64_t wait_ns;   // limit of the pipeline waits
  uint64_t stall_ns;  // test hook: warp 1 of the CTA that owns unit 0 delays its first stage's signal
};

struct Layout {
  int b_off, red_off, bar_off, grp_off, misc_off;
  size_t bytes;
};

__host__ __device__ inline Layout make_layout(int K, int nB, int TT) {
  Layout L;
  L.b_off = 0;                                          // nB x (BN x K fp16, swizzled; 1024-aligned)
  L.red_off = L.b_off + nB * K * BN * 2;                // 2 x kWG x BM x TT fp32
  L.bar_off = L.red_off + 2 * kWG * BM * TT * 4;        // a_full[kWG][3], done[kWG][3], red_full[2], red_empty[2],
                                                        // drain[kThreads / 32]
  L.grp_off = L.bar_off + (kWG * 6 + 4 + kThreads / 32) * 8;
  L.misc_off = L.grp_off + kMaxGroups * (int)sizeof(Group);
  L.bytes = (size_t)L.misc_off + 16 + 1024;             // + alignment slack
  return L;
}

// Byte offset of (row n, logical reduction index l) in a swizzled B operand.
__device__ __forceinline__ uint32_t b_offset(int n, int l) {
  const int byte = (l & 63) * 2;
  return (uint32_t)((l >> 6) * (BN * 128) + (n >> 3) * 1024 + (n & 7) * 128 + ((((byte >> 4) ^ (n & 7))) << 4) +
                    (byte & 15));
}

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

// fp16 high part and remainder of v.
__device__ __forceinline__ void split_half(float v, __half& hi, __half& lo) {
  hi = __float2half_rn(v);
  lo = __float2half_rn(v - __half2float(hi));
}

// h of group a (rows 0 .. 2T-1: high part and remainder of each token) into B buffer `dst`.
__device__ __forceinline__ void load_h(uint8_t* dst, const __half* hbuf, int a, int I, int T) {
  const __half* hb = hbuf + (size_t)a * 2 * kTok * I;
  for (int i = threadIdx.x; i < 2 * T * (I / 8); i += blockDim.x) {
    const int row = i / (I / 8), g8 = i - row * (I / 8);
    *reinterpret_cast<uint4*>(dst + b_offset(row, 8 * g8)) =
        *reinterpret_cast<const uint4*>(hb + (size_t)row * I + 8 * g8);
  }
}

// A unit's epilogue (local unit v of the CTA's range starting at unit ub).
// TT = 8: thread (wg, r) finishes row r for tokens 2wg and 2wg + 1; TT = 1:
// warpgroup 0 finishes token 0.  Gate/up: h = silu(gate) * up of each row pair
// (gate row in lanes 0-15, its up row 16 lanes above) into hbuf, for the fp16
// down kernel as fp16 high part and remainder (rows 2n, 2n + 1 of the group),
// for the FP8 one (H32) as fp32 (row n) with each 8-feature block in the FP8
// B operand's order (feature 2i + h at 4h + i); down: the expert's output
// rows.  Whole warps call it; every thread of the CTA arrives on red_empty.
template <int MODE, int TT, bool H32 = false>
__device__ __noinline__ void finish_unit(int v, int ub, int upe, const Group* groups, const float* red,
                                         uint64_t* red_full, uint64_t* red_empty, int kq, int T, int I, int H,
                                         __half* hbuf, float* expert_out, volatile int* abort_flag, int* status,
                                         uint64_t wait_ns, float own0 = 0.f, float own1 = 0.f) {
  const int tid = threadIdx.x, lane = tid & 31, wg = tid >> 7, r = tid & 127;
  const int u = ub + v, a = u / upe, m0 = (u - a * upe) * BM;
  const Group& gr = groups[a];
  mbar_wait_bounded(&red_full[v & 1], (v >> 1) & 1, abort_flag, status, wait_ns);
  constexpr int NT = TT == 1 ? 1 : 2;   // tokens per thread
  const int n0 = TT == 1 ? 0 : 2 * wg;
  if ((TT > 1 || wg == 0) && (gr.flags & 1)) {
    float vv[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) vv[t] = 0.f;
    // FP8 down kernel, eight tokens: warpgroup w stores every token but its own
    // two (2w, 2w + 1), which it passes in own0/own1; same terms, same order
    constexpr bool kOwn = H32 && MODE == 1 && TT == 8;
    constexpr int RT = kOwn ? TT - 2 : TT;
    for (int w = 0; w < kq; ++w) {
      if (kOwn && w == wg) {
        vv[0] += own0;
        vv[NT - 1] += own1;
        continue;
      }
      const float* rr = red + ((size_t)((v & 1) * kWG + w) * BM + r) * RT + (kOwn && n0 > 2 * w ? n0 - 2 : n0);
#pragma unroll
      for (int t = 0; t < NT; ++t) vv[t] += rr[t];
    }
    if constexpr (MODE == 0 && H32) {
      const int f = m0 / 2 + 16 * (r >> 5) + (r & 15);
      const int pos = (f & ~7) | ((f & 1) << 2) | ((f >> 1) & 3);
      float* hb = reinterpret_cast<float*>(hbuf) + (size_t)a * kTok * I;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float up = __shfl_down_sync(0xffffffffu, vv[t], 16);
        if ((lane & 16) == 0 && n0 + t < T) hb[(size_t)(n0 + t) * I + pos] = silu_f32(vv[t]) * up;
      }
    } else if constexpr (MODE == 0) {
      const int f = m0 / 2 + 16 * (r >> 5) + (r & 15);
      const int pos = (f & ~7) | (((f & 3) << 1) | ((f >> 2) & 1));
      __half* hb = hbuf + (size_t)a * 2 * kTok * I;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float up = __shfl_down_sync(0xffffffffu, vv[t], 16);
        if ((lane & 16) == 0 && n0 + t < T) {
          __half hh, hl;
          split_half(silu_f32(vv[t]) * up, hh, hl);
          hb[(size_t)(2 * (n0 + t)) * I + pos] = hh;
          hb[(size_t)(2 * (n0 + t) + 1) * I + pos] = hl;
        }
      }
    } else {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int q = gr.outq[n0 + t];
        if (q >= 0) expert_out[(size_t)q * H + m0 + r] = vv[t];
      }
    }
  }
  mbar_arrive(&red_empty[v & 1]);
}

// The pipeline of a warpgroup runs over the global stages g of its CTA (all
// units back to back; four stages per unrolled block, the register ring).
// Iteration g: wait for stage g - NA's MMAs (A buffer g mod NA is free again,
// the segments that ended in stage g - NA are readable); decode and store stage
// g; read back stage g - NA (after a unit's last stage the thread's partial
// sums go to the reduction buffer); publish stage g; and, on its warp's turn,
// issue stage g - 1.  MMAs from different threads are not ordered among
// themselves, so all stages of one accumulation segment are issued by the same
// warp: warp (segment mod 4).  SEG = the accumulation segment, min(G, K slice):
// 128 covers two stages (three A buffers, two D buffers), 64 one stage and 32
// half a stage (two A buffers, four D buffers).  A unit's epilogue (sum of the
// warpgroups' partials, SwiGLU or output rows) runs one unit later, so no warp
// waits for a slower one at unit boundaries; mbarriers hand the double-buffered
// reduction area over.  TT = token capacity (1 or 8): B row 2n is the fp16 high
// part of token n, row 2n + 1 its remainder, and accumulator columns 0 .. 2TT-1
// are the ones read back.
template <int MODE, int SEG, int TT>
__global__ void __launch_bounds__(kThreads, 1) ffn_decode_kernel(const FfnParams p) {
  grid_dependency_wait();   // everything the kernels before it wrote (down: h of the gate/up grid)
  grid_dependents_launch();
  constexpr int R = 4;                    // register ring depth = unroll
  constexpr int NA = SEG == 128 ? 3 : 2;  // A buffers per warpgroup
  constexpr int ND = SEG == 128 ? 2 : 4;  // D buffers per warpgroup
  constexpr int kD0 = 32 * NA;            // first D column of a warpgroup
  static_assert(32 * NA + 16 * ND <= kColsPerWG, "TMEM columns per warpgroup");
  static_assert(TT == 1 || TT == kTok, "token capacity");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const Layout L = make_layout(p.K, p.nB, TT);
  uint8_t* Bs = smem + L.b_off;
  const uint32_t b_bytes = (uint32_t)p.K * BN * 2;
  float* red = reinterpret_cast<float*>(smem + L.red_off);
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + L.bar_off);   // [kWG][3]: the 4 warps stored stage A
  uint64_t* done = a_full + kWG * 3;                                  // [kWG][3]: the stage's MMAs completed
  uint64_t* red_full = done + kWG * 3;                                // [2]: every partial of a unit written
  uint64_t* red_empty = red_full + 2;                                 // [2]: every epilogue of a unit read
  uint64_t* drain = red_empty + 2;                                    // [warps]: a warp's MMAs completed
  Group* groups = reinterpret_cast<Group*>(smem + L.grp_off);
  uint32_t* tmem_base_p = reinterpret_cast<uint32_t*>(smem + L.misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc_off + 4);

  // the possible active ids are read together with their count (one dependent
  // load less before the slot table)
  // groups: the active experts (parts 0, 1), then the shared one (parts 0, 2);
  // the shared-only launch reads no routing at all
  const int a_spec = (p.part != 2 && threadIdx.x < p.amax) ? __ldg(p.active + threadIdx.x) : p.E;
  int n_act = p.part == 2 ? 0 : *p.n_active;
  n_act = n_act < 0 ? 0 : (n_act > p.amax ? p.amax : n_act);
  const int ngroups = n_act + (p.part == 1 ? 0 : 1);
  const int upe = p.n_out / BM;
  const int U = ngroups * upe;
  const int ub = (int)((long long)blockIdx.x * U / gridDim.x);
  const int ue = (int)((long long)(blockIdx.x + 1) * U / gridDim.x);
  if (ub >= ue) return;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wg = tid >> 7, r = tid & 127, wq = warp & 3;

  // per-CTA table of the groups (expert, pointers, output rows)
  for (int a = tid; a < ngroups; a += blockDim.x) {
    const int e = a < n_act ? (a == tid ? a_spec : __ldg(p.active + a)) : p.E;
    const uint8_t* w = nullptr;
    const uint16_t* sc = nullptr;
    int flags = 0;
    if (e >= 0 && e <= p.E) {
      const qre_slot* sl = p.slots + e;
      w = MODE == 0 ? sl->w_gate_up : sl->w_down;
      sc = MODE == 0 ? sl->s_gate_up : sl->s_down;
      flags = (w && sc && ((reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(sc)) & 15) == 0) ? 1 : 0;
    }
    if (!flags && a >= ub / upe && a <= (ue - 1) / upe) set_status(p.status, QRE_DEV_NULL_SLOT);
    Group& dst = groups[a];
    dst.w = w;
    dst.s = sc;
    dst.e = e;
    dst.flags = flags;
#pragma unroll
    for (int n = 0; n < kTok; ++n) dst.outq[n] = (MODE == 1 && a == n_act && n < p.T) ? p.T * p.k + n : -1;
    if (MODE == 1 && a < n_act && flags) {
      const int lo = __ldg(p.offsets + e), hi = __ldg(p.offsets + e + 1);
      for (int q = lo; q < hi && q < lo + kTok; ++q) {
        const int tk = __ldg(p.perm + q) / p.k;
        if (tk >= 0 && tk < kTok) dst.outq[tk] = q;
      }
    }
  }
  if (tid == 0) {
    for (int i = 0; i < kWG * 3; ++i) {
      mbar_init(&a_full[i], 4);
      mbar_init(&done[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&red_full[i], 128 * p.kq);
      mbar_init(&red_empty[i], kThreads);
    }
    for (int i = 0; i < kThreads / 32; ++i) mbar_init(&drain[i], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(tmem_base_p, kWG * kColsPerWG);
    tmem_relinquish();
  }
  const int a_first = ub / upe;
  if constexpr (MODE == 0) {
    // B = tokens, row 2n the fp16 high part of token n, row 2n + 1 the remainder.
    // Rows of tokens n >= T are left as they are: they only feed accumulator
    // columns that nothing reads.
    for (int i = tid; i < p.T * (p.K / 8); i += blockDim.x) {
      const int n = i / (p.K / 8), g8 = i - n * (p.K / 8);
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)n * p.H + 8 * g8));
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
      float f[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        f[2 * j] = bf16_bits_to_float(wv[j] & 0xFFFFu);
        f[2 * j + 1] = bf16_bits_to_float(wv[j] >> 16);
      }
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {   // pair (x_j, x_{j+4})
        __half h0, l0, h1, l1;
        split_half(f[j], h0, l0);
        split_half(f[j + 4], h1, l1);
        hi[j] = h2_as_u32(__halves2half2(h0, h1));
        lo[j] = h2_as_u32(__halves2half2(l0, l1));
      }
      *reinterpret_cast<uint4*>(Bs + b_offset(2 * n, 8 * g8)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(Bs + b_offset(2 * n + 1, 8 * g8)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  } else {
    // B = h of the experts of this CTA's range (at most nB of them, by the launch)
    const int a_last = (ue - 1) / upe;
    for (int j = 0; j < p.nB && a_first + j <= a_last; ++j) load_h(Bs + j * b_bytes, p.hbuf, a_first + j, p.I, p.T);
    if (a_last - a_first >= p.nB && tid == 0) set_status(p.status, QRE_DEV_BAD_INDEX);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int NU = ue - ub;
  const int Kq = p.K / p.kq;
  const int nst = Kq / SK;
  const int NS = NU * nst;              // stages of each active warpgroup
  const int k0 = wg * Kq;

  auto epilogue = [&](int v) {
    finish_unit<MODE, TT>(v, ub, upe, groups, red, red_full, red_empty, p.kq, p.T, p.I, p.H, p.hbuf, p.expert_out,
                          abort_flag, p.status, p.wait_ns);
  };
  int epi = -1;   // a unit whose epilogue is due (it runs after the current block of stages)

  if (wg < p.kq) {
    const uint32_t tmem_wg = *tmem_base_p + wg * kColsPerWG;
    const uint32_t tlane = (uint32_t)(32 * wq) << 16;   // this warp's TMEM lane quarter
    const int KS = p.K / SK;              // chunks per row block
    const int KG = p.K >> p.lgG;
    const uint32_t idesc = umma_idesc_f16(BM, BN);
    const uint32_t bbase0 = smem_addr(Bs);

    // load cursor: the next stage to prefetch (unit lu, stage lst)
    int lu = ub, lst = 0;
    const uint4* lptr = nullptr;
    const unsigned short* lsp = nullptr;
    auto cursor_unit = [&](int u) {
      const int a = u / upe, m0 = (u - a * upe) * BM;
      const Group& gr = groups[a];
      if (gr.flags & 1) {
        lptr = reinterpret_cast<const uint4*>(gr.w + ((size_t)(m0 / BM) * KS + k0 / SK) * kChunk) + r;
        lsp = reinterpret_cast<const unsigned short*>(gr.s) + (size_t)(m0 / BM) * KG * BM + r;
      } else {
        lptr = nullptr;
        lsp = nullptr;
      }
    };
    cursor_unit(lu);
    uint4 ring[R][2];
    uint32_t sring[R];   // scales: SEG 32 both halves (low 16 bits: elements 0-31), else one
    // `first` = the stage starts a segment (SEG 128: only those load a scale)
    auto load_next = [&](uint4 (&dst)[2], uint32_t& sdst, bool first) {
      if (lptr) {
        dst[0] = __ldg(lptr + lst * (kChunk / 16));
        dst[1] = __ldg(lptr + lst * (kChunk / 16) + kChunk / 32);
        const int kk = k0 + lst * SK;
        if (SEG == 32)
          sdst = (uint32_t)__ldg(lsp + (size_t)(kk >> p.lgG) * BM) |
                 ((uint32_t)__ldg(lsp + (size_t)((kk + 32) >> p.lgG) * BM) << 16);
        else if (SEG == 64 || first)
          sdst = __ldg(lsp + (size_t)(kk >> p.lgG) * BM);
      } else {
        dst[0] = dst[1] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
        sdst = 0;
      }
      if (++lst == nst) {
        lst = 0;
        if (++lu < ue) cursor_unit(lu);
      }
    };
#pragma unroll
    for (int j = 0; j < R; ++j)
      if (j < NS) load_next(ring[j], sring[j], (j & 1) == 0);

    float acc[TT];
#pragma unroll
    for (int n = 0; n < TT; ++n) acc[n] = 0.f;
    // Segments that end in global stage e (odd: e is odd; stage est of local
    // unit eul; scale word sp): add them to acc; after a unit's last stage,
    // hand the partial sums over.
    auto readback = [&](int e, bool odd, int est, int eul, uint32_t sp) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const bool seg_end = SEG == 128 ? (odd && q == 3) : (SEG == 64 ? q == 3 : (q & 1) == 1);
        if (seg_end) {
          const int d = SEG == 128 ? ((e >> 1) & 1) : (SEG == 64 ? (e & 3) : ((2 * e + (q >> 1)) & 3));
          const float sc =
              __half2float(__ushort_as_half((unsigned short)(SEG == 32 && q >= 2 ? sp >> 16 : sp & 0xFFFFu)));
          if constexpr (TT == 1) {
            uint32_t dv[2];
            asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];"
                         : "=r"(dv[0]), "=r"(dv[1])
                         : "r"(tlane + tmem_wg + kD0 + 16 * d));
            tmem_ld_wait();
            acc[0] = fmaf(sc, __uint_as_float(dv[0]) + __uint_as_float(dv[1]), acc[0]);
          } else {
            uint32_t dv[16];
            tmem_ld_32x32b_x16(tlane + tmem_wg + kD0 + 16 * d, dv);
            tmem_ld_wait();
#pragma unroll
            for (int n = 0; n < TT; ++n)
              acc[n] = fmaf(sc, __uint_as_float(dv[2 * n]) + __uint_as_float(dv[2 * n + 1]), acc[n]);
          }
        }
      }
      if (est == nst - 1) {
        if (eul >= 2) mbar_wait_bounded(&red_empty[eul & 1], ((eul >> 1) - 1) & 1, abort_flag, p.status, p.wait_ns);
        float* rw = red + ((size_t)((eul & 1) * kWG + wg) * BM + r) * TT;
#pragma unroll
        for (int n = 0; n < TT; ++n) {
          rw[n] = acc[n];
          acc[n] = 0.f;
        }
        mbar_arrive(&red_full[eul & 1]);
      }
    };
    auto bbase_of = [&](int ul) {
      if constexpr (MODE == 1) return bbase0 + ((((ub + ul) / upe) - a_first) % p.nB) * b_bytes;
      return bbase0;
    };
    // lane 0 of the issuing warp: the four MMAs of global stage i (odd: i is odd;
    // stage ist of local unit iul; A buffer ib, whose phases have parity iph)
    auto issue = [&](int i, bool odd, int ist, int iul, int ib, int iph) {
      mbar_wait_bounded(&a_full[wg * 3 + ib], iph, abort_flag, p.status, p.wait_ns);
      tc_fence_after();
      const uint32_t bstage = bbase_of(iul) + (uint32_t)((k0 / SK + ist) * (BN * 128));
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int d = SEG == 128 ? ((i >> 1) & 1) : (SEG == 64 ? (i & 3) : ((2 * i + (q >> 1)) & 3));
        const bool fresh = SEG == 128 ? (!odd && q == 0) : (SEG == 64 ? q == 0 : (q & 1) == 0);
        umma_f16_tmem_a(tmem_wg + kD0 + 16 * d, tmem_wg + ib * 32 + 8 * q, umma_desc_sw128(bstage + 32 * q), idesc,
                        fresh ? 0u : 1u);
      }
      umma_commit(&done[wg * 3 + ib]);
    };
    auto issuer = [&](int i) { return ((SEG == 128 ? (i >> 1) : i) & 3) == wq; };

    uint32_t h1 = 0, h2 = 0, h3 = 0;   // scale words of global stages gs-1, gs-2, gs-3
    int st = 0, ul = 0;                // stage and local unit of gs
    // test hook (outside the stage loop, whose code size matters): warp 1 of
    // warpgroup 0 of the CTA owning unit 0 publishes its first stage late
    if (p.stall_ns && ub == 0 && wg == 0 && wq == 1 && lane == 0) debug_stall(p.stall_ns);
    int ab = 0, aph = 0;               // A buffer of gs and the parity of its phase there
    for (int gs0 = 0; gs0 < NS; gs0 += R) {
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int gs = gs0 + j;
        if (gs < NS) {
          // (0) this stage's weights and scales
          const uint32_t wd[8] = {ring[j][0].x, ring[j][0].y, ring[j][0].z, ring[j][0].w,
                                  ring[j][1].x, ring[j][1].y, ring[j][1].z, ring[j][1].w};
          // SEG 128: an odd stage continues the segment (and the scale) of the stage before
          const uint32_t sp = (SEG == 128 && (j & 1)) ? h1 : sring[j];
          // (1) stage gs - NA completed: A buffer ab is free, its segments are readable
          if (gs >= NA) {
            mbar_wait_bounded(&done[wg * 3 + ab], aph ^ 1, abort_flag, p.status, p.wait_ns);
            __syncwarp();
            tc_fence_after();
          }
          // (2) decode 64 nibbles into 32 fp16 pairs of this row, store them in TMEM
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t av[16];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              uint32_t pr[4];
              decode_nibbles(wd[4 * half + w], pr);
              av[4 * w + 0] = pr[0];
              av[4 * w + 1] = pr[1];
              av[4 * w + 2] = pr[2];
              av[4 * w + 3] = pr[3];
            }
            tmem_st_32x32b_x16(tlane + tmem_wg + ab * 32 + 16 * half, av);
          }
          // (3) while the store drains: read back stage gs - NA
          if (gs >= NA) {
            int est = st - NA, eul = ul;
            while (est < 0) {
              est += nst;
              --eul;
            }
            // a second unit end in one block (units shorter than a block): the
            // earlier unit's epilogue must run before this hand-over waits for it
            if (est == nst - 1 && epi >= 0) {
              epilogue(epi);
              epi = -1;
            }
            readback(gs - NA, ((j - NA) & 1) != 0, est, eul, NA == 3 ? h3 : h2);
            if (est == nst - 1 && eul >= 1) epi = eul - 1;
          }
          h3 = h2;
          h2 = h1;
          h1 = sp;
          // the slot is decoded: refill it R stages ahead
          if (gs + R < NS) load_next(ring[j], sring[j], (j & 1) == 0);
          // (4) publish the stored A
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_full[wg * 3 + ab]);
          // (5) issue the previous stage if it is this warp's turn
          if (gs >= 1 && issuer(gs - 1) && lane == 0) {
            const int ist = st > 0 ? st - 1 : nst - 1, iul = st > 0 ? ul : ul - 1;
            issue(gs - 1, ((j - 1) & 1) != 0, ist, iul, ab > 0 ? ab - 1 : NA - 1, ab > 0 ? aph : aph ^ 1);
          }
          __syncwarp();
          if (++st == nst) {
            st = 0;
            ++ul;
          }
          if (++ab == NA) {
            ab = 0;
            aph ^= 1;
          }
        }
      }
      // (6) soon after handing over unit v's partial sums, finish unit v - 1
      if (epi >= 0) {
        epilogue(epi);
        epi = -1;
      }
    }
    // tail: issue the last stage, read back the last stages, finish the last units
    if (issuer(NS - 1) && lane == 0)
      issue(NS - 1, ((NS - 1) & 1) != 0, st > 0 ? st - 1 : nst - 1, st > 0 ? ul : ul - 1, ab > 0 ? ab - 1 : NA - 1,
            ab > 0 ? aph : aph ^ 1);
    __syncwarp();
    for (int back = NA < NS ? NA : NS; back >= 1; --back) {
      const int e = NS - back;
      int eb = ab - back, eph = aph;
      if (eb < 0) {
        eb += NA;
        eph ^= 1;
      }
      mbar_wait_bounded(&done[wg * 3 + eb], eph, abort_flag, p.status, p.wait_ns);
      __syncwarp();
      tc_fence_after();
      int est = st - back, eul = ul;
      while (est < 0) {
        est += nst;
        --eul;
      }
      if (est == nst - 1 && epi >= 0) {
        epilogue(epi);
        epi = -1;
      }
      readback(e, (e & 1) != 0, est, eul, back == 1 ? h1 : (back == 2 ? h2 : h3));
      if (est == nst - 1 && eul >= 1) epi = eul - 1;
    }
    tc_fence_before();
    if (epi >= 0) epilogue(epi);
    epilogue(NU - 1);
  } else {
    // warpgroups without a K slice only finish units
    for (int v = 0; v < NU; ++v) epilogue(v);
  }

  // Every MMA must have completed before tensor memory is freed.  Without a
  // give-up the waits above saw every stage complete; after one, each warp's
  // issuing lane commits once more (tracking all its earlier MMAs) and waits.
  __syncthreads();
  if (*abort_flag) {
    if (lane == 0) {
      umma_commit(&drain[warp]);
      mbar_wait_drain(&drain[warp], 0, p.status);
    }
    __syncthreads();
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(*tmem_base_p, kWG * kColsPerWG);
  }
}

// ---------------------------------------------------------------- gate/up with FP8 weights in tensor memory
//
// For G = 128 both decode phases hold the weights in tensor memory as FP8
// E4M3 codes of the unsigned nibbles u = q + 8: the code byte is the nibble
// itself, worth u * 2^-9 (split_nibbles_e4m3), so the decode is a mask and a
// shift.  One byte per weight instead of two, so half the tcgen05.st traffic
// and half the MMAs (kind::f8f6f4 consumes K = 32), and a 128-element stage
// (one whole group) per synchronisation.  A packed 32-bit word (reduction
// indices 8w .. 8w + 7) becomes two TMEM columns, the even indices then the
// odd ones, and the B operand is filled in that same order: physical position
// 8w + 4h + i of a stage holds reduction index 8w + 2i + h.
// The activations (x for gate/up, h for down) enter as E4M3 too: for each
// token and group, v = x * 2^e (e puts the group's largest |x| in [128, 256))
// is written as terms t_j = 2^-4j * E4M3(2^4j * r_j) with r_0 = v and
// r_(j+1) = r_j - t_j, so every term is rounded in the normal E4M3 range.  Two
// terms hold a bf16 x exactly (its 8 significant bits split 4 + 4, the second
// residual fitting 4 bits after round-to-nearest) unless the element is below
// 2^-13 of its group's largest; h, an fp32 value, takes four (about 16
// significant bits).  Term j of token n is B row NT n + j (NT terms; N = 16,
// or 32 for eight tokens of h), holding the code of 2^4j * t_j; the readback
// adds the NT accumulator columns with weights 2^-4j.  The group's dot product
// is then
//   sum_k q_k x_k = 2^(9-e) * sum_k (u_k 2^-9) (t_0 + .. + t_(NT-1))_k - 8 * sum_k x_k,
// with the first sum from the tensor core (products exact, fp32 accumulation)
// and the correction precomputed per token and group from the same terms.
// Pipeline as in the 64-element kernel with segment = stage: two A buffers, two
// D buffers, item g read back during iteration g + 2, issued during g + 1 by
// warp g mod 4.
constexpr int SK8 = 128;                   // reduction elements per stage (one group)
constexpr int kA8 = SK8 / 4;               // TMEM columns of one A buffer (4 codes per column)
// E4M3 terms per activation element: x (bf16) two, h (fp32) four.
__host__ __device__ constexpr int n_terms(int MODE) { return MODE == 0 ? 2 : 4; }

// Accumulator columns of the NT terms of one token, term j weighted 2^-4j.
template <int NT>
__device__ __forceinline__ float add_terms(const uint32_t* c) {
  float d = __uint_as_float(c[NT - 1]);
#pragma unroll
  for (int j = NT - 2; j >= 0; --j) d = fmaf(d, 0.0625f, __uint_as_float(c[j]));
  return d;
}

// MMA N (B rows) of the FP8 kernel: NT terms per token, at least 16.
__host__ __device__ constexpr int bn8(int MODE, int TT) { return n_terms(MODE) * TT <= 16 ? 16 : 32; }

// Where shared memory allows, the weights stream through a ring of stages
// that every thread fills with cp.async (its own 4 x 16 bytes per stage, read
// back by itself, so only cp.async groups order them): kStages8 stages in
// flight without holding registers.  The down kernel for eight tokens fits
// its ring beside two experts' h (128 KB) because each warpgroup keeps the
// partial sums of the two tokens it finishes in registers instead of the
// reduction area (red_tt).
constexpr int kStages8 = 2;
constexpr int kStageBytes8 = BM * SK8 / 2;   // one warpgroup's stage: 128 rows x 128 nibbles
// fp32 partials per (warpgroup, row) in the reduction area
__host__ __device__ constexpr int red_tt(int MODE, int TT) { return (MODE == 1 && TT == 8) ? TT - 2 : TT; }

struct Layout8 {
  int b_off, ec_off, ring_off, red_off, bar_off, grp_off, misc_off;
  size_t bytes;
};

__host__ __device__ inline Layout8 make_layout8(int MODE, int K, int nB, int TT) {
  Layout8 L;
  L.b_off = 0;                                          // nB x (bn8 rows x K bytes, swizzled; 1024-aligned)
  L.ec_off = L.b_off + nB * bn8(MODE, TT) * K;          // nB x 2 x TT x K/128 fp32 factors (see Et)
  L.ring_off = (L.ec_off + nB * 2 * TT * (K / SK8) * 4 + 127) & ~127;   // [stage][kWG] x 8 KB
  L.red_off = L.ring_off + kStages8 * kWG * kStageBytes8;   // 2 x kWG x BM x red_tt fp32
  L.bar_off = L.red_off + 2 * kWG * BM * red_tt(MODE, TT) * 4;
  L.grp_off = L.bar_off + (kWG * 6 + 4 + kThreads / 32) * 8;
  L.misc_off = L.grp_off + kMaxGroups * (int)sizeof(Group);
  L.bytes = (size_t)L.misc_off + 16 + 1024;
  return L;
}

// Byte offset of (row n, reduction index l) in an E4M3 B operand of `rows` rows.
__device__ __forceinline__ uint32_t b8_offset(int n, int l, int rows) {
  const int byte = l & 127;
  return (uint32_t)((l >> 7) * (rows * 128) + (n >> 3) * 1024 + (n & 7) * 128 + ((((byte >> 4) ^ (n & 7))) << 4) +
                    (byte & 15));
}

// One B operand job of the FP8 kernel: (buffer jb, token n, group g) of job
// index `job`, whose raw activations are `raw` (gate/up: 8 bf16 of which this
// lane takes the even or odd ones; down: 4 fp32 h in B order).  Lane l writes
// physical positions 4l .. 4l + 3 of the group's four term rows, and lane 0 the
// group's 2^(9-e) and offset entries.  Out of line: one copy of the code for
// all jobs.
template <int MODE, int TT, int BN8, int NT>
__device__ __noinline__ void e4m3_b_job(int job, const uint4 raw, int T, int KG, uint8_t* Bs, float* Et,
                                        uint32_t b_bytes) {
  const int lane = threadIdx.x & 31;
  const int jb = job >= T * KG ? 1 : 0, tg = job - jb * (T * KG);   // at most two buffers
  const int n = tg / KG, g = tg - n * KG;
  float v[4];
  if constexpr (MODE == 0) {
    const int sh = 16 * (lane & 1);
    v[0] = bf16_bits_to_float((raw.x >> sh) & 0xFFFFu);
    v[1] = bf16_bits_to_float((raw.y >> sh) & 0xFFFFu);
    v[2] = bf16_bits_to_float((raw.z >> sh) & 0xFFFFu);
    v[3] = bf16_bits_to_float((raw.w >> sh) & 0xFFFFu);
  } else {
    v[0] = __uint_as_float(raw.x);   // h is stored in this order (H32 epilogue)
    v[1] = __uint_as_float(raw.y);
    v[2] = __uint_as_float(raw.z);
    v[3] = __uint_as_float(raw.w);
  }
  float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  // 2^e with m * 2^e in [128, 256): from the exponent field of m
  int ex = m > 0.f ? 7 - (int)((__float_as_uint(m) >> 23) & 0xFF) + 127 : 0;
  ex = ex < -100 ? -100 : (ex > 100 ? 100 : ex);
  const float up = __uint_as_float((uint32_t)(127 + ex) << 23), down = __uint_as_float((uint32_t)(127 - ex) << 23);
  uint32_t t[NT];    // 4 codes of each term
  float back = 0.f;  // sum of the represented values of this lane's 4 elements
#pragma unroll
  for (int j = 0; j < NT; ++j) t[j] = 0u;
#pragma unroll
  for (int k = 0; k < 2; ++k) {   // elements 2k, 2k + 1, converted as a pair
    float2 rem = make_float2(v[2 * k] * up, v[2 * k + 1] * up);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const float lift = (float)(1 << (4 * j)), drop = 1.0f / lift;   // powers of two: exact
      const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(make_float2(rem.x * lift, rem.y * lift),
                                                              __NV_SATFINITE, __NV_E4M3);
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(c, __NV_E4M3);
      const float2 cv = __half22float2(__half2(hr));
      t[j] |= (uint32_t)c << (16 * k);   // element 2k in the low byte
      rem.x -= cv.x * drop;
      rem.y -= cv.y * drop;
      back += (cv.x + cv.y) * drop;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) back += __shfl_xor_sync(0xffffffffu, back, o);
#pragma unroll
  for (int j = 0; j < NT; ++j)
    *reinterpret_cast<uint32_t*>(Bs + jb * b_bytes + b8_offset(NT * n + j, g * SK8 + 4 * lane, BN8)) = t[j];
  if (lane == 0) {
    float* ec = Et + jb * 2 * TT * KG;   // [KG][TT] pairs: a stage's factors of all tokens together
    ec[(g * TT + n) * 2] = 512.0f * down;   // the codes carry 2^-9
    ec[(g * TT + n) * 2 + 1] = 8.0f * back * down;
  }
}

// A unit of a host-mapped expert streams over the host link at a fraction of
// the rate of device memory.  With qre_set_host_unit_cost the FP8 kernels run
// an instance that cuts its contiguous unit ranges at equal cost, such a unit
// counted as `cost` device-memory units, so the host-resident experts of a
// call spread over more CTAs.  (A separate instance: in the default one the
// extra code measurably slowed the all-HBM decode.)

// This CTA's unit range [ub, ue) (x, y): contiguous ranges over the grid cut at
// equal cost, `cost` for units of host-mapped groups and 1 otherwise,
// when a host-mapped group is present and (down kernel, max_span_groups > 0)
// no range can then span more than two groups; else at equal unit counts.
// Out of line: it runs once per CTA and keeps its registers off the kernel.
__device__ __noinline__ int2 unit_range(const Group* groups, int ngroups, int upe, bool limit_span, int nB,
                                        int cost) {
  const long long U = (long long)ngroups * upe, grid = gridDim.x, c = blockIdx.x;
  long long C = 0;
  bool host = false;
  for (int a = 0; a < ngroups; ++a) {
    const bool h = (groups[a].flags & 2) != 0;
    host |= h;
    C += (long long)upe * (h ? cost : 1);
  }
  if (!host || (limit_span && (nB < 2 || C > grid * upe))) return make_int2((int)(c * U / grid), (int)((c + 1) * U / grid));
  // the first unit whose cost before it, times the grid, reaches `target`
  auto first_unit = [&](long long target) -> int {
    long long base = 0;
    for (int a = 0; a < ngroups; ++a) {
      const long long w = (groups[a].flags & 2) ? cost : 1;
      if ((base + (upe - 1) * w) * grid >= target) {
        const long long num = target - base * grid;
        return a * upe + (num <= 0 ? 0 : (int)((num + w * grid - 1) / (w * grid)));
      }
      base += upe * w;
    }
    return (int)U;
  };
  return make_int2(first_unit(c * C), first_unit((c + 1) * C));
}

template <int MODE, int TT, bool HC = false>
__global__ void __launch_bounds__(kThreads, 1) ffn_e4m3_kernel(const FfnParams p) {
  constexpr int kStages = kStages8;                 // shared-memory ring depth
  constexpr int R = kStages;                        // ring depth = unroll
  constexpr int NA = 2;                    // A buffers (and D buffers) per warpgroup
  constexpr int NT = n_terms(MODE);
  constexpr int BN8 = bn8(MODE, TT);       // MMA N
  constexpr int kD0 = NA * kA8;            // first D column
  static_assert(kD0 + NA * BN8 <= kColsPerWG, "TMEM columns per warpgroup");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const Layout8 L = make_layout8(MODE, p.K, p.nB, TT);
  uint8_t* Bs = smem + L.b_off;                                    // buffer j at j * b_bytes
  float* Et = reinterpret_cast<float*>(smem + L.ec_off);          // buffer j at j * 2 * TT * KG: [KG][TT] pairs
                                                                   // (2^(9-e), 8 * sum of the represented values)
  float* red = reinterpret_cast<float*>(smem + L.red_off);
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* done = a_full + kWG * 3;
  uint64_t* red_full = done + kWG * 3;
  uint64_t* red_empty = red_full + 2;
  uint64_t* drain = red_empty + 2;
  Group* groups = reinterpret_cast<Group*>(smem + L.grp_off);
  uint32_t* tmem_base_p = reinterpret_cast<uint32_t*>(smem + L.misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc_off + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int KG = p.K / SK8;
  // Both kernels are programmatic dependents (launch_dependent).  gate/up
  // waits for the dispatch before anything else and then lets the down kernel
  // be scheduled: down CTAs take the SMs that gate/up CTAs leave, build their
  // group table and fill their weight ring (dispatch outputs and weights, all
  // complete by then), and wait for the gate/up grid only before reading h.
  if constexpr (MODE == 0) {
    // While the dispatch still runs: bring the slot table into L2 (it is read
    // right after the wait, one dependent load before the first weights; a
    // line written meanwhile, e.g. by the cache manager, is current in L2).
    const int lines = ((p.E + 1) * (int)sizeof(qre_slot) + 127) / 128;
    if ((int)threadIdx.x < lines)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(p.slots) + 128 * threadIdx.x));
    grid_dependency_wait();
    grid_dependents_launch();
  }
  // B operand jobs: (buffer jb, token n, group g), one warp each, lane l
  // holding physical positions 4l .. 4l + 3 of the group (reduction indices
  // 8(l >> 1) + (l & 1) + 2i).  A warp's first kJB jobs have their loads in
  // flight before the group table: the tokens do not depend on the routing,
  // h only on the range.
  constexpr int kJB = 8;
  const float* hb32 = reinterpret_cast<const float*>(p.hbuf);
  // jobs of one buffer are (n, g) row-major, i.e. consecutive 128-element
  // blocks of the activation rows (x rows of H = KG * 128, h rows of I)
  const int tjobs = p.T * KG;   // jobs per buffer; at most two buffers
  auto job_load = [&](int job, int a0) -> uint4 {
    const int jb = job >= tjobs ? 1 : 0, rem = job - jb * tjobs;
    if constexpr (MODE == 0)
      return ldg_v4_early(p.x + (size_t)rem * SK8 + 8 * (lane >> 1));
    else
      return ldg_v4_early(hb32 + (size_t)(a0 + jb) * kTok * p.I + (size_t)rem * SK8 + 4 * lane);
  };
  // B workers: gate/up leaves warp 0 to the group table and builds B on warps
  // 1..15 before the group-table barrier (overlapping the slot-table loads);
  // down uses all 16 warps once h may be read.
  constexpr int kW0 = MODE == 0 ? 1 : 0, kNW = kThreads / 32 - kW0;
  const int wk = warp - kW0;
  uint4 pre[kJB];
  if constexpr (MODE == 0) {
#pragma unroll
    for (int b = 0; b < kJB; ++b)
      if (wk >= 0 && wk + kNW * b < p.T * KG) pre[b] = job_load(wk + kNW * b, 0);
  }

  // groups: the active experts (parts 0, 1), then the shared one (parts 0, 2);
  // the shared-only launch reads no routing at all
  const int a_spec = (p.part != 2 && threadIdx.x < p.amax) ? __ldg(p.active + threadIdx.x) : p.E;
  int n_act = p.part == 2 ? 0 : *p.n_active;
  n_act = n_act < 0 ? 0 : (n_act > p.amax ? p.amax : n_act);
  const int ngroups = n_act + (p.part == 1 ? 0 : 1);
  const int upe = p.n_out / BM;
  const int U = ngroups * upe;
  int ub = (int)((long long)blockIdx.x * U / gridDim.x);
  int ue = (int)((long long)(blockIdx.x + 1) * U / gridDim.x);
  if (ub >= ue) return;

  const int wg = tid >> 7, r = tid & 127, wq = warp & 3;
  const uint32_t b_bytes = (uint32_t)BN8 * p.K;
  int a_first = ub / upe, a_last = (ue - 1) / upe;
  int nbuf = MODE == 0 ? 1 : (a_last - a_first + 1 < p.nB ? a_last - a_first + 1 : p.nB);
  int njobs = nbuf * p.T * KG;
  auto b_fill = [&](int a0) {
    for (int b0 = 0; wk >= 0 && wk + kNW * b0 < njobs; b0 += kJB) {
      if (b0 > 0) {
#pragma unroll
        for (int b = 0; b < kJB; ++b)
          if (wk + kNW * (b0 + b) < njobs) pre[b] = job_load(wk + kNW * (b0 + b), a0);
      }
#pragma unroll
      for (int b = 0; b < kJB; ++b)
        if (wk + kNW * (b0 + b) < njobs)
          e4m3_b_job<MODE, TT, BN8, NT>(wk + kNW * (b0 + b), pre[b], p.T, KG, Bs, Et, b_bytes);
    }
  };

  int olo = 0, ohi = 0;   // down: the dispatch range of this thread's group (tid < n_act)
  for (int a = tid; a < ngroups; a += blockDim.x) {
    const int e = a < n_act ? (a == tid ? a_spec : __ldg(p.active + a)) : p.E;
    if (MODE == 1 && a < n_act && a == tid && e >= 0 && e < p.E) {
      olo = __ldg(p.offsets + e);   // in flight with the slot entry
      ohi = __ldg(p.offsets + e + 1);
    }
    const uint8_t* w = nullptr;
    const uint16_t* sc = nullptr;
    int flags = 0;
    if (e >= 0 && e <= p.E) {
      const qre_slot* sl = p.slots + e;
      w = MODE == 0 ? sl->w_gate_up : sl->w_down;
      sc = MODE == 0 ? sl->s_gate_up : sl->s_down;
      flags = (w && sc && ((reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(sc)) & 15) == 0) ? 1 : 0;
      if (flags && sl->tier != 0) flags |= 2;   // host-mapped: plain loads only
    }
    if (!flags && a >= a_first && a <= a_last) set_status(p.status, QRE_DEV_NULL_SLOT);
    Group& dst = groups[a];
    dst.w = w;
    dst.s = sc;
    dst.e = e;
    dst.flags = flags;
#pragma unroll
    for (int n = 0; n < kTok; ++n) dst.outq[n] = (MODE == 1 && a == n_act && n < p.T) ? p.T * p.k + n : -1;
  }
  if (tid == 0) {
    for (int i = 0; i < kWG * 3; ++i) {
      mbar_init(&a_full[i], 4);
      mbar_init(&done[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&red_full[i], 128 * p.kq);
      mbar_init(&red_empty[i], kThreads);
    }
    for (int i = 0; i < kThreads / 32; ++i) mbar_init(&drain[i], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(tmem_base_p, kWG * kColsPerWG);
    tmem_relinquish();
  }
  if constexpr (MODE == 0) {
    b_fill(0);
    fence_proxy_async_smem();   // B is read by the tensor core (async proxy)
  }
  // The weight stream does not depend on the activations: with the group
  // table in place every warpgroup puts its first ring stages in flight (down:
  // while the gate/up grid finishes, before h is read).
  __syncthreads();
  if constexpr (HC) {
    // Host-mapped groups in the table: re-cut the ranges at equal cost
    // (unit_range; every CTA had units when U >= grid, so none returned early
    // above); a CTA left without units gives its tensor memory back.
    if (U >= (int)gridDim.x) {
      const int2 rc = unit_range(groups, ngroups, upe, MODE == 1, p.nB, p.host_cost);
      if (rc.x != ub || rc.y != ue) {
        ub = rc.x;
        ue = rc.y;
        if (ub >= ue) {
          if (warp == 0) {
            tc_fence_after();
            tmem_dealloc(*tmem_base_p, kWG * kColsPerWG);
          }
          return;
        }
        a_first = ub / upe;
        a_last = (ue - 1) / upe;
        if (MODE == 1) {
          nbuf = a_last - a_first + 1 < p.nB ? a_last - a_first + 1 : p.nB;
          njobs = nbuf * p.T * KG;
        }
      }
    }
  }
  const int NU = ue - ub;
  const int Kq = p.K / p.kq;
  const int nst = Kq / SK8;
  const int NS = NU * nst;
  const int k0 = wg * Kq;
  const int g0 = k0 / SK8;           // first group of this warpgroup's slice
  const int KS = p.K / SK;           // 64-element chunks per row block

  int lu = ub, lst = 0;
  const uint4* lptr = nullptr;
  const unsigned short* lsp = nullptr;
  bool lhost = false;
  // Weight and scale cursors advanced per stage and per unit instead of
  // recomputed from the stage index (no division in the stage loop).
  int la = lu / upe, lmb = lu - la * upe;   // the cursor's group and row block
  auto cursor_unit = [&]() {
    const int a = la, mb = lmb;
    const Group& gr = groups[a];
    if (gr.flags & 1) {
      lptr = reinterpret_cast<const uint4*>(gr.w + ((size_t)mb * KS + k0 / SK) * kChunk) + r;
      lsp = reinterpret_cast<const unsigned short*>(gr.s) + ((size_t)mb * KG + g0) * BM + r;
      lhost = (gr.flags & 2) != 0;
    } else {
      lptr = nullptr;
      lsp = nullptr;
    }
  };
  cursor_unit();
  uint32_t sring[R];                // weight scales of the stages in flight
  // shared-memory ring: this thread's 16 bytes of each quarter
  // of slot 0; slot j, quarter c at + j * kWG * kStageBytes8 + c * 2048
  uint8_t* const sbuf = smem + L.ring_off + wg * kStageBytes8 + r * 16;
  constexpr uint32_t kQuarter = kChunk / 2;   // bytes between a thread's four 16-byte pieces of a stage
  // ring slot j <- the next stage of this warpgroup's slice
  auto load_next = [&](int j) {
    if (lptr) {
      // chunks 2*lst and 2*lst + 1 of the slice
      const uint4* c = lptr;
      uint8_t* d = sbuf + j * (kWG * kStageBytes8);
      if (lhost) {
#pragma unroll
        for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(d + q * kQuarter) = __ldg(c + q * (kQuarter / 16));
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) cp_async_16(d + q * kQuarter, c + q * (kQuarter / 16));
      }
      sring[j] = __ldg(lsp);
      lptr += 2 * kChunk / 16;
      lsp += BM;
    } else {
      const uint4 z = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
#pragma unroll
      for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(sbuf + j * (kWG * kStageBytes8) + q * kQuarter) = z;
      sring[j] = 0;
    }
    cp_async_commit();
    if (++lst == nst) {
      lst = 0;
      if (++lmb == upe) {
        lmb = 0;
        ++la;
      }
      if (++lu < ue) cursor_unit();
    }
  };
  if (wg < p.kq) {
#pragma unroll
    for (int j = 0; j < R; ++j) {
      if (j < NS) {
        load_next(j);
      } else {
        cp_async_commit();   // one group per ring slot, loaded or not
      }
    }
  }

  // down: everything above (group table, first weight stages) overlaps the end
  // of the gate/up grid; h is read only once that grid has completed
  if constexpr (MODE == 1) {
    grid_dependency_wait();
    grid_dependents_launch();
#pragma unroll
    for (int b = 0; b < kJB; ++b)
      if (wk + kNW * b < njobs) pre[b] = job_load(wk + kNW * b, a_first);
    // the expert_out rows of each routed group's tokens (read by the epilogues
    // only): their perm loads travel together with the h loads above
    for (int a = tid; a < n_act; a += blockDim.x) {
      Group& dst = groups[a];
      if (!(dst.flags & 1)) continue;
      const bool mine = a == tid;   // always, as n_act < blockDim.x
      const int lo = mine ? olo : __ldg(p.offsets + dst.e), hi = mine ? ohi : __ldg(p.offsets + dst.e + 1);
      for (int q = lo; q < hi && q < lo + kTok; ++q) {
        const int tk = __ldg(p.perm + q) / p.k;
        if (tk >= 0 && tk < kTok) dst.outq[tk] = q;
      }
    }
  }
  // B: gate/up one buffer of the tokens, down one buffer of h per expert of the
  // range (at most nB, by the launch).
  if (MODE == 1 && a_last - a_first >= p.nB && tid == 0) set_status(p.status, QRE_DEV_BAD_INDEX);
  if constexpr (MODE == 1) b_fill(a_first);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();


  // eight-token down kernel: this thread's partials of its own two tokens, by unit parity
  float own[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  auto epilogue = [&](int v) {
    finish_unit<MODE, TT, true>(v, ub, upe, groups, red, red_full, red_empty, p.kq, p.T, p.I, p.H, p.hbuf,
                                p.expert_out, abort_flag, p.status, p.wait_ns, (v & 1) ? own[1][0] : own[0][0],
                                (v & 1) ? own[1][1] : own[0][1]);
  };
  int epi = -1;

  if (wg < p.kq) {
    const uint32_t tmem_wg = *tmem_base_p + wg * kColsPerWG;
    const uint32_t tlane = (uint32_t)(32 * wq) << 16;
    const uint32_t idesc = umma_idesc_e4m3(BM, BN8);
    const uint32_t bbase = smem_addr(Bs);

    // down: the local units from u_split on belong to the range's second group
    // (its h in the second B buffer; a range spans at most nB <= 2 groups)
    const int u_split = (a_first + 1) * upe - ub;
    float acc[TT];
#pragma unroll
    for (int n = 0; n < TT; ++n) acc[n] = 0.f;
    // stage est of local unit eul (D buffer db, weight scale sp) completed: add it
    auto readback = [&](int est, int eul, int db, uint32_t sp) {
      const float sc = __half2float(__ushort_as_half((unsigned short)sp));
      const int g = g0 + est;
      const float* ec = MODE == 0 ? Et : Et + (eul >= u_split ? 2 * TT * KG : 0);
      if constexpr (TT == 1) {
        uint32_t dv[4];
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(dv[0]), "=r"(dv[1]), "=r"(dv[2]), "=r"(dv[3])
                     : "r"(tlane + tmem_wg + kD0 + BN8 * db));
        tmem_ld_wait();
        const float d = add_terms<NT>(dv);
        const float2 q = *reinterpret_cast<const float2*>(ec + 2 * g);   // (2^(9-e), correction)
        acc[0] = fmaf(sc, fmaf(d, q.x, -q.y), acc[0]);
      } else {
        uint32_t dv[BN8];
        if constexpr (BN8 == 32)
          tmem_ld_32x32b_x32(tlane + tmem_wg + kD0 + BN8 * db, dv);
        else
          tmem_ld_32x32b_x16(tlane + tmem_wg + kD0 + BN8 * db, dv);
        tmem_ld_wait();
        const float4* eg = reinterpret_cast<const float4*>(ec + g * 2 * TT);   // (2^(9-e), C) per token
#pragma unroll
        for (int n2 = 0; n2 < TT / 2; ++n2) {
          const float4 q = eg[n2];
          const float d0 = add_terms<NT>(dv + NT * (2 * n2)), d1 = add_terms<NT>(dv + NT * (2 * n2 + 1));
          acc[2 * n2] = fmaf(sc, fmaf(d0, q.x, -q.y), acc[2 * n2]);
          acc[2 * n2 + 1] = fmaf(sc, fmaf(d1, q.z, -q.w), acc[2 * n2 + 1]);
        }
      }
      if (est == nst - 1) {
        if (epi >= 0) {
          epilogue(epi);
          epi = -1;
        }
        if (eul >= 2) mbar_wait_bounded(&red_empty[eul & 1], ((eul >> 1) - 1) & 1, abort_flag, p.status, p.wait_ns);
        constexpr int RT = red_tt(MODE, TT);
        float* rw = red + ((size_t)((eul & 1) * kWG + wg) * BM + r) * RT;
        if constexpr (RT == TT) {
#pragma unroll
          for (int n = 0; n < TT; ++n) {
            rw[n] = acc[n];
            acc[n] = 0.f;
          }
        } else {
          // tokens 2wg, 2wg + 1 stay in registers for this warpgroup's own epilogue
          const float m0 = wg == 0 ? acc[0] : (wg == 1 ? acc[2] : (wg == 2 ? acc[4] : acc[6]));
          const float m1 = wg == 0 ? acc[1] : (wg == 1 ? acc[3] : (wg == 2 ? acc[5] : acc[7]));
          if (eul & 1) {
            own[1][0] = m0;
            own[1][1] = m1;
          } else {
            own[0][0] = m0;
            own[0][1] = m1;
          }
#pragma unroll
          for (int n = 0; n < TT; ++n) {
            if ((n >> 1) != wg) rw[n < 2 * wg ? n : n - 2] = acc[n];
            acc[n] = 0.f;
          }
        }
        mbar_arrive(&red_full[eul & 1]);
        if (eul >= 1) epi = eul - 1;
      }
    };
    // lane 0 of warp (stage mod 4): the 4 MMAs of global stage i (stage ist of
    // local unit iul), A/D buffer i & 1
    auto issue = [&](int i, int ist, int iul) {
      const int ib = i & 1;
      mbar_wait_bounded(&a_full[wg * 3 + ib], (i >> 1) & 1, abort_flag, p.status, p.wait_ns);
      tc_fence_after();
      const uint32_t bbuf = MODE == 0 ? 0u : (iul >= u_split ? b_bytes : 0u);
      const uint32_t bstage = bbase + bbuf + (uint32_t)((g0 + ist) * (BN8 * 128));
      const uint64_t bdesc = umma_desc_sw128(bstage);   // + 2 per 32 bytes inside the swizzle row
#pragma unroll
      for (int q = 0; q < 4; ++q)
        umma_e4m3_tmem_a(tmem_wg + kD0 + BN8 * ib, tmem_wg + ib * kA8 + 8 * q, bdesc + (uint64_t)(2 * q), idesc,
                         q ? 1u : 0u);
      umma_commit(&done[wg * 3 + ib]);
    };

    uint32_t h1 = 0, h2 = 0;   // weight scales of stages gs-1, gs-2
    int st = 0, ul = 0;
    int rst = 0, rul = 0;      // the next stage to read back (gs - 2) and its local unit
    auto readback_next = [&](int db, uint32_t sp) {
      readback(rst, rul, db, sp);
      if (++rst == nst) {
        rst = 0;
        ++rul;
      }
    };
    // test hook (outside the stage loop, whose code size matters): warp 1 of
    // warpgroup 0 of the CTA owning unit 0 publishes its first stage late
    if (p.stall_ns && ub == 0 && wg == 0 && wq == 1 && lane == 0) debug_stall(p.stall_ns);
    for (int gs0 = 0; gs0 < NS; gs0 += R) {
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int gs = gs0 + j, ab = j & 1;   // gs0 is a multiple of R (even): buffer = gs & 1 = j & 1
        if (gs < NS) {
          // (1) stage gs - 2 completed: A buffer ab is free, its D readable
          if (gs >= 2) {
            mbar_wait_bounded(&done[wg * 3 + ab], ((gs - 2) >> 1) & 1, abort_flag, p.status, p.wait_ns);
            __syncwarp();
            tc_fence_after();
          }
          // (2) split 128 nibbles of this row into 128 E4M3 codes, store them in TMEM
          {
            uint4 cur[4];
            cp_async_wait_group<kStages - 1>();   // slot j's group (the oldest in flight) has landed
#pragma unroll
            for (int q = 0; q < 4; ++q)
              cur[q] = *reinterpret_cast<const uint4*>(sbuf + j * (kWG * kStageBytes8) + q * kQuarter);
            uint32_t av[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint32_t wd[4] = {cur[c].x, cur[c].y, cur[c].z, cur[c].w};
#pragma unroll
              for (int w = 0; w < 4; ++w) split_nibbles_e4m3(wd[w], av[8 * c + 2 * w], av[8 * c + 2 * w + 1]);
            }
            tmem_st_32x32b_x32(tlane + tmem_wg + ab * kA8, av);
          }
          const uint32_t sp = sring[j];
          if (gs + R < NS) {
            load_next(j);
          } else {
            cp_async_commit();   // keeps the group count in step with the stages
          }
          // (3) while the store drains: read back stage gs - 2
          if (gs >= 2) readback_next(ab, h2);
          h2 = h1;
          h1 = sp;
          // (4) publish the stored A
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_full[wg * 3 + ab]);
          // (5) issue stage gs - 1 if it is this warp's turn
          if (gs >= 1 && ((gs - 1) & 3) == wq && lane == 0) issue(gs - 1, st > 0 ? st - 1 : nst - 1, st > 0 ? ul : ul - 1);
          __syncwarp();
          if (++st == nst) {
            st = 0;
            ++ul;
          }
        }
      }
      if (epi >= 0) {
        epilogue(epi);
        epi = -1;
      }
    }
    if (((NS - 1) & 3) == wq && lane == 0) issue(NS - 1, st > 0 ? st - 1 : nst - 1, st > 0 ? ul : ul - 1);
    __syncwarp();
    for (int back = NS < 2 ? NS : 2; back >= 1; --back) {
      const int e = NS - back;
      mbar_wait_bounded(&done[wg * 3 + (e & 1)], (e >> 1) & 1, abort_flag, p.status, p.wait_ns);
      __syncwarp();
      tc_fence_after();
      readback_next(e & 1, back == 1 ? h1 : h2);
    }
    tc_fence_before();
    if (epi >= 0) epilogue(epi);
    epilogue(NU - 1);
  } else {
    for (int v = 0; v < NU; ++v) epilogue(v);
  }

  // Every MMA must have completed before tensor memory is freed.  Without a
  // give-up the waits above saw every stage complete; after one, each warp's
  // issuing lane commits once more (tracking all its earlier MMAs) and waits.
  __syncthreads();
  if (*abort_flag) {
    if (lane == 0) {
      umma_commit(&drain[warp]);
      mbar_wait_drain(&drain[warp], 0, p.status);
    }
    __syncthreads();
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(*tmem_base_p, kWG * kColsPerWG);
  }
}

int ilog2(int v) {
  int l = 0;
  while ((1 << (l + 1)) <= v) ++l;
  return l;
}

// Warpgroups that split K: whole stages each, and accumulation segments that
// are either whole groups or whole K slices.
int pick_kq(int K, int G) {
  for (int kq : {4, 2, 1}) {
    const int Kq = K / kq;
    if (K % kq == 0 && Kq % SK == 0 && (Kq % G == 0 || G % Kq == 0)) return kq;
  }
  return 0;
}

int smem_needed(int K, int nB, int TT) {
  const size_t b = make_layout(K, nB, TT).bytes;
  // at least ~120 KB so that no second CTA (and no second TMEM allocation) shares an SM
  return (int)(b > 120 * 1024 ? b : 120 * 1024);
}

template <int MODE, int SEG, int TT>
cudaError_t launch_k(const FfnParams& p, int grid, int smem, cudaStream_t stream) {
  const cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(ffn_decode_kernel<MODE, SEG, TT>), smem);
  if (err != cudaSuccess) return err;
  return launch_dependent(ffn_decode_kernel<MODE, SEG, TT>, dim3(grid), dim3(kThreads), smem, stream, p);
}

template <int MODE, int TT>
cudaError_t launch_tt(const FfnParams& p, int seg, int grid, int smem, cudaStream_t stream) {
  if (seg == 128) return launch_k<MODE, 128, TT>(p, grid, smem, stream);
  if (seg == 64) return launch_k<MODE, 64, TT>(p, grid, smem, stream);
  return launch_k<MODE, 32, TT>(p, grid, smem, stream);
}

int smem_needed8(int MODE, int K, int nB, int TT) {
  const size_t b = make_layout8(MODE, K, nB, TT).bytes;
  return (int)(b > 120 * 1024 ? b : 120 * 1024);
}

template <int MODE, int TT>
cudaError_t launch_e4m3(const FfnParams& p, int grid, int smem, cudaStream_t stream) {
  auto kernel = p.host_cost > 1 ? ffn_e4m3_kernel<MODE, TT, true> : ffn_e4m3_kernel<MODE, TT, false>;
  const cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(kernel), smem);
  if (err != cudaSuccess) return err;
  return launch_dependent(kernel, dim3(grid), dim3(kThreads), smem, stream, p);
}

// One CTA per SM.  The down kernels hold the B operand (h) of every expert of
// their range in shared memory, so their ranges span at most nB experts: with
// two buffers at least one CTA per group (ranges of at most one expert's
// units), with one buffer one unit per CTA.
long long decode_grid(int MODE, int nB, long long units, int amax, int sms) {
  long long grid = units < sms ? units : sms;
  if (MODE == 1) grid = nB == 2 ? (grid > amax + 1 ? grid : amax + 1) : units;
  return grid;
}

// FP8 weights in tensor memory need G = 128 (whole-group stages in every K
// slice) and the B operand in shared memory; shared-memory bytes and buffers.
bool e4m3_plan(int MODE, int K, int G, int TT, int* nB, int* smem) {
  const int budget = device_max_smem_optin();
  const int kq = pick_kq(K, G);
  if (G != SK8 || kq == 0 || (K / kq) % SK8 != 0) return false;
  *nB = (MODE == 1 && smem_needed8(MODE, K, 2, TT) <= budget) ? 2 : 1;
  *smem = smem_needed8(MODE, K, *nB, TT);
  return *smem <= budget;
}

// fp8: both phases take the FP8 kernel (they share the h layout), else both
// the fp16 one.
template <int MODE>
cudaError_t launch_mode(const FfnParams& base, long long units, bool fp8, cudaStream_t stream) {
  FfnParams p = base;
  const int sms = device_sm_count();
  const int budget = device_max_smem_optin();
  const int TT = p.T == 1 ? 1 : kTok;
  p.lgG = ilog2(p.G);
  if (fp8) {
    int smem = 0;
    if (e4m3_plan(MODE, p.K, p.G, TT, &p.nB, &smem)) {
      p.kq = pick_kq(p.K, p.G);
      const int grid = (int)decode_grid(MODE, p.nB, units, (int)(units / (p.n_out / BM)) - 1, sms);
      if (TT == 1) return launch_e4m3<MODE, 1>(p, grid, smem, stream);
      return launch_e4m3<MODE, kTok>(p, grid, smem, stream);
    }
  }
  p.kq = pick_kq(p.K, p.G);
  const int Kq = p.K / p.kq;
  const int seg = Kq < p.G ? Kq : p.G;
  p.nB = (MODE == 1 && smem_needed(p.K, 2, TT) <= budget) ? 2 : 1;
  const int smem = smem_needed(p.K, p.nB, TT);
  const long long grid = decode_grid(MODE, p.nB, units, (int)(units / (p.n_out / BM)) - 1, sms);
  if (TT == 1) return launch_tt<MODE, 1>(p, seg, (int)grid, smem, stream);
  return launch_tt<MODE, kTok>(p, seg, (int)grid, smem, stream);
}

}  // namespace

bool ffn_decode_supported(const qre_layer_shape& s) {
  const int budget = device_max_smem_optin();
  const bool pow2 = s.group == 32 || s.group == 64 || s.group == 128;
  return pow2 && pick_kq(s.hidden, s.group) && pick_kq(s.inter, s.group) && (2 * s.inter) % BM == 0 &&
         s.hidden % BM == 0 && smem_needed(s.hidden, 1, kTok) <= budget && smem_needed(s.inter, 1, kTok) <= budget;
}

size_t ffn_ws_bytes(const qre_layer_shape& s, int T) {
  const long long pk = (long long)T * s.top_k;
  const long long amax = pk < s.n_experts ? pk : s.n_experts;
  return (size_t)(amax + 1) * 2 * kTok * s.inter * sizeof(__half);
}

size_t ffn_shared_ws_bytes(const qre_layer_shape& s, int) { return (size_t)2 * kTok * s.inter * sizeof(__half); }

cudaError_t launch_ffn_decode(const qre_layer_shape& s, int T, const uint16_t* x, const qre_slot* slots,
                              const int32_t* offsets, const int32_t* perm, const int32_t* active,
                              const int32_t* n_active, float* expert_out, void* ws, int* status,
                              cudaStream_t stream, int part) {
  if (!ffn_decode_supported(s)) return cudaErrorInvalidValue;
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
  p.hbuf = static_cast<__half*>(ws);
  p.expert_out = expert_out;
  p.status = status;
  p.part = part;
  p.host_cost = host_unit_cost();
  p.wait_ns = wait_limit_ns();
  p.stall_ns = test_stall_ns();
  const long long pk = (long long)T * s.top_k;
  p.amax = (int)(pk < s.n_experts ? pk : s.n_experts);
  p.K = s.hidden;
  p.n_out = 2 * s.inter;
  const int TT = T == 1 ? 1 : kTok;
  int nb = 0, sm = 0;
  const bool fp8 = e4m3_plan(0, s.hidden, s.group, TT, &nb, &sm) && e4m3_plan(1, s.inter, s.group, TT, &nb, &sm);
  // most groups a launch of this part can have (the grid is sized for them)
  const long long gmax = part == 2 ? 1 : (part == 1 ? p.amax : p.amax + 1);
  cudaError_t err = launch_mode<0>(p, gmax * (p.n_out / BM), fp8, stream);
  if (err != cudaSuccess) return err;

  p.K = s.inter;
  p.n_out = s.hidden;
  return launch_mode<1>(p, gmax * (p.n_out / BM), fp8, stream);
}

}  // namespace qre
