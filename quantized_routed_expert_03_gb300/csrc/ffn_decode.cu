// ffn_decode.cu -- bandwidth-bound fused dequant + SwiGLU expert FFN for T <= 8.
//
// The decode step of a routed MoE layer reads every byte of the union of the
// experts its tokens picked, plus the shared expert, once (glm53-flash-offload
// README, "Batched decode": streams share the per-layer expert union).  The work
// is a matrix-vector product per expert over 4-bit weights and the bound is HBM
// bandwidth, so the packed weights must stream at full rate while everything
// else stays under that.
//
// Layout of the work (5th-generation tensor cores, weights in tensor memory)
//   * A unit is 128 consecutive rows of one expert's matrix (UMMA M = 128; for
//     gate/up four blocks of 16 gate rows, each followed by its 16 up rows).
//     Units of all active experts and the shared expert are split into equal
//     contiguous ranges, one per CTA; one CTA per SM.
//   * The four warpgroups of a CTA split the reduction length K.  Thread r of a
//     warpgroup owns weight row r of the unit and tensor-memory lane r.  The
//     packed weights are stored in 4 KB chunks of 128 rows x 64 reduction
//     elements, so each warp's 16-byte loads cover 512 contiguous bytes; they are
//     prefetched up to four stages ahead, across unit boundaries (host-resident
//     experts are read the same way, zero-copy).  Each thread decodes its 64
//     nibbles per stage into fp16 pairs of exact integer codes and writes them
//     into its lane with tcgen05.st.
//   * One tcgen05.mma (A from tensor memory, B from shared memory, M=128, N=16,
//     K=16) is cheap for the tensor core but takes a warp on the order of a
//     hundred cycles to issue, while issues from different warps overlap.  So
//     every warp issues: stage g of a warpgroup is issued by its warp g mod 4,
//     once all four warps have arrived on the stage's mbarrier, and completes
//     on one commit per stage; no warp waits for the others between stages.
//   * B holds the tokens (T <= 8) in shared memory, 128-byte swizzled: rows 0-7
//     the fp16 high parts, rows 8-15 the fp16 remainders (x - high), so the
//     products stay accurate to about fp32.  The weights are exact codes, so the
//     only rounding is the fp32 accumulation.
//   * Every quantization group accumulates into its own buffer (four rotate); one
//     stage later the owning threads read it back (tcgen05.ld), add the two
//     halves and apply the group's fp16 scale in fp32.
//   * The four warpgroups' partial rows are added in fixed order (deterministic);
//     gate/up pairs each gate row with its up row (16 lanes apart, a shuffle) and
//     stores h = silu(g) * u as fp16 high part and remainder for the down kernel;
//     down writes the expert's output rows.
//   * Inside every group of 8 reduction elements the tokens and h are stored in
//     the order the nibble decode yields weight pairs (0,4,1,5,2,6,3,7), which
//     leaves every dot product unchanged.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

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
  int lgS;          // log2 of the accumulation segment: min(G, K / kq)
  int nB;           // B buffers in shared memory (down kernel: experts resident at once)
  int amax;         // largest possible number of active experts, min(E, T*k)
  const uint16_t* x;
  const qre_slot* slots;
  const int32_t* offsets;
  const int32_t* perm;
  const int32_t* active;
  const int32_t* n_active;
  __half* hbuf;       // [(amax+1)][2][kTok][I]: h high parts, then remainders (reordered in 8-groups)
  float* expert_out;  // [T*k + T][H]
  int* status;
};

struct Layout {
  int b_off, red_off, bar_off, grp_off, misc_off;
  size_t bytes;
};

__host__ __device__ inline Layout make_layout(int K, int nB) {
  Layout L;
  L.b_off = 0;                                          // nB x (BN x K fp16, swizzled; 1024-aligned)
  L.red_off = L.b_off + nB * K * BN * 2;                // 2 x kWG x BM x kTok fp32
  L.bar_off = L.red_off + 2 * kWG * BM * kTok * 4;      // a_full[kWG][3], done[kWG][3]
  L.grp_off = L.bar_off + kWG * 6 * 8;
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

// h of group a (high parts and remainders of the first T tokens) into B buffer `dst`.
__device__ __forceinline__ void load_h(uint8_t* dst, const __half* hbuf, int a, int I, int T) {
  const __half* hb = hbuf + (size_t)a * 2 * kTok * I;
  for (int i = threadIdx.x; i < 2 * T * (I / 8); i += blockDim.x) {
    const int j = i / (I / 8), g8 = i - j * (I / 8);
    const int row = j < T ? j : 8 + (j - T);   // part * 8 + token
    *reinterpret_cast<uint4*>(dst + b_offset(row, 8 * g8)) =
        *reinterpret_cast<const uint4*>(hb + (size_t)row * I + 8 * g8);
  }
}

// NA: A buffers per warpgroup.  Stage g's MMAs are issued during iteration g + 1
// by lane 0 of one warp of the warpgroup and complete on done[g mod NA].  MMAs
// from different threads are not ordered among themselves, so every stage of an
// accumulation segment is issued by the same warp: warp (segment mod 4).
// iteration g waits for stage g - NA, which frees A buffer g mod NA and makes
// the accumulation segments that ended in stage g - NA readable.  With
// NA = 3 a segment covers two stages (two D buffers suffice), with NA = 2 it
// covers at most one (four D buffers).
template <int MODE, int R, int NA>
__global__ void __launch_bounds__(kThreads, 1) ffn_decode_kernel(const FfnParams p) {
  constexpr int ND = NA == 3 ? 2 : 4;
  constexpr int SPS = NA == 3 ? 2 : 1;    // stages per accumulation segment (at least)
  constexpr int kD0 = 32 * NA;            // first D column of a warpgroup
  static_assert(32 * NA + 16 * ND <= kColsPerWG, "TMEM columns per warpgroup");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const Layout L = make_layout(p.K, p.nB);
  uint8_t* Bs = smem + L.b_off;
  const uint32_t b_bytes = (uint32_t)p.K * BN * 2;
  float* red = reinterpret_cast<float*>(smem + L.red_off);
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + L.bar_off);   // [kWG][3]: the 4 warps stored stage A
  uint64_t* done = a_full + kWG * 3;                                  // [kWG][3]: the stage's MMAs completed
  Group* groups = reinterpret_cast<Group*>(smem + L.grp_off);
  uint32_t* tmem_base_p = reinterpret_cast<uint32_t*>(smem + L.misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc_off + 4);

  int n_act = *p.n_active;
  n_act = n_act < 0 ? 0 : (n_act > p.amax ? p.amax : n_act);
  const int ngroups = n_act + 1;
  const int upe = p.n_out / BM;
  const int U = ngroups * upe;
  const int ub = (int)((long long)blockIdx.x * U / gridDim.x);
  const int ue = (int)((long long)(blockIdx.x + 1) * U / gridDim.x);
  if (ub >= ue) return;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wg = tid >> 7, r = tid & 127, wq = warp & 3;

  // per-CTA table of the groups (expert, pointers, output rows)
  for (int a = tid; a < ngroups; a += blockDim.x) {
    const int e = a < n_act ? __ldg(p.active + a) : p.E;
    const uint8_t* w = nullptr;
    const uint16_t* sc = nullptr;
    int flags = 0;
    if (e >= 0 && e <= p.E) {
      const qre_slot* sl = p.slots + e;
      w = MODE == 0 ? sl->w_gate_up : sl->w_down;
      sc = MODE == 0 ? sl->s_gate_up : sl->s_down;
      flags = (w && sc && ((reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(sc)) & 15) == 0) ? 1 : 0;
    }
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
    // B = tokens: rows 0-7 fp16 high parts, 8-15 remainders.  Rows of tokens
    // n >= T are left as they are: they only feed accumulator columns n, n + 8,
    // which nothing reads.
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
      *reinterpret_cast<uint4*>(Bs + b_offset(n, 8 * g8)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(Bs + b_offset(8 + n, 8 * g8)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  } else {
    // B = h of the first nB experts of this CTA's range
    const int a_last = (ue - 1) / upe;
    for (int j = 0; j < p.nB && a_first + j <= a_last; ++j) load_h(Bs + j * b_bytes, p.hbuf, a_first + j, p.I, p.T);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem_wg = *tmem_base_p + wg * kColsPerWG;
  const uint32_t tlane = (uint32_t)(32 * wq) << 16;   // this warp's TMEM lane quarter
  const int Kq = p.K / p.kq;
  const int nst = Kq / SK;
  const bool active_wg = wg < p.kq;
  const int k0 = wg * Kq;
  const int KS = p.K / SK;              // chunks per row block
  const int KG = p.K >> p.lgG;
  const int segL = 1 << p.lgS;
  const int spu = Kq >> p.lgS;          // accumulation segments per unit
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
  uint32_t sring[R];   // the stage's two scales (elements 0-31 low half, 32-63 high half)
  auto load_next = [&](uint4 (&dst)[2], uint32_t& sdst) {
    if (lptr) {
      dst[0] = __ldg(lptr + lst * (kChunk / 16));
      dst[1] = __ldg(lptr + lst * (kChunk / 16) + kChunk / 32);
      const int kk = k0 + lst * SK;
      sdst = (uint32_t)__ldg(lsp + (size_t)(kk >> p.lgG) * BM) |
             ((uint32_t)__ldg(lsp + (size_t)((kk + 32) >> p.lgG) * BM) << 16);
    } else {
      dst[0] = dst[1] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
      sdst = 0;
    }
    if (++lst == nst) {
      lst = 0;
      if (++lu < ue) cursor_unit(lu);
    }
  };
  if (active_wg) {
#pragma unroll
    for (int j = 0; j < R; ++j)
      if (lu < ue) load_next(ring[j], sring[j]);
  }

  float acc[kTok];
  // Adds the accumulation segments that end in unit stage `st` (scales sp) to
  // acc; the stage's MMAs have completed.
  auto readback = [&](int st, int ul, uint32_t sp) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int kk = st * SK + 16 * q;
      if (((kk + 16) & (segL - 1)) == 0) {
        const int d = (ul * spu + (kk >> p.lgS)) & (ND - 1);
        uint32_t dv[16];
        tmem_ld_32x32b_x16(tlane + tmem_wg + kD0 + 16 * d, dv);
        tmem_ld_wait();
        const float sc = __half2float(__ushort_as_half((unsigned short)(q < 2 ? sp & 0xFFFFu : sp >> 16)));
#pragma unroll
        for (int n = 0; n < kTok; ++n) acc[n] = fmaf(sc, __uint_as_float(dv[n]) + __uint_as_float(dv[n + 8]), acc[n]);
      }
    }
  };
  auto wait_done = [&](int gs) {
    mbar_wait_bounded(&done[wg * 3 + gs % NA], (gs / NA) & 1, abort_flag, p.status);
    __syncwarp();
    tc_fence_after();
  };
  // the warp that issues global stage gs
  auto issuer = [&](int gs) { return ((gs / SPS) & 3) == wq; };
  // lane 0 of the issuing warp: the four MMAs of global stage gs (unit stage st)
  auto issue = [&](int gs, int st, int ul, uint32_t bbase) {
    mbar_wait_bounded(&a_full[wg * 3 + gs % NA], (gs / NA) & 1, abort_flag, p.status);
    tc_fence_after();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int kk = st * SK + 16 * q;
      const int d = (ul * spu + (kk >> p.lgS)) & (ND - 1);
      const int kb = k0 + kk;
      const uint64_t bdesc = umma_desc_sw128(bbase + (uint32_t)((kb >> 6) * (BN * 128) + (kb & 63) * 2));
      umma_f16_tmem_a(tmem_wg + kD0 + 16 * d, tmem_wg + (gs % NA) * 32 + 8 * q, bdesc, idesc,
                      (kk & (segL - 1)) ? 1u : 0u);
    }
    umma_commit(&done[wg * 3 + gs % NA]);
  };

  int g = 0, buf = 0, cur_a = a_first, bsel = 0;
  for (int u = ub, ul = 0; u < ue; ++u, ++ul) {
    const int a = u / upe, m0 = (u - a * upe) * BM;
    const Group& gr = groups[a];
    if (!(gr.flags & 1) && tid == 0) set_status(p.status, QRE_DEV_NULL_SLOT);
    if constexpr (MODE == 1) {
      if (a != cur_a) {
        cur_a = a;
        const int la = a - a_first;
        bsel = la % p.nB;
        if (la >= p.nB) {   // buffer bsel held expert la - nB, whose MMAs all completed: refill it
          __syncthreads();
          load_h(Bs + bsel * b_bytes, p.hbuf, a, p.I, p.T);
          fence_proxy_async_smem();
          __syncthreads();
        }
      }
    }
    const uint32_t bbase = bbase0 + bsel * b_bytes;
#pragma unroll
    for (int n = 0; n < kTok; ++n) acc[n] = 0.f;

    if (active_wg) {
      uint32_t h1 = 0, h2 = 0, h3 = 0;   // scales of unit stages st-1, st-2, st-3
      for (int st0 = 0; st0 < nst; st0 += R) {
#pragma unroll
        for (int j = 0; j < R; ++j) {
          const int st = st0 + j, gs = g + st, ab = gs % NA;
          // (1) stage gs - NA completed: A buffer ab is free, its segments are readable
          if (gs >= NA) wait_done(gs - NA);
          // (2) decode 64 nibbles into 32 fp16 pairs of this row, store them in TMEM
          {
            const uint32_t wd[8] = {ring[j][0].x, ring[j][0].y, ring[j][0].z, ring[j][0].w,
                                    ring[j][1].x, ring[j][1].y, ring[j][1].z, ring[j][1].w};
            uint32_t av[32];
#pragma unroll
            for (int w = 0; w < 8; ++w) {
              uint32_t pr[4];
              decode_nibbles(wd[w], pr);
              av[4 * w + 0] = pr[0];
              av[4 * w + 1] = pr[1];
              av[4 * w + 2] = pr[2];
              av[4 * w + 3] = pr[3];
            }
            tmem_st_32x32b_x32(tlane + tmem_wg + ab * 32, av);
          }
          // (3) while the store drains: segments of unit stage st - NA
          if (st >= NA) readback(st - NA, ul, NA == 3 ? h3 : h2);
          // (4) scales of this stage, prefetch R stages ahead
          h3 = h2;
          h2 = h1;
          h1 = sring[j];
          if (lu < ue) load_next(ring[j], sring[j]);
          // (5) publish the stored A
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_full[wg * 3 + ab]);
          // (6) issue the previous stage if it is this warp's turn
          if (st >= 1 && issuer(gs - 1) && lane == 0) issue(gs - 1, st - 1, ul, bbase);
          __syncwarp();
        }
      }
      // unit end: issue the last stage, wait for the unit's last stages, read them back
      const int gl = g + nst - 1;
      if (issuer(gl) && lane == 0) issue(gl, nst - 1, ul, bbase);
      __syncwarp();
      const int first = nst > NA ? nst - NA : 0;
      for (int st = first; st < nst; ++st) {
        wait_done(g + st);
        const int back = nst - st;   // 1 = the last stage
        readback(st, ul, back == 1 ? h1 : (back == 2 ? h2 : h3));
      }
      tc_fence_before();
      float* rw = red + ((size_t)(buf * kWG + wg) * BM + r) * kTok;
#pragma unroll
      for (int n = 0; n < kTok; n += 4)
        *reinterpret_cast<float4*>(rw + n) = make_float4(acc[n], acc[n + 1], acc[n + 2], acc[n + 3]);
    }
    g += nst;
    __syncthreads();
    {
      // epilogue: thread (wg, r) finishes row r for tokens 2wg, 2wg + 1
      const int n0 = 2 * wg;
      float v0 = 0.f, v1 = 0.f;
      for (int w = 0; w < p.kq; ++w) {
        const float* rr = red + ((size_t)(buf * kWG + w) * BM + r) * kTok + n0;
        v0 += rr[0];
        v1 += rr[1];
      }
      if (gr.flags & 1) {
        if constexpr (MODE == 0) {
          // lanes 0-15 of each warp hold gate rows, lanes 16-31 the matching up rows
          const float up0 = __shfl_down_sync(0xffffffffu, v0, 16);
          const float up1 = __shfl_down_sync(0xffffffffu, v1, 16);
          const int f = m0 / 2 + 16 * (r >> 5) + (r & 15);
          const int pos = (f & ~7) | (((f & 3) << 1) | ((f >> 2) & 1));
          __half* hb = p.hbuf + (size_t)a * 2 * kTok * p.I;
          if ((lane & 16) == 0) {
            __half hh, hl;
            if (n0 < p.T) {
              split_half(silu_f32(v0) * up0, hh, hl);
              hb[(size_t)n0 * p.I + pos] = hh;
              hb[(size_t)(kTok + n0) * p.I + pos] = hl;
            }
            if (n0 + 1 < p.T) {
              split_half(silu_f32(v1) * up1, hh, hl);
              hb[(size_t)(n0 + 1) * p.I + pos] = hh;
              hb[(size_t)(kTok + n0 + 1) * p.I + pos] = hl;
            }
          }
        } else {
          const int q0 = gr.outq[n0], q1 = gr.outq[n0 + 1];
          if (q0 >= 0) p.expert_out[(size_t)q0 * p.H + m0 + r] = v0;
          if (q1 >= 0) p.expert_out[(size_t)q1 * p.H + m0 + r] = v1;
        }
      }
    }
    buf ^= 1;
  }

  tc_fence_before();
  __syncthreads();
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

int smem_needed(int K, int nB) {
  const size_t b = make_layout(K, nB).bytes;
  // at least ~120 KB so that no second CTA (and no second TMEM allocation) shares an SM
  return (int)(b > 120 * 1024 ? b : 120 * 1024);
}

template <int MODE, int R, int NA>
cudaError_t launch_r(const FfnParams& p, int grid, int smem, cudaStream_t stream) {
  cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(ffn_decode_kernel<MODE, R, NA>), smem);
  if (err != cudaSuccess) return err;
  ffn_decode_kernel<MODE, R, NA><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int MODE, int NA>
cudaError_t launch_na(const FfnParams& p, int nst, int grid, int smem, cudaStream_t stream) {
  if (nst % 4 == 0) return launch_r<MODE, 4, NA>(p, grid, smem, stream);
  if (nst % 2 == 0) return launch_r<MODE, 2, NA>(p, grid, smem, stream);
  return launch_r<MODE, 1, NA>(p, grid, smem, stream);
}

template <int MODE>
cudaError_t launch_mode(const FfnParams& base, int grid, cudaStream_t stream) {
  FfnParams p = base;
  p.kq = pick_kq(p.K, p.G);
  const int Kq = p.K / p.kq;
  p.lgG = ilog2(p.G);
  p.lgS = ilog2(Kq < p.G ? Kq : p.G);
  const int budget = device_max_smem_optin();
  p.nB = (MODE == 1 && smem_needed(p.K, 2) <= budget) ? 2 : 1;
  const int smem = smem_needed(p.K, p.nB);
  const int nst = Kq / SK;
  // segments of two stages (G = 128 within a K slice): three A buffers, two D buffers
  if (p.lgS == 7) return launch_na<MODE, 3>(p, nst, grid, smem, stream);
  return launch_na<MODE, 2>(p, nst, grid, smem, stream);
}

}  // namespace

bool ffn_decode_supported(const qre_layer_shape& s) {
  const int budget = device_max_smem_optin();
  const bool pow2 = s.group == 32 || s.group == 64 || s.group == 128;
  return pow2 && pick_kq(s.hidden, s.group) && pick_kq(s.inter, s.group) && (2 * s.inter) % BM == 0 &&
         s.hidden % BM == 0 && smem_needed(s.hidden, 1) <= budget && smem_needed(s.inter, 1) <= budget;
}

size_t ffn_ws_bytes(const qre_layer_shape& s, int T) {
  const long long pk = (long long)T * s.top_k;
  const long long amax = pk < s.n_experts ? pk : s.n_experts;
  return (size_t)(amax + 1) * 2 * kTok * s.inter * sizeof(__half);
}

cudaError_t launch_ffn_decode(const qre_layer_shape& s, int T, const uint16_t* x, const qre_slot* slots,
                              const int32_t* offsets, const int32_t* perm, const int32_t* active,
                              const int32_t* n_active, float* expert_out, void* ws, int* status,
                              cudaStream_t stream) {
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
  const long long pk = (long long)T * s.top_k;
  p.amax = (int)(pk < s.n_experts ? pk : s.n_experts);
  const int sms = device_sm_count();

  p.K = s.hidden;
  p.n_out = 2 * s.inter;
  long long units = (long long)(p.amax + 1) * (p.n_out / BM);
  cudaError_t err = launch_mode<0>(p, (int)(units < sms ? units : sms), stream);
  if (err != cudaSuccess) return err;

  p.K = s.inter;
  p.n_out = s.hidden;
  units = (long long)(p.amax + 1) * (p.n_out / BM);
  return launch_mode<1>(p, (int)(units < sms ? units : sms), stream);
}

}  // namespace qre
