// ffn_prefill.cu -- the expert FFN for T > 8 as a grouped GEMM on tcgen05/TMEM.
//
// Prefill pushes thousands of tokens through one MoE layer (the RTX PRO 6000
// recipe prefills in chunks of 4096 tokens, the glm53-flash-offload README in
// chunks of 8192); each expert sees ~T*k/E tokens, enough to make its FFN a
// dense contraction.  The weights are the M side of the MMA (128 output rows
// per tile), the expert's tokens the N side (up to 256 per tile): D[feature,
// token] += W[feature, k] * X[token, k].
//
// Three kernels:
//   gather   Xg[q] = fp16(x[token of pick perm[q]]) for the T*k sorted picks,
//            then Xg[T*k + t] = fp16(x[t]) for the shared expert.  Every
//            expert's tokens become a contiguous row range of Xg.  Inside each
//            group of 8 reduction elements the order is (0,4,1,5,2,6,3,7), the
//            order in which the 4-bit decode yields weight pairs; h16 uses the
//            same order, so no operand needs a permute.
//   GEMM 1   per tile (expert, 128 rows of the interleaved gate/up matrix, <=256
//            tokens); the epilogue pairs each gate row with its up row (they sit
//            16 TMEM lanes apart) and writes h = silu(g) * u as fp16 to h16.
//   GEMM 2   per tile (expert, 128 rows of W_down, <=256 tokens) from h16 rows;
//            the epilogue writes fp32 rows of expert_out (row q = pick at sorted
//            position q; row T*k + t = shared expert for token t).
// Both GEMMs are one persistent warp-specialised kernel, one CTA per SM:
//   warp 0      TMA loads of the token operand (128-byte swizzle) into a 4-stage ring
//   warp 1      allocates 512 TMEM columns (two 128x256 fp32 accumulators) and
//               issues tcgen05.mma (M=128, N<=256, K=16) from one thread
//   warp 18     bulk-copies each stage's packed weights (one 4 KB chunk of the
//               tiled format) and its group scales into a ring of its own in
//               shared memory (host-mapped experts: plain loads by the warp)
//   warps 2-9   dequantize the weight operand from that ring: two threads per
//               row each decode 32 nibbles per stage, multiply by the group
//               scale in fp16 and store the 128-byte swizzled rows the MMA
//               expects
//   warps 10-17 epilogue: tcgen05.ld of the finished accumulator while the MMA
//               warp fills the other one; two warps per TMEM lane quarter take
//               the tile's 32-token column chunks in turn.  GEMM 1 stages each
//               chunk's h through a small shared-memory transpose so that every
//               lane stores one token's 16 features as two 16-byte writes.
// Operands are fp16 (x bf16 -> fp16 is exact in fp16's normal range; dequantized
// weights and h are rounded to fp16), accumulation fp32.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace qre {
namespace {

constexpr int BM = 128;                 // weight rows per tile
constexpr int BN = 256;                 // tokens per tile (max)
constexpr int BK = 64;                  // reduction elements per stage: one 128-byte swizzle row
constexpr int NSTAGE = 4;
constexpr int A_STAGE = BM * BK * 2;    // 16 KB
constexpr int B_STAGE = BN * BK * 2;    // 32 KB
constexpr int kWarps = 19;          // 0 TMA, 1 MMA, 2-9 dequant, 10-17 epilogue, 18 weight copies
constexpr int kEpiWarps = 8;
constexpr int kEpiScratch = 32 * 32;   // bytes per epilogue warp: 32 tokens x 16 fp16 features
constexpr int kDqWarps = 8;
constexpr int kWChunk = BM * BK / 2;   // packed bytes of one stage: the 4 KB chunk (m0 / 128, kb)
constexpr int kWSlot = kWChunk + 512;  // + the stage's group scales (two groups of 128 rows at most)
constexpr int kMaxWStages = 8;
constexpr int kDqThreads = 256;
constexpr int kThreads = kWarps * 32;
constexpr int kTmemCols = 512;
constexpr int kAccCols = 256;

struct PrefillParams {
  int H, I, E, k, G, T;
  int K;        // reduction length: H (gate/up) or I (down)
  int n_out;    // weight rows: 2I or H
  int amax;     // largest possible number of active experts
  int part;     // groups: 0 routed + shared, 1 routed only, 2 shared only
  int xrow0;    // expert_out row of Xg / h16 row 0 (P for the shared-only part, which keeps its own)
  const qre_slot* slots;
  const int32_t* offsets;
  const int32_t* active;
  const int32_t* n_active;
  __half* h16;         // [T*k + T][I]
  float* expert_out;   // [T*k + T][H]
  int* status;
  uint64_t wait_ns;    // limit of the pipeline waits
  uint64_t stall_ns;   // test hook: the TMA warp of CTA 0 delays its first load (0 = off)
  int wst;             // stages of the weight ring (2 .. kMaxWStages, what shared memory holds)
};

struct SmemLayout {
  static constexpr int a_off = 0;
  static constexpr int b_off = NSTAGE * A_STAGE;
  static constexpr int bar_off = b_off + NSTAGE * B_STAGE;
  // full_a[NS], full_b[NS], empty[NS], acc_full[2], acc_empty[2], wfull[8], wempty[8]
  static constexpr int nbars = 3 * NSTAGE + 4 + 2 * kMaxWStages;
  static constexpr int misc_off = bar_off + nbars * 8;   // tmem base, abort flag, group count, tile count
  static constexpr int epi_off = misc_off + 16;                 // kEpiWarps x kEpiScratch (16-byte aligned)
  static constexpr int tab_off = epi_off + kEpiWarps * kEpiScratch;
  // the weight ring follows the group table, 128-byte aligned
  __host__ __device__ static int ring_off(int E) { return (tab_off + 3 * (E + 2) * 4 + 127) & ~127; }
  static size_t bytes(int E, int wst) { return (size_t)ring_off(E) + (size_t)wst * kWSlot + 1024; }
};

// ---------------------------------------------------------------- gather

// Rows q in [q0, q1) of the pick order (q >= T*k: the shared expert's token q - T*k),
// written at Xg row q - q0.  A thread converts kGatherChunks 16-byte pieces of
// one row (columns c0 + j * H / kGatherChunks): one perm load and all
// its token loads in flight together, every store coalesced across the warp.
constexpr int kGatherChunks = 4;
__global__ void __launch_bounds__(256) gather_x_kernel(int T, int H, int k, long long q0, long long q1,
                                                       const uint16_t* __restrict__ x,
                                                       const int32_t* __restrict__ perm, __half* __restrict__ xg,
                                                       int* status) {
  grid_dependency_wait();   // perm, from the dispatch
  grid_dependents_launch();
  const long long P = (long long)T * k;
  const int tpr = H / (8 * kGatherChunks);   // threads per row
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (q1 - q0) * tpr) return;
  const long long qi = i / tpr;               // row within this launch's range
  const int c0 = (int)(i - qi * tpr) * 8;     // first of the thread's columns
  const long long q = q0 + qi;
  const int t = q < P ? __ldg(perm + q) / k : (int)(q - P);
  uint4 v[kGatherChunks];
#pragma unroll
  for (int j = 0; j < kGatherChunks; ++j)
    v[j] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H + c0 + j * tpr * 8));
  bool bad = false;
#pragma unroll
  for (int j = 0; j < kGatherChunks; ++j) {
    float f[8];
    f[0] = bf16_bits_to_float(v[j].x & 0xFFFFu); f[1] = bf16_bits_to_float(v[j].x >> 16);
    f[2] = bf16_bits_to_float(v[j].y & 0xFFFFu); f[3] = bf16_bits_to_float(v[j].y >> 16);
    f[4] = bf16_bits_to_float(v[j].z & 0xFFFFu); f[5] = bf16_bits_to_float(v[j].z >> 16);
    f[6] = bf16_bits_to_float(v[j].w & 0xFFFFu); f[7] = bf16_bits_to_float(v[j].w >> 16);
    uint32_t o[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {   // pair order (x_m, x_{m+4}), the order the weight decode produces
      const __half2 h = __floats2half2_rn(f[m], f[m + 4]);
      bad |= __hisinf(__low2half(h)) || __hisinf(__high2half(h));
      o[m] = h2_as_u32(h);
    }
    *reinterpret_cast<uint4*>(xg + (size_t)(q - q0) * H + c0 + j * tpr * 8) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (bad) set_status(status, QRE_DEV_FP16_RANGE);
}

// ---------------------------------------------------------------- GEMM

struct Tile {
  int g;       // group: active index, or n_act for the shared expert
  int e;       // expert id (E = shared)
  int row0;    // first row of the group in Xg / h16 / expert_out
  int M;       // tokens in the group
  int m0;      // first weight row
  int n0;      // first token of the tile within the group
  int n;       // tokens in this tile
};

__device__ __forceinline__ Tile decode_tile(int t, int ngroups, const int* tstart, const int* row0, const int* gm,
                                            int mt_per, int n_act, const int32_t* active, int E) {
  int lo = 0, hi = ngroups - 1;
  while (lo < hi) {  // last g with tstart[g] <= t
    const int mid = (lo + hi + 1) >> 1;
    if (tstart[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  Tile tl;
  tl.g = lo;
  tl.e = lo < n_act ? __ldg(active + lo) : E;
  tl.row0 = row0[lo];
  tl.M = gm[lo];
  const int local = t - tstart[lo];
  const int nt = local / mt_per, mt = local - nt * mt_per;
  tl.m0 = mt * BM;
  tl.n0 = nt * BN;
  tl.n = min(BN, tl.M - tl.n0);
  return tl;
}

// Eight nibbles (k .. k+7 from the low end of w) -> eight fp16 values q*s in
// pair order (q0,q4) (q1,q5) (q2,q6) (q3,q7).  The token operand (gather) and h
// (GEMM 1 epilogue) are stored with the same order inside every group of 8
// reduction elements, so the products pair up as in natural order.
__device__ __forceinline__ uint4 dequant8(uint32_t w, __half2 s2) {
  uint32_t p[4];
  decode_nibbles(w, p);
  uint4 r;
  r.x = h2_as_u32(__hmul2(u32_as_h2(p[0]), s2));
  r.y = h2_as_u32(__hmul2(u32_as_h2(p[1]), s2));
  r.z = h2_as_u32(__hmul2(u32_as_h2(p[2]), s2));
  r.w = h2_as_u32(__hmul2(u32_as_h2(p[3]), s2));
  return r;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) prefill_gemm_kernel(const PrefillParams p,
                                                                   const __grid_constant__ CUtensorMap tmap_b) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* As = smem + SmemLayout::a_off;
  uint8_t* Bs = smem + SmemLayout::b_off;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SmemLayout::bar_off);
  uint64_t* full_a = bars;
  uint64_t* full_b = bars + NSTAGE;
  uint64_t* empty = bars + 2 * NSTAGE;
  uint64_t* acc_full = bars + 3 * NSTAGE;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* wfull = acc_empty + 2;           // [wst]: a stage's weights and scales landed
  uint64_t* wempty = wfull + kMaxWStages;    // [wst]: the dequantizing warps read them
  uint8_t* wring = smem + SmemLayout::ring_off(p.E);
  uint32_t* tmem_base_p = reinterpret_cast<uint32_t*>(smem + SmemLayout::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SmemLayout::misc_off + 4);
  int* counts_p = reinterpret_cast<int*>(smem + SmemLayout::misc_off + 8);  // ngroups, ntiles
  int* tstart = reinterpret_cast<int*>(smem + SmemLayout::tab_off);
  int* grow0 = tstart + (p.E + 2);
  int* gM = grow0 + (p.E + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = p.T * p.k;
  const int mt_per = p.n_out / BM;
  const int KB = p.K / BK;

  // groups: the active experts (parts 0, 1), then the shared one (parts 0, 2)
  int n_act = p.part == 2 ? 0 : *p.n_active;
  n_act = n_act < 0 ? 0 : (n_act > p.amax ? p.amax : n_act);
  const int ngroups = n_act + (p.part == 1 ? 0 : 1);

  // group table: rows, tokens and first tile of every group (one warp)
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < ngroups; base += 32) {
      const int g = base + lane;
      int tiles = 0;
      if (g < ngroups) {
        int r0, m;
        if (g < n_act) {
          const int e = __ldg(p.active + g);
          r0 = __ldg(p.offsets + e);
          m = __ldg(p.offsets + e + 1) - r0;
        } else {
          r0 = P;
          m = p.T;
        }
        grow0[g] = r0;
        gM[g] = m;
        tiles = ((m + BN - 1) / BN) * mt_per;
      }
      int inc = tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      if (g < ngroups) tstart[g] = carry + inc - tiles;
      carry += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) {
      tstart[ngroups] = carry;
      counts_p[0] = ngroups;
      counts_p[1] = carry;
    }
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full_a[s], kDqThreads);
      mbar_init(&full_b[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiWarps * 32);
    }
    for (int w = 0; w < p.wst; ++w) {
      mbar_init(&wfull[w], 1);
      mbar_init(&wempty[w], kDqWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(tmem_base_p, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_p;
  const int ntiles = counts_p[1];

  if (warp == 0) {
    // ---------------- token operand: TMA
    if (lane == 0) {
      if (p.stall_ns && blockIdx.x == 0) debug_stall(p.stall_ns);
      int it = 0;
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const Tile tl = decode_tile(t, ngroups, tstart, grow0, gM, mt_per, n_act, p.active, p.E);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % NSTAGE;
          if (!mbar_wait_bounded(&empty[s], ((it / NSTAGE) & 1) ^ 1, abort_flag, p.status, p.wait_ns)) goto b_done;
          mbar_arrive_expect_tx(&full_b[s], B_STAGE);
          tma_load_2d(Bs + (size_t)s * B_STAGE, &tmap_b, kb * BK, tl.row0 + tl.n0 - p.xrow0, &full_b[s]);
        }
      }
    b_done:
      const int first = it > NSTAGE ? it - NSTAGE : 0;
      for (int j = first; j < it; ++j)
        mbar_wait_drain(&full_b[j % NSTAGE], (j / NSTAGE) & 1, p.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issue (one thread)
    if (lane == 0) {
      int it = 0, lt = 0, last = -1;
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++lt) {
        const Tile tl = decode_tile(t, ngroups, tstart, grow0, gM, mt_per, n_act, p.active, p.E);
        const int buf = lt & 1;
        if (!mbar_wait_bounded(&acc_empty[buf], ((lt >> 1) & 1) ^ 1, abort_flag, p.status, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * kAccCols;
        const int n_mma = (tl.n + 15) & ~15;
        const uint32_t idesc = umma_idesc_f16(BM, n_mma);
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % NSTAGE;
          const uint32_t ph = (it / NSTAGE) & 1;
          if (!mbar_wait_bounded(&full_a[s], ph, abort_flag, p.status, p.wait_ns) ||
              !mbar_wait_bounded(&full_b[s], ph, abort_flag, p.status, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a0 = umma_desc_sw128(smem_addr(As + (size_t)s * A_STAGE));
          const uint64_t b0 = umma_desc_sw128(smem_addr(Bs + (size_t)s * B_STAGE));
#pragma unroll
          for (int j = 0; j < BK / 16; ++j)  // advance 16 elements = 32 bytes inside the swizzle row
            umma_f16(d_tmem, a0 + (uint64_t)(2 * j), b0 + (uint64_t)(2 * j), idesc, (kb | j) != 0);
          umma_commit(&empty[s]);
        }
        umma_commit(&acc_full[buf]);
        last = lt;
        if (!ok) break;
      }
      // TMEM is freed below: every MMA issued here must have completed first
      if (last >= 0) mbar_wait_drain(&acc_full[last & 1], (last >> 1) & 1, p.status);
    }
  } else if (warp < 10) {
    // ---------------- weight operand: dequantize into the swizzled stage
    const int dq = threadIdx.x - 64;        // 0..255
    const int r = dq & 127;                 // row within the tile
    const int hf = dq >> 7;                 // which 32 of the stage's 64 reduction elements
    const int sw = r & 7;
    const uint32_t row_off = (uint32_t)(r >> 3) * 1024 + (uint32_t)sw * 128;
    // in a ring slot: this thread's 16 bytes of the chunk (2048 * hf + 16 * r)
    // and its row's scale in the stage's first or second group
    const int wofs = 2048 * hf + 16 * r;
    const int sofs = kWChunk + ((32 * hf) / p.G) * (BM * 2) + 2 * r;
    int it = 0, w = 0, wph = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const Tile tl = decode_tile(t, ngroups, tstart, grow0, gM, mt_per, n_act, p.active, p.E);
      const qre_slot* sl = p.slots + tl.e;
      const uint8_t* wb = MODE == 0 ? sl->w_gate_up : sl->w_down;
      const uint16_t* sb = MODE == 0 ? sl->s_gate_up : sl->s_down;
      const bool valid = wb && sb && ((reinterpret_cast<uintptr_t>(wb) | reinterpret_cast<uintptr_t>(sb)) & 15) == 0;
      if (!valid && dq == 0) set_status(p.status, QRE_DEV_NULL_SLOT);
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % NSTAGE;
        const bool go = mbar_wait_bounded(&empty[s], ((it / NSTAGE) & 1) ^ 1, abort_flag, p.status, p.wait_ns);
        const bool wok = mbar_wait_bounded(&wfull[w], wph, abort_flag, p.status, p.wait_ns);
        if (go && wok) {
          const uint8_t* slot = wring + w * kWSlot;
          uint4 wv = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
          unsigned short sv = 0;
          if (valid) {
            wv = *reinterpret_cast<const uint4*>(slot + wofs);
            sv = *reinterpret_cast<const unsigned short*>(slot + sofs);
          }
          const __half2 s2 = __half2half2(__ushort_as_half(sv));
          const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
          uint8_t* stage = As + (size_t)s * A_STAGE + row_off;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 v = dequant8(words[c], s2);
            *reinterpret_cast<uint4*>(stage + (((4 * hf + c) ^ sw) << 4)) = v;
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&wempty[w]);   // this warp is done with the ring slot
        mbar_arrive(&full_a[s]);
        if (++w == p.wst) {
          w = 0;
          wph ^= 1;
        }
      }
    }
  } else if (warp == 18) {
    // ---------------- weight copies: the packed chunk and group scales of each stage
    int it = 0, w = 0, wph = 0;
    const int KG = p.K / p.G;
    const uint32_t sbytes = 256u * (p.G < BK ? (uint32_t)(BK / p.G) : 1u);   // scales of the stage's groups
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const Tile tl = decode_tile(t, ngroups, tstart, grow0, gM, mt_per, n_act, p.active, p.E);
      const qre_slot* sl = p.slots + tl.e;
      const uint8_t* wb = MODE == 0 ? sl->w_gate_up : sl->w_down;
      const uint16_t* sb = MODE == 0 ? sl->s_gate_up : sl->s_down;
      const bool valid = wb && sb && ((reinterpret_cast<uintptr_t>(wb) | reinterpret_cast<uintptr_t>(sb)) & 15) == 0;
      const bool host = sl->tier != 0;
      const uint8_t* wsrc = valid ? wb + (size_t)(tl.m0 / BM) * (p.K / BK) * kWChunk : nullptr;
      const uint16_t* ssrc = valid ? sb + (size_t)(tl.m0 / BM) * KG * BM : nullptr;
      for (int kb = 0; kb < KB; ++kb, ++it) {
        // warp-uniform exit (the host-mapped path below synchronizes the warp)
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&wempty[w], wph ^ 1, abort_flag, p.status, p.wait_ns)))
          goto w_done;
        uint8_t* dst = wring + w * kWSlot;
        const size_t g0 = (size_t)(kb * BK) / p.G;   // first group of the stage
        if (valid && !host) {
          if (lane == 0) {
            mbar_arrive_expect_tx(&wfull[w], kWChunk + sbytes);
            bulk_copy_g2s(dst, wsrc + (size_t)kb * kWChunk, kWChunk, &wfull[w]);
            bulk_copy_g2s(dst + kWChunk, ssrc + g0 * BM, sbytes, &wfull[w]);
          }
        } else {
          if (valid) {   // host-mapped expert: the warp copies with plain 16-byte loads
            const uint4* src = reinterpret_cast<const uint4*>(wsrc + (size_t)kb * kWChunk);
            for (int i = lane; i < kWChunk / 16; i += 32) reinterpret_cast<uint4*>(dst)[i] = __ldg(src + i);
            const uint4* ss = reinterpret_cast<const uint4*>(ssrc + g0 * BM);
            for (int i = lane; i < (int)sbytes / 16; i += 32) reinterpret_cast<uint4*>(dst + kWChunk)[i] = __ldg(ss + i);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&wfull[w]);
        }
        if (++w == p.wst) {
          w = 0;
          wph ^= 1;
        }
      }
    }
  w_done:
    // copies still in flight land before the CTA exits
    if (lane == 0) {
      const int first = it > p.wst ? it - p.wst : 0;
      for (int j = first; j < it; ++j) mbar_wait_drain(&wfull[j % p.wst], (j / p.wst) & 1, p.status);
    }
  } else {
    // ---------------- epilogue
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int half = (warp - 10) >> 2;    // which 32-token chunks: even (0) or odd (1)
    // GEMM 1: this warp's transpose scratch, 32 rows (tokens) of 32 bytes (16
    // features); the two 16-byte halves of row j are swapped when (j >> 2) & 1,
    // which keeps both the 2-byte writes and the 16-byte reads conflict-free.
    uint8_t* scratch = smem + SmemLayout::epi_off + (warp - 10) * kEpiScratch;
    int lt = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++lt) {
      const Tile tl = decode_tile(t, ngroups, tstart, grow0, gM, mt_per, n_act, p.active, p.E);
      const int buf = lt & 1;
      // warp-uniform: the chunk loop below uses whole-warp shuffles
      const bool have =
          __all_sync(0xffffffffu, mbar_wait_bounded(&acc_full[buf], (lt >> 1) & 1, abort_flag, p.status, p.wait_ns));
      tc_fence_after();
      if (have) {
        const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + buf * kAccCols;
        bool overflow = false;
        for (int c0 = 32 * half; c0 < tl.n; c0 += 64) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tbase + c0, v);
          tmem_ld_wait();
          if constexpr (MODE == 0) {
            // lanes 0-15 hold gate rows, lanes 16-31 the matching up rows;
            // feature f = lane of the warp's 16 (group-of-8 order: i at 2(i%4) + i/4)
            const int f = lane & 15;
            const int pos = (f & 8) | ((f & 3) << 1) | ((f >> 2) & 1);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float up = __shfl_down_sync(0xffffffffu, __uint_as_float(v[j]), 16);
              if (lane < 16) {
                const float g = __uint_as_float(v[j]);
                const __half hh = __float2half_rn(__fdividef(g, 1.0f + __expf(-g)) * up);
                overflow |= __hisinf(hh) && c0 + j < tl.n;
                const int sw = (pos >> 3) ^ ((j >> 2) & 1);
                *reinterpret_cast<__half*>(scratch + j * 32 + sw * 16 + (pos & 7) * 2) = hh;
              }
            }
            __syncwarp();
            // lane L: token c0 + L, the warp's 16 features (32 bytes) in h16 order
            const int n = c0 + lane;
            if (n < tl.n) {
              const int s0 = (lane >> 2) & 1;
              const uint4 lo = *reinterpret_cast<const uint4*>(scratch + lane * 32 + s0 * 16);
              const uint4 hi = *reinterpret_cast<const uint4*>(scratch + lane * 32 + (s0 ^ 1) * 16);
              uint4* dst = reinterpret_cast<uint4*>(p.h16 + (size_t)(tl.row0 + tl.n0 + n - p.xrow0) * p.I +
                                                    tl.m0 / 2 + 16 * q);
              dst[0] = lo;
              dst[1] = hi;
            }
            __syncwarp();
          } else {
            const int col = tl.m0 + 32 * q + lane;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int n = c0 + j;
              if (n < tl.n) p.expert_out[(size_t)(tl.row0 + tl.n0 + n) * p.H + col] = __uint_as_float(v[j]);
            }
          }
        }
        if (MODE == 0 && __any_sync(0xffffffffu, overflow) && lane == 0) set_status(p.status, QRE_DEV_FP16_RANGE);
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[buf]);
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------- host

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D fp16 row-major [rows][cols] -> boxes of 64 columns x 256 rows, 128-byte swizzle.
bool make_tmap(CUtensorMap* m, const void* base, long long rows, int cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {BK, BN};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

}  // namespace

bool make_tmap_bf16(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t ffn_prefill_ws_bytes(const qre_layer_shape& s, int T) {
  const size_t rows = (size_t)T * s.top_k + T;
  return align256(rows * s.hidden * 2) + align256(rows * s.inter * 2);
}

size_t ffn_prefill_shared_ws_bytes(const qre_layer_shape& s, int T) {
  return align256((size_t)T * s.hidden * 2) + align256((size_t)T * s.inter * 2);
}

// Weight-ring stages that fit next to everything else in shared memory.
int weight_stages(int E) {
  const long long spare = (long long)device_max_smem_optin() - (long long)SmemLayout::bytes(E, 0);
  const long long n = spare / kWSlot;
  return (int)(n > kMaxWStages ? kMaxWStages : n);
}

bool ffn_prefill_supported(const qre_layer_shape& s) {
  return s.hidden % BK == 0 && s.inter % BK == 0 && (2 * s.inter) % BM == 0 && s.hidden % BM == 0 &&
         weight_stages(s.n_experts) >= 2;
}

cudaError_t launch_ffn_prefill(const qre_layer_shape& s, int T, const uint16_t* x, const qre_slot* slots,
                               const int32_t* offsets, const int32_t* perm, const int32_t* active,
                               const int32_t* n_active, float* expert_out, void* ws, int* status,
                               cudaStream_t stream, int part) {
  const long long P = (long long)T * s.top_k;
  // Xg / h16 rows: the pick rows and/or the shared rows of this part; the
  // shared-only part keeps its T rows in a workspace of its own
  const long long q0 = part == kFfnShared ? P : 0, q1 = part == kFfnRouted ? P : P + T;
  const long long rows = part == kFfnShared ? T : P + T;
  __half* xg = static_cast<__half*>(ws);
  __half* h16 = reinterpret_cast<__half*>(static_cast<uint8_t*>(ws) + align256((size_t)rows * s.hidden * 2));

  {
    const long long n = (q1 - q0) * (s.hidden / (8 * kGatherChunks));
    if (n > 0) {
      cudaError_t e = launch_dependent(gather_x_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, stream, T,
                                       s.hidden, s.top_k, q0, q1, x, perm, xg, status);
      if (e != cudaSuccess) return e;
    }
  }
  CUtensorMap tx, th;
  if (!make_tmap(&tx, xg, rows, s.hidden) || !make_tmap(&th, h16, rows, s.inter)) return cudaErrorInvalidValue;

  PrefillParams p{};
  p.H = s.hidden;
  p.I = s.inter;
  p.E = s.n_experts;
  p.k = s.top_k;
  p.G = s.group;
  p.T = T;
  p.amax = (int)(P < s.n_experts ? P : s.n_experts);
  p.slots = slots;
  p.offsets = offsets;
  p.active = active;
  p.n_active = n_active;
  p.h16 = h16;
  p.expert_out = expert_out;
  p.status = status;
  p.part = part;
  p.xrow0 = (int)q0;
  p.wait_ns = wait_limit_ns();
  p.stall_ns = test_stall_ns();
  p.wst = weight_stages(s.n_experts);
  const size_t smem = SmemLayout::bytes(s.n_experts, p.wst);
  const int grid = device_sm_count();

  p.K = s.hidden;
  p.n_out = 2 * s.inter;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(prefill_gemm_kernel<0>), (int)smem);
  if (e != cudaSuccess) return e;
  prefill_gemm_kernel<0><<<grid, kThreads, smem, stream>>>(p, tx);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  p.K = s.inter;
  p.n_out = s.hidden;
  e = ensure_smem_limit(reinterpret_cast<const void*>(prefill_gemm_kernel<1>), (int)smem);
  if (e != cudaSuccess) return e;
  prefill_gemm_kernel<1><<<grid, kThreads, smem, stream>>>(p, th);
  return cudaGetLastError();
}

}  // namespace qre
