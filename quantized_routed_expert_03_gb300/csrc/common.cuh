// common.cuh -- device helpers shared by the library's kernels (sm_103a).
//
// Inline PTX for mbarriers, cp.async copies, programmatic launch control, the
// 4-bit decodes, the global timer used to bound every wait, and the device
// status word.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/qre.h"

namespace qre {

// Every spin-wait in this library gives up after a limit, records
// QRE_DEV_TIMEOUT in the status word and lets the kernel finish.  The pipeline
// waits take the limit as a kernel parameter (this value unless a test lowers
// it, qre_debug_wait_test); the waits that must end before tensor memory is
// freed always use this value.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void set_status(int* status, int bits) {
  if (status) atomicOr(status, bits);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase of `bar` with the given parity, for at most limit_ns
// from the first failed poll.  Gives up early when *abort is set by another
// warp; on expiry sets *abort and QRE_DEV_TIMEOUT.  Returns true when the phase
// completed.
// The polling loop is out of line: the hot loops that wait on barriers keep
// only the first poll and a call, which keeps their code small enough for the
// instruction cache.
// Each poll may suspend the thread until the phase completes or for at most
// about 1 us (the suspend-time hint), so the deadline is checked at that
// granularity whatever the hardware's own suspend limit is.
__device__ __forceinline__ bool mbar_try_wait_1us(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(1000u)
      : "memory");
  return done != 0;
}
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort, int* status,
                                                   uint64_t limit_ns) {
  const uint64_t deadline = global_timer_ns() + limit_ns;
  while (!mbar_try_wait_1us(bar, parity)) {
    if (abort && *abort) return false;
    if (global_timer_ns() > deadline) {
      if (abort) *abort = 1;
      set_status(status, QRE_DEV_TIMEOUT);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort, int* status,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort, status, limit_ns);
}
// The wait before tensor memory is freed or a kernel exits with copies in
// flight: not cut short by the abort flag, and always the full kWaitLimitNs
// (what it waits for, issued tensor-core work or bulk copies, completes on its
// own).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, nullptr, status, kWaitLimitNs);
}

// Test hook (qre_debug_wait_test): spins for ns nanoseconds of the global timer.
static __device__ __noinline__ void debug_stall(uint64_t ns) {
  const uint64_t end = global_timer_ns() + ns;
  while (global_timer_ns() < end) {
  }
}

// ---------------------------------------------------------------- async copies

// 16-byte asynchronous copy global -> shared (cached in L2 only).
__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
// Closes this thread's current group of cp.async copies (an empty group if it
// issued none), and waits until at most N of its groups are still in flight.
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ unsigned short lds16(uint32_t addr) {
  unsigned short v;
  asm("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// ---------------------------------------------------------------- PDL

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- 4-bit decode

__device__ __forceinline__ uint32_t h2_as_u32(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }

// Decodes the eight nibbles u0..u7 of one 32-bit word (u_i at bits 4i..4i+3)
// into four fp16 pairs holding the signed codes q = u - 8, exactly:
//   p[0] = (q0, q4), p[1] = (q1, q5), p[2] = (q2, q6), p[3] = (q3, q7)
// (low half first).  OR-ing a nibble into the mantissa of fp16 1024 gives
// 1024 + u (low nibble) or 1024 + 16u (high nibble of a byte); one subtract or
// one fused multiply-add removes the offset.  All steps are exact in fp16.
__device__ __forceinline__ void decode_nibbles(uint32_t w, uint32_t (&p)[4]) {
  const uint32_t lo_mask = 0x000F000Fu, hi_mask = 0x00F000F0u, magic = 0x64006400u;
  const __half2 k1032 = u32_as_h2(0x64086408u);   // 1032 = 1024 + 8
  const __half2 k1_16 = u32_as_h2(0x2C002C00u);   // 1/16
  const __half2 km72 = u32_as_h2(0xD480D480u);    // -72 = -(64 + 8)
  const uint32_t w8 = w >> 8;
  p[0] = h2_as_u32(__hsub2(u32_as_h2((w & lo_mask) | magic), k1032));
  p[1] = h2_as_u32(__hfma2(u32_as_h2((w & hi_mask) | magic), k1_16, km72));
  p[2] = h2_as_u32(__hsub2(u32_as_h2((w8 & lo_mask) | magic), k1032));
  p[3] = h2_as_u32(__hfma2(u32_as_h2((w8 & hi_mask) | magic), k1_16, km72));
}

// The nibbles u of a packed word as E4M3 codes, the code byte being the nibble
// itself: exponent field u >> 3 and mantissa u & 7 make u < 8 the subnormal
// u * 2^-9 and u >= 8 the normal (1 + (u & 7) / 8) * 2^-6 = u * 2^-9, so every
// code is worth exactly u * 2^-9.  lo holds the low nibbles of the four bytes
// (even reduction indices), hi the high ones (odd indices).
__device__ __forceinline__ void split_nibbles_e4m3(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = w & 0x0F0F0F0Fu;
  hi = (w >> 4) & 0x0F0F0F0Fu;
}

// 16-byte read-only load that stays where it is written (volatile asm is not
// moved across other volatile asm, such as later cp.async copies).
__device__ __forceinline__ uint4 ldg_v4_early(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }


}  // namespace qre
