// attn_common.cuh -- pieces shared by the attention kernels: parameters, the device error
// word, bounded barrier waits and the row-softmax helpers.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "ptx.cuh"
#include "rotary.cuh"
#include "tile_layout.cuh"

namespace neox {

// Error word (per device).  Bit 0: a bounded wait ran out; bit 1: a device-side input
// check failed; bit 2: a rotated query/key value did not fit its fp16 operand.  Bits
// 8..15: the site.
__device__ unsigned int g_device_error = 0;
constexpr unsigned int kErrTimeout = 1u;
constexpr unsigned int kErrBadInput = 2u;  // an input read on the device was out of range
constexpr unsigned int kErrRange = 4u;     // |rotated q or k| > 65504 where fp16 operands are used

// A wait that has not completed after this long is treated as a hang: the kernel records
// it, stops its own work and exits cleanly instead of blocking the GPU.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

struct AttnParams {
  const float2* cs;    // cos/sin table [>= S][r/2]
  uint16_t* out;       // bf16 [B, S, H, D]
  float* lse;          // fp32 [B, H, S]
  int B, S, H, r;      // r = rotary_dim
  int r16;             // r rounded up to a multiple of 16 (columns of lo products)
  int side_cols;       // r16 rounded up to a multiple of 32 (side tile width), 0 if r == 0
  float scale_log2;    // log2(e) / sqrt(D)
  int num_units;       // work units (persistent kernel)
  int nk, nv;          // K and V ring depths (1..4), set at launch from the shared-memory budget
  uint64_t wait_limit_ns;
};

__device__ __forceinline__ void record_error(unsigned int code, unsigned int site) {
  atomicOr(&g_device_error, code | (site << 8));
}

// Bounded wait on an mbarrier phase, slow path: polls until the phase completes, the CTA
// aborts, or the limit runs out (then the abort flag is raised and the error recorded).
// Kept out of line so the many wait sites do not each carry a copy.
__device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             uint64_t limit_ns, unsigned int site) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_test(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      record_error(kErrTimeout, site);
      return false;
    }
  }
}

// Returns false if the CTA is aborting or the limit ran out.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint64_t limit_ns,
                                           unsigned int site) {
  if (mbar_test(bar, parity)) return true;
  return wait_phase_slow(bar, parity, abort_flag, limit_ns, site);
}

// The same wait fully inline, for code running with a raised register count (setmaxnreg),
// where ptxas cannot place a call.
__device__ __forceinline__ bool wait_phase_inline(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  uint64_t limit_ns, unsigned int site) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_test(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      record_error(kErrTimeout, site);
      return false;
    }
  }
}

// The same bounded wait with the CTA's abort flag given as a 32-bit shared-memory address
// (fewer live registers than a generic pointer in the register-heavy roles).
__device__ __forceinline__ int flag_ld(uint32_t a) {
  int v;
  asm volatile("ld.volatile.shared.b32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void flag_st(uint32_t a, int v) {
  asm volatile("st.volatile.shared.b32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ bool wait_phase_s(uint32_t bar, uint32_t parity, uint32_t abort_addr, uint64_t limit_ns,
                                             unsigned int site) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_test(bar, parity)) return true;
    if (flag_ld(abort_addr)) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      flag_st(abort_addr, 1);
      record_error(kErrTimeout, site);
      return false;
    }
  }
}

// Drain wait used on the abort path: waits for an in-flight async operation to land,
// ignoring the abort flag, still bounded.
__device__ __forceinline__ void drain_phase(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) break;
  }
}

__device__ __forceinline__ float fmax3(float a, float b, float c) { return fmaxf(fmaxf(a, b), c); }

}  // namespace neox
