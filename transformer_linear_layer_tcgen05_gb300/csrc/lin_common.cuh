// lin_common.cuh -- device helpers shared by the GEMM kernels: bounded
// mbarrier waits, the stable silu of the SwiGLU forms, binary16 packing and
// the 128-byte swizzle address function.
#pragma once

#include <cuda_fp16.h>

#include "lin_internal.h"
#include "lin_ptx.cuh"

#ifndef LIN_DEVICE_CHECKS
#define LIN_DEVICE_CHECKS 0
#endif

namespace lin {

// ---------------------------------------------------------------- checks

// Record a failed check in the status record [status, site, value]: the
// first failure of any kind keeps the record.
__device__ __forceinline__ void report_check(int* status, int site, long long value) {
  if (status && atomicCAS(status, KSTATUS_OK, KSTATUS_CHECK) == KSTATUS_OK) {
    status[1] = site;
    *reinterpret_cast<long long*>(status + 2) = value;
  }
}

// Checked build (LIN_DEVICE_CHECKS=1): true when the access guarded by `ok`
// may go ahead; otherwise the failure is recorded and the caller skips the
// access. In the default build it is true and compiles away.
__device__ __forceinline__ bool dcheck(bool ok, int* status, int site, long long value) {
#if LIN_DEVICE_CHECKS
  if (!ok) report_check(status, site, value);
  return ok;
#else
  (void)ok;
  (void)status;
  (void)site;
  (void)value;
  return true;
#endif
}

// ---------------------------------------------------------------- waiting

struct WaitCtl {
  uint64_t timeout_ns;
  volatile int* abort;  // shared-memory flag: some role gave up
  int* status;          // device status word
};

// Wait for completion of the barrier phase with parity `parity`. Returns
// false if the wait ran out (and records the timeout) or, when
// `honor_abort`, if another role already gave up.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                           bool honor_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
#pragma unroll 1
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (honor_abort && *c.abort) return false;
    if (global_timer_ns() - t0 > c.timeout_ns) {
      *c.abort = 1;
      atomicCAS(c.status, KSTATUS_OK, KSTATUS_TIMEOUT);
      return false;
    }
  }
}

// Same with cluster-scope acquire: for barriers that peers of the cluster
// arrive on (remote arrives, multicast commits).
__device__ __forceinline__ bool wait_phase_cluster(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                                   bool honor_abort = true) {
  if (mbar_try_wait_acq_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
#pragma unroll 1
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait_acq_cluster(bar, parity)) return true;
    if (honor_abort && *c.abort) return false;
    if (global_timer_ns() - t0 > c.timeout_ns) {
      *c.abort = 1;
      atomicCAS(c.status, KSTATUS_OK, KSTATUS_TIMEOUT);
      return false;
    }
  }
}

// Warp-uniform wait: every lane waits (each needs the acquire), and the warp
// proceeds only if all lanes succeeded.
__device__ __forceinline__ bool warp_wait_phase(uint32_t bar, uint32_t parity, const WaitCtl& c) {
  const bool ok = wait_phase(bar, parity, c);
  return __all_sync(0xffffffffu, ok);
}

// The same with cluster-scope acquire (a barrier that a peer's commit completes).
__device__ __forceinline__ bool warp_wait_phase_cluster(uint32_t bar, uint32_t parity,
                                                        const WaitCtl& c) {
  const bool ok = wait_phase_cluster(bar, parity, c);
  return __all_sync(0xffffffffu, ok);
}

// Lane 0 waits (it is the lane that issues the copies or UMMAs that follow);
// the result is broadcast so the warp stays converged.
__device__ __forceinline__ bool lane0_wait_phase(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                                 int lane) {
  bool ok = true;
  if (lane == 0) ok = wait_phase(bar, parity, c);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// ---------------------------------------------------------------- activation

// silu(x) = x * sigma(x) with the stable, sign-branched sigmoid of page
// 09_backward_ffn ("SiLU'"; note 2 of "WGSL-Spesifik Notlar"):
//   x >= 0: 1 / (1 + exp(-x))      x < 0: exp(x) / (1 + exp(x)).
// Both branches evaluate exp at -|x| <= 0, so it cannot overflow; the branch
// is a select on the numerator. Very negative x underflows to 0.
__device__ __forceinline__ float silu_stable(float x) {
  const float e = __expf(-fabsf(x));
  const float num = x >= 0.0f ? 1.0f : e;
  return x * __fdividef(num, 1.0f + e);
}

// nan_guard of the pages' shared preamble: x if it is finite (x == x and
// |x| < FLT_MAX, the pages' is_finite), else 0.
__device__ __forceinline__ float nan_guard(float x) {
  return (x == x && fabsf(x) < 3.40282347e+38f) ? x : 0.0f;
}

// The SwiGLU backward of page 09_backward_ffn ("SwiGLU backward" and
// "ffn_swiglu_backward"): with s = sigma(gate) (the stable sigmoid above),
// dgate = g * u * silu'(gate), silu'(x) = s * (1 + x * (1 - s)), and
// dup = g * silu(gate), each through nan_guard.
__device__ __forceinline__ void swiglu_backward(float g, float gate, float u, float& dgate,
                                                float& dup) {
  const float e = __expf(-fabsf(gate));
  const float s = __fdividef(gate >= 0.0f ? 1.0f : e, 1.0f + e);
  dgate = nan_guard(g * u * (s * (1.0f + gate * (1.0f - s))));
  dup = nan_guard(g * (gate * s));
}

// Same function in six instructions: exp(-|x|) by the hardware ex2, and the
// reciprocal of d = 1 + exp(-|x|), which lies in [1, 2], by the hardware
// reciprocal approximation (about 1 ulp there). Measured faster than a
// Newton-Raphson reciprocal on the FMA pipe, which needs five instructions
// more per element.
__device__ __forceinline__ float silu_stable_fast(float x) {
  const float e = ex2_approx(fabsf(x) * -1.4426950408889634f);   // exp(-|x|)
  const float r = rcp_approx(1.0f + e);
  const float num = x >= 0.0f ? 1.0f : e;
  return x * (num * r);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);   // round-to-nearest-even
  return *reinterpret_cast<const uint32_t*>(&h);
}

// ---------------------------------------------------------------- transform

// Swizzled byte offset of 16-byte chunk `c` of row `r` in a [rows][128 B]
// tile with the 128-byte swizzle (chunk index XOR row mod 8), the layout both
// TMA (SWIZZLE_128B) and the UMMA K-major descriptor use.
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t c) {
  return r * 128u + ((c ^ (r & 7u)) << 4);
}

// The same for a [rows][64 B] tile with the 64-byte swizzle (TMA
// SWIZZLE_64B: 16-byte chunk index XOR address bits 7-8, i.e. (r / 2) mod 4).
// A warp reading chunk c of 32 consecutive rows touches every bank once per
// eight rows.
__device__ __forceinline__ uint32_t sw64(uint32_t r, uint32_t c) {
  return r * 64u + ((c ^ ((r >> 1) & 3u)) << 4);
}

}  // namespace lin
