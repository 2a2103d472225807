// selftest.cuh -- exercise the failure path of the bounded waits on the GPU,
// and expose the expert epilogue's silu for accuracy tests.
//
// Every wait of the library's kernels on an mbarrier gives up after a time
// limit, sets the device error word (MOE_DEV_ERR_TIMEOUT, read and reset by
// moe_last_error) and lets the kernel return, so that a stuck pipeline ends
// with an error instead of hanging the GPU.  k_selftest_wait runs that path
// on purpose: one thread waits on an mbarrier that nothing arrives on, with
// a short limit.  No fault, no trap: the kernel returns normally and the
// context stays usable.
#pragma once

#include "experts_tc.cuh"

__global__ void __launch_bounds__(32) k_selftest_wait(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_barrier_init();
  // phase 0 of a fresh barrier with one expected arrival: it never completes
  bool done = mbar_try_wait(b, 0);
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; !done && it < (1u << 28); ++it) {
    done = mbar_try_wait(b, 0);
    if ((it & 63u) == 63u && global_timer_ns() - t0 > limit_ns) break;
  }
  if (!done) atomicOr(&g_moe_dev_error, MOE_DEV_ERR_TIMEOUT);
}

// The expert epilogue's silu, elementwise (moe_selftest_silu).
__global__ void __launch_bounds__(256) k_selftest_silu(const float* __restrict__ z,
                                                       float* __restrict__ out, int n) {
  const int i = blockIdx.x * 256 + threadIdx.x;
  if (i < n) out[i] = silu_fast(z[i]);
}
