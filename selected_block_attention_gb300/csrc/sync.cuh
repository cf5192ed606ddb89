// Bounded synchronisation for the warp-specialised kernels.
//
// Every wait gives up after the launch's limit (Abort::limit; by default
// kWaitTimeoutCycles): it records where it gave up in the
// kernel's error word (first failure wins), raises the CTA's abort flag and returns
// false; every later wait of the CTA then returns false at once, so all roles unwind
// to the kernel's final barrier.  No role loop uses an unbounded hardware barrier
// (bar.sync): warpgroup-wide synchronisation goes through an mbarrier instead.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace sba {

struct DevError {
  unsigned flags;  // kDevErrTimeout | kDevErrInput
  unsigned where;  // first timeout: (kernel << 24) | (role << 16) | barrier id
  int item;        // work item being processed at the first timeout
};

struct Abort {
  volatile int* flag;
  DevError* err;
  unsigned kernel_id;
  long long limit;  // SM cycles a wait may take before the CTA gives up
};

// Below this limit (SM cycles) the probes never suspend the thread: a converged warp's
// try_wait sleeps until the phase completes (or a system-dependent time passes), so a
// short limit would otherwise never be looked at.
constexpr long long kShortWaitLimit = 1LL << 20;

// Bounded wait of one thread on an mbarrier phase.
__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, const Abort& ab,
                                             unsigned role, unsigned bar_id, int item) {
  const uint32_t a = ptx::smem_u32(bar);
  const bool short_limit = ab.limit < kShortWaitLimit;
  auto probe = [&]() {
    return short_limit ? ptx::mbar_test_wait(a, parity) : ptx::mbar_try_wait(a, parity);
  };
  if (probe()) return true;
  const long long t0 = clock64();
  while (true) {
    if (probe()) return true;
    if (*ab.flag) return false;
    if (clock64() - t0 > ab.limit) {
      atomicOr(&ab.err->flags, kDevErrTimeout);
      const unsigned code = (ab.kernel_id << 24) | (role << 16) | (bar_id & 0xFFFFu);
      if (atomicCAS(&ab.err->where, 0u, code) == 0u) ab.err->item = item;
      *ab.flag = 1;
      return false;
    }
  }
}

// Whole-warp wait: every lane waits, the result is made warp-uniform so the lanes
// keep one control flow even if the deadline falls between two lanes' checks.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const Abort& ab,
                                          unsigned role, unsigned bar_id, int item) {
  const bool ok = bounded_wait(bar, parity, ab, role, bar_id, item);
  return __all_sync(0xffffffffu, ok);
}

// Barrier over `nwarps` whole warps built on an mbarrier initialised with count
// nwarps: each warp arrives once (lane 0, after __syncwarp), then every thread waits
// for the phase.  `phase` is the caller's running count of uses (its parity is taken).
__device__ __forceinline__ bool warps_barrier(uint64_t* bar, uint32_t& phase, const Abort& ab,
                                             unsigned role, unsigned bar_id, int item) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(bar);
  const bool ok = warp_wait(bar, phase & 1u, ab, role, bar_id, item);
  phase ^= 1u;
  return ok;
}

// Bounded drain: wait for a phase without flagging anything (used at teardown for
// copies that were issued before an abort).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = ptx::smem_u32(bar);
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait(a, parity) && clock64() - t0 < kWaitTimeoutCycles) {
  }
}

}  // namespace sba
