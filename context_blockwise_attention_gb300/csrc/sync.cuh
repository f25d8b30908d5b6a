// Bounded waits and the abort protocol of the warp-specialised tensor-core kernels.
//
// Every mbarrier wait gives up after a time limit (%globaltimer): it then records
// CP_ERR_TIMEOUT | (site << 8) in the caller's status word, raises a CTA-wide abort flag in shared
// memory, and every role leaves its loops; copies and MMAs already issued are waited for (again
// with a limit) before the CTA frees its tensor memory and exits.
#pragma once

#include "cpattn.h"
#include "ptx.cuh"

namespace cpattn {
namespace sync {

struct Ctl {
  volatile int* abort;
  int32_t* status;
  int64_t timeout_ns;
};

__device__ __forceinline__ void raise_abort(const Ctl& c, int site) {
  *c.abort = 1;
  if (c.status != nullptr) atomicCAS(c.status, 0, CP_ERR_TIMEOUT | (site << 8));
}

// Waits for phase `parity` of `bar`; false when the kernel is aborting or the limit expired (in
// which case this wait starts the abort).  kProbe: test the phase once with the non-suspending
// test_wait before the try_wait loop.  Without the probe the attention forward is 1.5-6.5 %
// faster (same-box A/B); the D = 64 backward is 1.2 % faster with it.
template <bool kProbe = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const Ctl& c, int site) {
  if (kProbe && ptx::mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*c.abort) return false;
      if (static_cast<int64_t>(ptx::globaltimer() - t0) > c.timeout_ns) {
        raise_abort(c, site);
        return false;
      }
    }
  }
}

// Every lane of the warp waits; the outcome is the same for the whole warp.
template <bool kProbe = false>
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const Ctl& c, int site) {
  const bool ok = wait_bounded<kProbe>(bar, parity, c, site);
  return __all_sync(0xffffffffu, ok);
}

// Teardown wait: ignores the abort flag (the copy or MMA must really finish) but stays bounded.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, int64_t timeout_ns) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (static_cast<int64_t>(ptx::globaltimer() - t0) > timeout_ns) return;
  }
}

// The k-th unit of CTA b of a persistent grid: rounds of `grid` units, forward on even rounds,
// backward on odd ones (longest-first unit numbering then balances the rounds).
__device__ __forceinline__ int64_t unit_of(int64_t k, int64_t b, int64_t grid) {
  return k * grid + ((k & 1) ? (grid - 1 - b) : b);
}

}  // namespace sync
}  // namespace cpattn
