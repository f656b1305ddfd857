// Pieces shared by the attention kernels and the host code of libfa.so:
// the device error word protocol, bounded mbarrier waits and the prefill
// tile plan.
#pragma once

#include <cstdint>

#include "sm103.cuh"

namespace fa {

// A bounded wait gives up after this long; no wait in these kernels is
// legitimately longer than a few microseconds.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

// Device error word: err[0] holds flags (bit 0 = a bounded wait ran out,
// bit 1 = a protocol check of an FA_DEBUG build failed), err[1] the site code
// of the first wait or check that failed.
constexpr unsigned int kErrTimeout = 1u;
constexpr unsigned int kErrCheck = 2u;

// Site codes (which wait ran out), reported by fa_check_device_error.
enum WaitSite : int {
  kSiteQFull = 1,
  kSiteKvFull = 2,
  kSiteKvEmpty = 3,
  kSiteSFull = 4,
  kSitePFull = 5,
  kSiteOFull = 6,
  kSiteDrain = 7,
  kSiteQEmpty = 8,
  kSiteOEmpty = 9,
  kSiteItemFull = 10,   // block-sparse forward: the next item index was published
  kSiteItemEmpty = 11,  // block-sparse forward: an item slot was read by every role
  kSiteCheckFwd = 20,  // FA_DEBUG: the forward's roles disagree (items, ring, phases)
  kSiteCheckBwd = 21,  // FA_DEBUG: the backward's roles completed different tile counts
  kSiteCheckGqa = 22,  // FA_DEBUG: the GQA decode's roles disagree on the tiles of a split
  kSiteSelftest = 100,
};

__device__ __forceinline__ void record_timeout(unsigned int* err, int site) {
  atomicOr(&err[0], kErrTimeout);
  atomicCAS(&err[1], 0u, static_cast<unsigned int>(site));
}

__device__ __forceinline__ void record_check(unsigned int* err, int site) {
  atomicOr(&err[0], kErrCheck);
  atomicCAS(&err[1], 0u, static_cast<unsigned int>(site));
}

// Wait for the phase of `bar` with the given parity to complete. Gives up and
// returns false when `timeout_ns` passes (recording the site and raising the
// CTA's abort flag) or when another thread of the CTA has raised the flag.
__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned int* err, int site, uint64_t timeout_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      if (abort_flag != nullptr) *abort_flag = 1;
      record_timeout(err, site);
      return false;
    }
  }
}

// bounded_wait for a barrier that also receives arrivals from the peer CTA of a
// pair: the wait acquires at cluster scope, so the peer's writes released by
// its arrival are visible afterwards.
__device__ __forceinline__ bool bounded_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                     unsigned int* err, int site,
                                                     uint64_t timeout_ns = kWaitTimeoutNs) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      if (abort_flag != nullptr) *abort_flag = 1;
      record_timeout(err, site);
      return false;
    }
  }
}

// Number of K/V tiles a Q tile starting at row `q_start` visits, with square
// tiles of `block` rows: all of them without a mask; under the causal mask
// only those not entirely above the diagonal, i.e. tiles 0 .. last_row/block
// (CMU 15-779 Lecture 5 notes §6.2, "skip whole blocks").
__host__ __device__ __forceinline__ int fwd_kv_tiles(int q_start, int N, int block, int causal) {
  if (q_start >= N) return 0;
  const int tiles = (N + block - 1) / block;
  if (!causal) return tiles;
  const int last_row = (q_start + block - 1 < N - 1) ? q_start + block - 1 : N - 1;
  return last_row / block + 1;
}

}  // namespace fa
