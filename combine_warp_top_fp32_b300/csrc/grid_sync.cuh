// grid_sync.cuh — the one device-wide wait of the fused dispatch kernel, and
// the bounded waits on its bulk copies.
//
// The fused kernel is launched cooperatively (every CTA resident at once), so
// a grid barrier cannot wait on a CTA that has not started. Every wait is
// still bounded: after `limit` polls the waiting thread gives up and the
// caller records kStatusTimeout, which ep_get_error reports as
// EP_ERR_TIMEOUT (the NCCL EP article, §4.2–4.3: report a failed wait as an
// error instead of hanging).
#pragma once

#include "ep_device.cuh"

namespace ep {

// Barrier words in the workspace: arrivals of the current round and the
// round number. The last CTA to arrive zeroes the arrivals and then advances
// the round; the others wait for the round to change. Arrivals are back at 0
// after every completed barrier, so a workspace zeroed once serves every call.
struct GridBarrier {
  unsigned* count;
  unsigned* round;
};

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void red_add_release_gpu(unsigned* p, unsigned v) {
  asm volatile("red.add.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// All threads of the CTA call it. Returns true once every one of `expected`
// CTAs has arrived (their writes before the barrier are then visible to every
// thread of this CTA), false if thread 0 gave up after `limit` polls. The
// CTA's writes reach thread 0 through the CTA barrier; thread 0's arrival is
// a release and its wait an acquire at GPU scope. The last CTA to arrive
// also stores `reset_value` to `*reset` (when given) before it lets the others
// go, so a counter used after the barrier starts from a known value.
// *round_after (when given) receives the round the barrier completes: the
// same in every CTA, and different in consecutive uses of the words.
__device__ __forceinline__ bool grid_barrier(GridBarrier bar, unsigned expected, long long limit,
                                             unsigned* reset = nullptr, unsigned reset_value = 0u,
                                             unsigned* round_after = nullptr) {
  __shared__ int passed_s;
  __shared__ unsigned round_s;
  __syncthreads();
  if (threadIdx.x == 0) {
    int passed = 1;
    const unsigned r = ld_acquire_gpu(bar.round);
    round_s = r + 1u;
    const unsigned prev = atom_add_acq_rel_gpu(bar.count, 1u);
    if (prev == expected - 1) {
      *reinterpret_cast<volatile unsigned*>(bar.count) = 0u;
      if (reset) *reinterpret_cast<volatile unsigned*>(reset) = reset_value;
      red_add_release_gpu(bar.round, 1u);
    } else {
      long long polls = 0;
      while (ld_acquire_gpu(bar.round) == r) {
        if (++polls > limit) {
          passed = 0;
          break;
        }
        __nanosleep(16);
      }
    }
    passed_s = passed;
  }
  __syncthreads();
  if (round_after) *round_after = round_s;
  return passed_s != 0;
}

// The arrival half of a split grid barrier, by one thread after a CTA
// barrier (so the CTA's writes before it are ordered before the arrival): the
// last of `expected` CTAs to arrive zeroes the arrivals and advances the round.
// The wait half is a bounded poll until the round differs from the one seen at
// the barrier before (every CTA knows it).
__device__ __forceinline__ void grid_arrive(GridBarrier bar, unsigned expected) {
  const unsigned prev = atom_add_acq_rel_gpu(bar.count, 1u);
  if (prev == expected - 1) {
    *reinterpret_cast<volatile unsigned*>(bar.count) = 0u;
    red_add_release_gpu(bar.round, 1u);
  }
}

// ---- mbarrier + 1-D bulk copy (global -> this CTA's shared memory) ----------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned arrivals) {
  asm volatile("mbarrier.init.shared.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(arrivals) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Copies `bytes` (a multiple of 16; both addresses 16-byte aligned) from
// global memory into shared memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Waits for phase `parity` of `bar` to complete; false after `limit` polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, long long limit) {
  for (long long polls = 0; polls <= limit; ++polls) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

}  // namespace ep
