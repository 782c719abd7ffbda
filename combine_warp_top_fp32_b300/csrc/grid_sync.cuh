// grid_sync.cuh — the device-wide waits of the fused dispatch kernel, and
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

// Barrier words in the workspace: an arrival count and a round number
// (count_barrier / split_arrive below). Both are back at their resting state
// after every completed launch, so a workspace zeroed once serves every call.
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

// The single launch's two grid-wide waits on one arrival count. The first
// completes when the count reaches `expected` (every CTA arrived once): no
// CTA resets anything, so the waiters see completion one L2 round trip after
// the last arrival. The second (split_arrive, below) counts on to
// 2 * expected; its last arrival zeroes the count and `reset` (the scatter's
// token counter) and advances the round, which the second wait polls. The
// words are back at zero after every launch. All threads of the CTA call
// count_barrier; it returns false if thread 0 gave up after `limit` polls.
// *round_out (thread 0's read, shared with the CTA) is the round while the
// second wait is incomplete.
__device__ __forceinline__ bool count_barrier(GridBarrier bar, unsigned expected, long long limit,
                                              unsigned* round_out) {
  __shared__ int passed_s;
  __shared__ unsigned round_s;
  __syncthreads();
  if (threadIdx.x == 0) {
    int passed = 1;
    const unsigned prev = atom_add_acq_rel_gpu(bar.count, 1u);
    round_s = ld_acquire_gpu(bar.round);  // unchanged until the second wait completes
    if (prev + 1u < expected) {
      long long polls = 0;
      while (ld_acquire_gpu(bar.count) < expected) {
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
  *round_out = round_s;
  return passed_s != 0;
}

// The second wait's arrival (one thread, after a CTA barrier): the last of
// 2 * expected arrivals zeroes the count and *reset, then advances the round.
__device__ __forceinline__ void split_arrive(GridBarrier bar, unsigned expected, unsigned* reset) {
  const unsigned prev = atom_add_acq_rel_gpu(bar.count, 1u);
  if (prev == 2u * expected - 1u) {
    *reinterpret_cast<volatile unsigned*>(bar.count) = 0u;
    *reinterpret_cast<volatile unsigned*>(reset) = 0u;
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
