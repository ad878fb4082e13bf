// decode_common.cuh -- device pieces shared by the single-CTA decode kernel and the
// two-CTA (cluster) decode kernel: launch parameters, bounded mbarrier waits, the
// softmax warps' named barrier, and small arithmetic helpers.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "mla_decode.h"
#include "plan_format.h"
#include "ptx.cuh"

namespace mla {

constexpr long long kWaitBudget = 2000000000LL;  // cycles (~1 s) before a wait gives up
constexpr long long kWaitBudgetTest = 4000000LL; // ~2 ms: the budget of a call that tests the timeout path

struct Params {
  const PlanUnit* units;   // the plan's unit table (one record per CTA, or per CTA pair)
  const __nv_bfloat16* q;  // the e4m3 path converts its Q tile from global memory
  int q_rows;              // rows of q (sum q_lens * H)
  const int32_t* page_table;
  int pt_stride, num_pages, H;
  const int32_t* seq_lens;
  const int32_t* q_lens;
  float score_scale_log2;  // sm_scale * kv_scale * log2(e)
  float out_scale;         // kv_scale (1 for a bf16 cache)
  __nv_bfloat16* out;
  float* lse;
  __nv_bfloat16* part_o;  // split partials of O (bf16, each normalised by its split's l)
  float* part_lse;
  int32_t* status;
  long long wait_budget;  // cycles a bounded wait may take (kWaitBudget; kWaitBudgetTest in a timeout test)
  int skip_copy;          // page of the first unit whose copy is never issued (timeout test), or -1
};

__device__ __forceinline__ void report(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

// Warp-uniform bounded wait. The whole warp polls together and goes on once every lane has
// seen the phase complete (each lane's own test acquires it; with kCluster at cluster
// scope), so the warp never diverges while it waits: a lane-0 spin loop with the other
// lanes parked at a shuffle cost every role ~10 % of its pace (1M q=8 bf16 392.7 -> 349.2
// us, q=1 38.9 -> 35.8 us when changed).
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, const Params& p) {
  auto poll = [&]() { return kCluster ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity); };
  if (__all_sync(0xffffffffu, poll())) return true;
  const long long t0 = clock64();
  while (true) {
    if (__all_sync(0xffffffffu, poll())) return true;
    if (__shfl_sync(0xffffffffu, *abort, 0)) return false;
    if (__shfl_sync(0xffffffffu, clock64() - t0 > p.wait_budget ? 1 : 0, 0)) {
      if ((threadIdx.x & 31) == 0) {
        *abort = 1;
        report(p.status, MLA_DEVICE_WAIT_TIMEOUT);
      }
      return false;
    }
  }
}

// Barriers among the softmax warps only (named barrier 1). Every softmax warp reaches
// every one of them the same number of times, whatever happens to the unit: decisions
// that end the loop are taken from a barrier's OR-reduction, so all warps take them
// together.
constexpr int kSoftmaxWarps = 8;  // two per TMEM lane quadrant, each owning half of the columns
constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr uint32_t kSoftmaxBar = 1;
__device__ __forceinline__ void softmax_sync() { ptx::bar_sync(kSoftmaxBar, kSoftmaxThreads); }
__device__ __forceinline__ bool softmax_any(bool pred) { return ptx::bar_red_or(kSoftmaxBar, kSoftmaxThreads, pred); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Waits (bounded) until the tcgen05 operations this lane issued have completed.
__device__ __forceinline__ void drain_mmas(uint64_t* done, long long budget) {
  ptx::mma_commit(done);
  long long t0c = clock64();
  while (!ptx::mbar_try_wait(done, 0) && clock64() - t0c < budget) {
  }
}

}  // namespace mla
