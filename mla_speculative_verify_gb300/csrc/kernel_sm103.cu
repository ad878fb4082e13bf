// kernel_sm103.cu -- fused MLA speculative-verify decode for GB300 (sm_103a).
//
// One CTA processes one plan unit: a tile of at most kRowsCap packed query rows
// (row = token * H + head; the q verify tokens of a fold group are folded into the
// rows, sglang PR #33650 "Why" paragraph) against one page-aligned key range of
// one request. The cache streams through shared memory once per unit, one 64-key
// page per pipeline stage (one 3-D TMA box per page), and both products run on the
// tcgen05 tensor cores with the accumulators in tensor memory, in the transposed
// orientation:
//
//   S^T[key, row]  = K[key, 0:576] . Q[row, 0:576]^T    (M = 64 keys, N = rows, K = 576)
//   O^T[dv, row]  += V^T[dv, key] . P^T[key, row]        (M = 128 dv x 4 blocks, N = rows, K = 64 keys)
//
// so the MMA N dimension is the packed-row count rounded up to 16 and no MMA work is
// spent on padding rows to 64 or 128. V^T is the same shared-memory page as K, read
// MN-major (the latent cache rows hold V in columns 0..511; flashinfer PR #5602 "What
// r52 changes": the latent K stages are held until PV).
//
// One thread issues a tcgen05.mma only every ~60 cycles, while an N = 16..48 MMA
// needs 20..45 cycles of tensor time, so four warps issue in parallel: warp 1+p owns
// K-chunks of the S^T product (into its own partial accumulator S_p, summed by the
// softmax) and dv block p of the O^T product.
//
// Warp roles (one CTA per SM, one page in flight while the other is consumed):
//   warp 0     TMA producer: the Q tile once, then one page per stage
//   warps 1-4  MMA issue (one elected lane each); for an fp8 cache they first expand
//              their own chunks of the e4m3 page to bf16 in place (exact; kv_scale is
//              folded into the score and output scales)
//   warps 5-8  softmax: each thread owns one key of the S^T tile (a TMEM lane); online
//              softmax with a lazy per-row reference: the reference moves, and O^T is
//              rescaled in TMEM, only when a score exceeds it by kRefSlack octaves (the
//              conditional rescale of flashinfer PR #5602); then the epilogue: O / l to
//              bf16 out and LSE, or fp32 partials for the merge kernel
//
// Every mbarrier wait is bounded; on expiry the kernel ORs MLA_DEVICE_WAIT_TIMEOUT into
// the status word, stops the unit, drains its in-flight copies and frees its TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "mla_decode.h"
#include "plan_format.h"
#include "ptx.cuh"
#include "status.h"

namespace mla {

// ------------------------------------------------------------------ tile geometry
constexpr int kRowsCap = 48;                       // packed rows per CTA (shared-memory bound)
constexpr int kTileKeys = 64;                      // keys per stage = one page
constexpr int kChunks = 9;                         // 576 = 9 x 64 columns (128-byte swizzle rows)
constexpr int kQChunkBytes = kRowsCap * 128;       // 6144
constexpr int kQBytes = kChunks * kQChunkBytes;    // 55296
constexpr int kKvChunkBytes = kTileKeys * 128;     // 8192
constexpr int kSlotBytes = kChunks * kKvChunkBytes;  // 73728 (bf16 page)
constexpr int kFp8StageOff = kSlotBytes / 2;       // an e4m3 page lands in the upper half of its slot
constexpr int kFp8ChunkBytes = kTileKeys * 64;     // 4096
constexpr int kPtBytes = kTileKeys * 128;          // P^T tile: 64 keys x (<= 64 rows) bf16
constexpr int kOffQ = 0;
constexpr int kOffKv = kOffQ + kQBytes;
constexpr int kOffPt = kOffKv + 2 * kSlotBytes;
constexpr int kOffMisc = kOffPt + 2 * kPtBytes;
constexpr int kMiscBytes = 4096;
constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-CTA shared memory");
static_assert(kOffKv % 1024 == 0 && kOffPt % 1024 == 0 && kOffMisc % 1024 == 0, "1024-byte swizzle atoms");

constexpr int kMmaWarps = 4;
constexpr int kThreads = 32 * (1 + kMmaWarps + 4);  // producer, MMA warps, softmax warps
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;       // O^T block b at columns 64 b (N <= 64)
constexpr uint32_t kTmemS = 256;     // partial S^T p at columns 256 + 64 p
constexpr float kRefSlack = 8.0f;    // octaves a score may exceed the row reference before it moves
constexpr long long kWaitBudget = 2000000000LL;  // cycles (~1 s) before a wait gives up

// K-steps (16 columns each) of the S^T product owned by MMA warp p: [9 p, 9 p + 9) of
// the 36; the e4m3 expansion of a page is split by 64-column chunks instead
// ([chunk_lo(p), chunk_lo(p + 1)) = 3, 2, 2, 2 of the 9 chunks).
constexpr int kKSteps = kChunks * 4;
constexpr int kKStepsPerWarp = kKSteps / 4;
__host__ __device__ __forceinline__ int chunk_lo(int p) { return p == 0 ? 0 : 1 + 2 * p; }

// Rows of an M = 64 accumulator occupy 16 TMEM lanes per 32-lane quadrant:
// row r -> lane 32 * (r / 16) + r % 16.
__device__ __forceinline__ int m64_row_of_lane(int quadrant, int lane) { return lane < 16 ? quadrant * 16 + lane : -1; }

struct Params {
  const uint8_t* plan;
  const int32_t* page_table;
  int pt_stride, num_pages, H;
  const int32_t* seq_lens;
  const int32_t* q_lens;
  float score_scale_log2;  // sm_scale * kv_scale * log2(e)
  float out_scale;         // kv_scale (1 for a bf16 cache)
  __nv_bfloat16* out;
  float* lse;
  float* part_o;
  float* part_lse;
  int32_t* status;
};

struct Misc {
  uint64_t bar_q;
  uint64_t kv_full[2], kv_empty[2];
  uint64_t s_full, s_empty;
  uint64_t p_full[2], pt_empty[2];
  uint64_t mma_done;
  uint64_t grp_softmax, grp_mma;  // bounded barriers among the 4 warps of a group
  uint32_t tmem_base;
  int abort;
  int unit[8];
  int req[4];
  int flags[2][4];
  alignas(16) float ref[64];  // read as float4
  alignas(16) float alpha[64];
  alignas(16) int lim[64];
  alignas(16) float colred[4][64];
  alignas(16) float lsum[64];
};
static_assert(offsetof(Misc, ref) % 16 == 0, "float4 reads of ref need 16-byte alignment");
static_assert(sizeof(Misc) <= kMiscBytes, "misc block too small");

__device__ __forceinline__ void report(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

// Bounded wait: false when the budget ran out or another warp aborted the unit.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort, int32_t* status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > kWaitBudget) {
      *abort = 1;
      report(status, MLA_DEVICE_WAIT_TIMEOUT);
      return false;
    }
  }
}

// Warp-uniform bounded wait: lane 0 polls, the result is broadcast to the warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int32_t* status) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = wait_bar(bar, parity, abort, status) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Barrier among the four warps of a group, built on an mbarrier (count 4) so that it
// is bounded like every other wait: a warp that gave up never leaves the others stuck.
__device__ __forceinline__ bool group_sync(uint64_t* bar, uint32_t& phase, volatile int* abort, int32_t* status) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(bar);
  const bool ok = warp_wait(bar, phase & 1, abort, status);
  ++phase;
  return ok;
}

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

// e4m3 x4 (one 32-bit word) -> bf16 x4 (two 32-bit words), exact, through the
// hardware conversions (for pages that hold a zero, subnormal or NaN code).
__device__ __forceinline__ void e4m3x4_to_bf16x4_cvt(uint32_t w, uint32_t& lo, uint32_t& hi) {
  __half2_raw h0 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFFu), __NV_E4M3);
  __half2_raw h1 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
  float2 f0 = __half22float2(*reinterpret_cast<__half2*>(&h0));
  float2 f1 = __half22float2(*reinterpret_cast<__half2*>(&h1));
  lo = pack_bf16(f0.x, f0.y);
  hi = pack_bf16(f1.x, f1.y);
}

// e4m3 x4 -> bf16 x4 with integer operations, exact for normal codes. A normal e4m3
// code s.eeee.mmm equals (-1)^s 2^(e-7) (1 + m/8); the bf16 with exponent field e + 120
// and mantissa m << 4 holds the same value, so each 16-bit half is
// ((c & 0x7F) << 4) + (120 << 7) with the sign moved to bit 15.
__device__ __forceinline__ void e4m3x4_to_bf16x4_normal(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t a = __byte_perm(w, 0u, 0x4140);  // codes 0, 1 in the low bytes of the halves
  const uint32_t b = __byte_perm(w, 0u, 0x4342);  // codes 2, 3
  lo = (((a & 0x007F007Fu) << 4) + 0x3C003C00u) | ((a & 0x00800080u) << 8);
  hi = (((b & 0x007F007Fu) << 4) + 0x3C003C00u) | ((b & 0x00800080u) << 8);
}

// Nonzero when one of the four codes is zero/subnormal (exponent 0) or NaN (S.1111.111):
// those need the exact conversion.
__device__ __forceinline__ uint32_t e4m3x4_special(uint32_t w) {
  const uint32_t ex = w & 0x78787878u;                  // zero byte <=> zero exponent
  const uint32_t nn = (w & 0x7F7F7F7Fu) ^ 0x7F7F7F7Fu;  // zero byte <=> NaN code
  return (((ex - 0x01010101u) & ~ex) | ((nn - 0x01010101u) & ~nn)) & 0x80808080u;
}

struct SoftmaxArgs {
  Misc* ms;
  uint8_t* sKv;
  uint8_t* sPt;
  uint32_t tmem;
  int qd, lane, sidx, nrows, qrow0, kv_begin, kv_end, ntiles, part_row0, ctx, qlen, tok0;
  volatile int* abort;
};

// Softmax warps for a tile of 16 NCH packed rows. Lanes 0..15 of a warp read their key's
// S^T row from TMEM (the M = 64 accumulator uses 16 lanes per quadrant) and hand the
// upper 8 of every 16 columns to lanes 16..31, so each thread works on 8 NCH columns of
// one key: columns 16 c + 8 half + j, c < NCH, j < 8.
template <int NCH>
__device__ __forceinline__ void softmax_role(const SoftmaxArgs& a, const Params& p) {
  constexpr int NC = 8 * NCH;
  Misc* ms = a.ms;
  const int lane = a.lane, qd = a.qd, sidx = a.sidx;
  const int half = lane >> 4;
  const int krow = qd * 16 + (lane & 15);  // key row of this thread in the 64-key tile
  const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
  volatile int* abort = a.abort;
  uint32_t gphase = 0;
  if (sidx < 64) {
    int lim = 0;
    if (sidx < a.nrows) {
      const int i = (a.qrow0 + sidx) / p.H - a.tok0;  // verify token of this packed row
      lim = a.ctx - a.qlen + i + 1;
    }
    ms->lim[sidx] = lim;
    ms->ref[sidx] = -INFINITY;
  }
  bool ok = group_sync(&ms->grp_softmax, gphase, abort, p.status) && !*abort;
  int lim_min = a.kv_end;
  for (int n = 0; n < a.nrows; ++n) lim_min = min(lim_min, ms->lim[n]);
  float l_acc[NC];
#pragma unroll
  for (int i = 0; i < NC; ++i) l_acc[i] = 0.f;
  const float scale = p.score_scale_log2;
  for (int t = 0; ok && t < a.ntiles; ++t) {
    const int sb = t & 1;
    ok = warp_wait(&ms->s_full, t & 1, abort, p.status);
    if (!ok) break;
    ptx::tc_fence_after();
    // S^T = sum of the four partial accumulators, then split the columns over the halves
    float x[NC];
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      float s0[16], s1[16], s2[16];
      ptx::tmem_ld16(a.tmem + kTmemS + lane_off + 16 * c, s0);
      ptx::tmem_ld16(a.tmem + kTmemS + 64 + lane_off + 16 * c, s1);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) s0[j] += s1[j];
      ptx::tmem_ld16(a.tmem + kTmemS + 128 + lane_off + 16 * c, s1);
      ptx::tmem_ld16(a.tmem + kTmemS + 192 + lane_off + 16 * c, s2);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) s0[j] += s1[j] + s2[j];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float hi = __shfl_sync(0xffffffffu, s0[8 + j], lane & 15);
        x[8 * c + j] = half ? hi : s0[j];
      }
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&ms->s_empty);
    const int key = a.kv_begin + t * kTileKeys + krow;
    const int tile_last = a.kv_begin + t * kTileKeys + kTileKeys - 1;
    const bool unmasked = tile_last < a.kv_end && tile_last < lim_min;  // tile-uniform fast path
    bool need = false;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const int n0 = 16 * c + 8 * half;
      const float4 r0 = *reinterpret_cast<const float4*>(&ms->ref[n0]);
      const float4 r1 = *reinterpret_cast<const float4*>(&ms->ref[n0 + 4]);
      const float rr[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float v = x[8 * c + j] * scale;
        if (!unmasked) v = (key < a.kv_end && key < ms->lim[n0 + j]) ? v : -INFINITY;
        x[8 * c + j] = v;
        need |= v > rr[j] + kRefSlack;
      }
    }
    const unsigned vote = __any_sync(0xffffffffu, need);
    if (lane == 0) ms->flags[sb][qd] = vote ? 1 : 0;
    ok = group_sync(&ms->grp_softmax, gphase, abort, p.status);
    if (!ok) break;
    const bool moved = ms->flags[sb][0] | ms->flags[sb][1] | ms->flags[sb][2] | ms->flags[sb][3];
    if (moved) {
      // column maxima over this tile's keys (16 keys per half-warp), then move each
      // row's reference up to its maximum
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        float m = x[i];
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((lane & 15) == 0) ms->colred[qd][16 * (i / 8) + 8 * half + (i % 8)] = m;
      }
      ok = group_sync(&ms->grp_softmax, gphase, abort, p.status);
      if (!ok) break;
      if (sidx < 16 * NCH) {
        const float cm = fmaxf(fmaxf(ms->colred[0][sidx], ms->colred[1][sidx]), fmaxf(ms->colred[2][sidx], ms->colred[3][sidx]));
        const float old = ms->ref[sidx];
        const float nw = fmaxf(old, cm);
        ms->alpha[sidx] = (nw == old) ? 1.f : ex2(old - nw);
        ms->ref[sidx] = nw;
      }
      ok = group_sync(&ms->grp_softmax, gphase, abort, p.status);
      if (!ok) break;
#pragma unroll
      for (int i = 0; i < NC; ++i) l_acc[i] *= ms->alpha[16 * (i / 8) + 8 * half + (i % 8)];
      if (t >= 1) {
        // O^T holds tiles < t: wait for PV(t-1), then scale each row's column by alpha
        ok = warp_wait(&ms->pt_empty[(t - 1) & 1], ((t - 1) >> 1) & 1, abort, p.status);
        if (!ok) break;
        ptx::tc_fence_after();
#pragma unroll 1
        for (int blk = 0; blk < 4; ++blk) {
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            float o[16];
            const uint32_t ta = a.tmem + kTmemO + 64 * blk + lane_off + 16 * c;
            ptx::tmem_ld16(ta, o);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] *= ms->alpha[16 * c + j];
            ptx::tmem_st16(ta, o);
          }
        }
        ptx::tmem_st_wait();
      }
    }
    // probabilities relative to the (possibly moved) reference, packed to bf16
    uint32_t pk[NC / 2];
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const int n0 = 16 * c + 8 * half;
      const float4 r0 = *reinterpret_cast<const float4*>(&ms->ref[n0]);
      const float4 r1 = *reinterpret_cast<const float4*>(&ms->ref[n0 + 4]);
      const float rr[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        const float v0 = x[8 * c + j], v1 = x[8 * c + j + 1];
        const float p0 = v0 == -INFINITY ? 0.f : ex2(v0 - rr[j]);
        const float p1 = v1 == -INFINITY ? 0.f : ex2(v1 - rr[j + 1]);
        l_acc[8 * c + j] += p0;
        l_acc[8 * c + j + 1] += p1;
        pk[(8 * c + j) / 2] = pack_bf16(p0, p1);
      }
    }
    if (t >= 2) {
      ok = warp_wait(&ms->pt_empty[sb], ((t - 2) >> 1) & 1, abort, p.status);
      if (!ok) break;
    }
    uint8_t* line = a.sPt + sb * kPtBytes + krow * 128;
#pragma unroll
    for (int c = 0; c < NCH; ++c)
      *reinterpret_cast<uint4*>(line + ((((2 * c + half) ^ (krow & 7)) & 7) << 4)) =
          make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
    if (key >= a.kv_end) {
      // a cache slot past the key range: zero its value columns so P = 0 meets V = 0
      uint8_t* row = a.sKv + sb * kSlotBytes + krow * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(row + (4 * half + c) * kKvChunkBytes + 16 * j) = make_uint4(0, 0, 0, 0);
    }
    ptx::fence_async_smem();
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&ms->p_full[sb]);
  }
  // ------------------------------------------------------------ epilogue
  if (ok) ok = warp_wait(&ms->pt_empty[(a.ntiles - 1) & 1], ((a.ntiles - 1) >> 1) & 1, abort, p.status);
  if (ok) {
    ptx::tc_fence_after();
#pragma unroll
    for (int i = 0; i < NC; ++i) {
      float s = l_acc[i];
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if ((lane & 15) == 0) ms->colred[qd][16 * (i / 8) + 8 * half + (i % 8)] = s;
    }
    ok = group_sync(&ms->grp_softmax, gphase, abort, p.status);
  }
  if (ok) {
    if (sidx < a.nrows) {
      const float L = ms->colred[0][sidx] + ms->colred[1][sidx] + ms->colred[2][sidx] + ms->colred[3][sidx];
      ms->lsum[sidx] = L;
      const float lse_v = L > 0.f ? (ms->ref[sidx] + lg2(L)) * 0.69314718055994531f : -INFINITY;
      if (a.part_row0 < 0) {
        if (p.lse) p.lse[a.qrow0 + sidx] = lse_v;
      } else {
        p.part_lse[a.part_row0 + sidx] = lse_v;
      }
    }
    ok = group_sync(&ms->grp_softmax, gphase, abort, p.status);
  }
  if (ok) {
    const int dv_in_blk = qd * 32 + lane;
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
      const int dv = blk * 128 + dv_in_blk;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        float o[16];
        ptx::tmem_ld16(a.tmem + kTmemO + 64 * blk + lane_off + 16 * c, o);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int n = 16 * c + j;
          if (n < a.nrows) {
            const float L = ms->lsum[n];
            const float v = L > 0.f ? o[j] * (p.out_scale / L) : 0.f;
            if (a.part_row0 < 0)
              p.out[(size_t)(a.qrow0 + n) * kDv + dv] = __float2bfloat16_rn(v);
            else
              p.part_o[(size_t)(a.part_row0 + n) * kDv + dv] = v;
          }
        }
      }
    }
  }
}

template <bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
    fold_decode_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_kv, Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base (the 128-byte swizzle atoms), kept in the shared window
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
  Misc* ms = (Misc*)(smem + kOffMisc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort = &ms->abort;

  ptx::pdl_launch_dependents();

  const PlanHeader* ph = (const PlanHeader*)p.plan;
  if (tid == 0) {
    const PlanUnit* u = (const PlanUnit*)(p.plan + ph->units_off) + blockIdx.x;
    const PlanRequest* r = (const PlanRequest*)(p.plan + ph->req_off) + u->b;
    ms->unit[0] = u->b; ms->unit[1] = u->qrow0; ms->unit[2] = u->nrows; ms->unit[3] = u->kv_begin;
    ms->unit[4] = u->kv_end; ms->unit[5] = u->part_row0;
    ms->req[0] = r->ctx; ms->req[1] = r->q; ms->req[2] = r->tok0;
    int bad = (p.seq_lens[u->b] != r->ctx || p.q_lens[u->b] != r->q) ? 1 : 0;
    if (bad) report(p.status, MLA_DEVICE_PLAN_MISMATCH);
    ms->abort = bad;
    ptx::mbar_init(&ms->bar_q, 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&ms->kv_full[i], 1);
      ptx::mbar_init(&ms->kv_empty[i], kMmaWarps);
      ptx::mbar_init(&ms->p_full[i], 4);
      ptx::mbar_init(&ms->pt_empty[i], kMmaWarps);
    }
    ptx::mbar_init(&ms->s_full, kMmaWarps);
    ptx::mbar_init(&ms->s_empty, 4);
    ptx::mbar_init(&ms->mma_done, kMmaWarps);
    ptx::mbar_init(&ms->grp_softmax, 4);
    ptx::mbar_init(&ms->grp_mma, kMmaWarps);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&ms->tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();

  const int b = ms->unit[0], qrow0 = ms->unit[1], nrows = ms->unit[2];
  const int kv_begin = ms->unit[3], kv_end = ms->unit[4], part_row0 = ms->unit[5];
  const int ctx = ms->req[0], qlen = ms->req[1], tok0 = ms->req[2];
  const int ntiles = (kv_end - kv_begin + kTileKeys - 1) / kTileKeys;
  const int nmma = (nrows + 15) & ~15;   // MMA N (rows rounded up to 16)
  const int nch = nmma / 16;             // 16-column chunks of S^T / O^T
  const uint32_t tmem = ms->tmem_base;
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sKv = smem + kOffKv;
  uint8_t* sPt = smem + kOffPt;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int issued = 0;
    bool q_issued = false;
    if (!*abort) {
      q_issued = true;
      if (lane == 0) {
        ptx::prefetch_tmap(&tmap_q);
        ptx::prefetch_tmap(&tmap_kv);
        ptx::mbar_arrive_expect_tx(&ms->bar_q, kQBytes);
        ptx::tma_load_3d(sQ, &tmap_q, &ms->bar_q, 0, qrow0, 0);
      }
      const int32_t* pt_row = p.page_table + (size_t)b * p.pt_stride + kv_begin / kPage;
      for (int t0 = 0; t0 < ntiles && !*abort; t0 += 32) {
        int pid = 0;
        if (t0 + lane < ntiles) {
          pid = pt_row[t0 + lane];
          if (pid < 0 || pid >= p.num_pages) {
            report(p.status, MLA_DEVICE_BAD_PAGE);
            pid = 0;
          }
        }
        const int cnt = min(32, ntiles - t0);
        for (int i = 0; i < cnt; ++i) {
          const int page = __shfl_sync(0xffffffffu, pid, i);
          const int t = t0 + i, slot = t & 1;
          int ok = 1;
          if (lane == 0) {
            if (t >= 2) ok = wait_bar(&ms->kv_empty[slot], ((t - 2) >> 1) & 1, abort, p.status);
            if (ok) {
              uint8_t* dst = sKv + slot * kSlotBytes;
              if (kFp8) {
                ptx::mbar_arrive_expect_tx(&ms->kv_full[slot], kChunks * kFp8ChunkBytes);
                ptx::tma_load_3d(dst + kFp8StageOff, &tmap_kv, &ms->kv_full[slot], 0, page * kPage, 0);
              } else {
                ptx::mbar_arrive_expect_tx(&ms->kv_full[slot], kSlotBytes);
                ptx::tma_load_3d(dst, &tmap_kv, &ms->kv_full[slot], 0, page * kPage, 0);
              }
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          issued = t + 1;
        }
      }
    }
    // Drain: every issued copy must land before the CTA may exit (at most the last two
    // pages can still be in flight; earlier ones were consumed by the MMAs).
    if (lane == 0) {
      for (int t = max(0, issued - 2); t < issued; ++t) {
        long long t0c = clock64();
        while (!ptx::mbar_try_wait(&ms->kv_full[t & 1], (t >> 1) & 1) && clock64() - t0c < kWaitBudget) {
        }
      }
      if (q_issued) {
        long long t0c = clock64();
        while (!ptx::mbar_try_wait(&ms->bar_q, 0) && clock64() - t0c < kWaitBudget) {
        }
      }
    }
  } else if (warp <= kMmaWarps) {
    // ------------------------------------------------------------ MMA issue (+ fp8 expand)
    const int pw = warp - 1;                   // 0..3
    const int c_lo = chunk_lo(pw), c_hi = chunk_lo(pw + 1);
    const uint32_t sq = ptx::smem_addr(sQ), skv = ptx::smem_addr(sKv), spt = ptx::smem_addr(sPt);
    const uint32_t idesc_s = ptx::idesc_bf16(64, nmma, 0, 0);    // S^T: K-major K tile, K-major Q
    const uint32_t idesc_o = ptx::idesc_bf16(128, nmma, 1, 1);   // O^T: MN-major V^T, MN-major P^T
    const uint32_t d_s = tmem + kTmemS + 64 * pw, d_o = tmem + kTmemO + 64 * pw;
    uint32_t gphase = 0;
    bool ok = !*abort && warp_wait(&ms->bar_q, 0, abort, p.status);
    bool issued_any = false;
    // Event loop: issue whichever product is ready, O^T first. S^T(t1) needs page t1 and
    // the softmax's read of S^T(t1-1); O^T(t2) needs P^T(t2). O^T(t2) must not wait for
    // page t2+1, or the slot of page t2 (and so the load of page t2+2) would be held back.
    int t1 = 0, t2 = 0;
    long long idle_t0 = clock64();
    while (ok && t2 < ntiles) {
      bool progressed = false;
      if (t2 < t1) {
        int rdy = 0;
        if (lane == 0) rdy = ptx::mbar_test_wait(&ms->p_full[t2 & 1], (t2 >> 1) & 1);
        if (__shfl_sync(0xffffffffu, rdy, 0)) {
          const int ub = t2 & 1;
          ptx::tc_fence_after();
          if (lane == 0) {
            const uint32_t v0 = skv + ub * kSlotBytes + 2 * pw * kKvChunkBytes, pt0 = spt + ub * kPtBytes;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint64_t ad = ptx::smem_desc(v0 + 2048 * k, kKvChunkBytes, 1024, ptx::kSwizzle128B);
              uint64_t bd = ptx::smem_desc(pt0 + 2048 * k, 8192, 1024, ptx::kSwizzle128B);
              ptx::mma_bf16_ss(d_o, ad, bd, idesc_o, (t2 > 0 || k > 0) ? 1u : 0u);
            }
            ptx::mma_commit(&ms->kv_empty[ub]);
            ptx::mma_commit(&ms->pt_empty[ub]);
          }
          __syncwarp();
          ++t2;
          progressed = true;
        }
      }
      if (t1 < ntiles && t1 <= t2 + 1) {
        int rdy = 0;
        if (lane == 0)
          rdy = ptx::mbar_test_wait(&ms->kv_full[t1 & 1], (t1 >> 1) & 1) &&
                (t1 == 0 || ptx::mbar_test_wait(&ms->s_empty, (t1 - 1) & 1));
        if (__shfl_sync(0xffffffffu, rdy, 0)) {
          const int slot = t1 & 1;
          if (kFp8) {
            // this warp's chunks: read every e4m3 byte first (the bf16 rows overwrite the
            // e4m3 staging area of other chunks), then write the bf16 rows. Lane l reads the
            // 16-byte pieces l, l+32, ... of a chunk (conflict-free): key 8i + l/4, columns
            // 16 (l%4) .. 16 (l%4) + 15.
            uint8_t* base = sKv + slot * kSlotBytes;
            uint4 raw[3][8];
#pragma unroll
            for (int ci = 0; ci < 3; ++ci)
              if (c_lo + ci < c_hi)
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  raw[ci][i] = *reinterpret_cast<const uint4*>(base + kFp8StageOff + (c_lo + ci) * kFp8ChunkBytes +
                                                               i * 512 + 16 * lane);
            ok = group_sync(&ms->grp_mma, gphase, abort, p.status);
            if (!ok) break;
            const int j = lane & 3;
            // one warp-uniform decision per page: integer expansion unless this warp's share
            // holds a code that needs the exact conversion (zero, subnormal, NaN)
            uint32_t special = 0;
#pragma unroll
            for (int ci = 0; ci < 3; ++ci)
              if (c_lo + ci < c_hi)
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  special |= e4m3x4_special(raw[ci][i].x) | e4m3x4_special(raw[ci][i].y) |
                             e4m3x4_special(raw[ci][i].z) | e4m3x4_special(raw[ci][i].w);
            if (!__any_sync(0xffffffffu, special != 0u)) {
#pragma unroll
              for (int ci = 0; ci < 3; ++ci)
                if (c_lo + ci < c_hi)
#pragma unroll
                  for (int i = 0; i < 8; ++i) {
                    const int key = 8 * i + (lane >> 2);
                    uint8_t* line = base + (c_lo + ci) * kKvChunkBytes + key * 128;
                    uint4 o0, o1;
                    e4m3x4_to_bf16x4_normal(raw[ci][i].x, o0.x, o0.y);
                    e4m3x4_to_bf16x4_normal(raw[ci][i].y, o0.z, o0.w);
                    e4m3x4_to_bf16x4_normal(raw[ci][i].z, o1.x, o1.y);
                    e4m3x4_to_bf16x4_normal(raw[ci][i].w, o1.z, o1.w);
                    *reinterpret_cast<uint4*>(line + (((2 * j) ^ (key & 7)) << 4)) = o0;
                    *reinterpret_cast<uint4*>(line + (((2 * j + 1) ^ (key & 7)) << 4)) = o1;
                  }
            } else {
#pragma unroll
              for (int ci = 0; ci < 3; ++ci)
                if (c_lo + ci < c_hi)
#pragma unroll
                  for (int i = 0; i < 8; ++i) {
                    const int key = 8 * i + (lane >> 2);
                    uint8_t* line = base + (c_lo + ci) * kKvChunkBytes + key * 128;
                    uint4 o0, o1;
                    e4m3x4_to_bf16x4_cvt(raw[ci][i].x, o0.x, o0.y);
                    e4m3x4_to_bf16x4_cvt(raw[ci][i].y, o0.z, o0.w);
                    e4m3x4_to_bf16x4_cvt(raw[ci][i].z, o1.x, o1.y);
                    e4m3x4_to_bf16x4_cvt(raw[ci][i].w, o1.z, o1.w);
                    *reinterpret_cast<uint4*>(line + (((2 * j) ^ (key & 7)) << 4)) = o0;
                    *reinterpret_cast<uint4*>(line + (((2 * j + 1) ^ (key & 7)) << 4)) = o1;
                  }
            }
            ptx::fence_async_smem();
            // the K-steps of this warp's S^T MMAs span chunks expanded by other warps
            ok = group_sync(&ms->grp_mma, gphase, abort, p.status);
            if (!ok) break;
          }
          ptx::tc_fence_after();
          if (lane == 0) {
            const uint32_t a0 = skv + slot * kSlotBytes;
#pragma unroll
            for (int i = 0; i < kKStepsPerWarp; ++i) {
              const int ks = kKStepsPerWarp * pw + i, c = ks >> 2, k = ks & 3;
              uint64_t ad = ptx::smem_desc(a0 + c * kKvChunkBytes + 32 * k, 16, 1024, ptx::kSwizzle128B);
              uint64_t bd = ptx::smem_desc(sq + c * kQChunkBytes + 32 * k, 16, 1024, ptx::kSwizzle128B);
              ptx::mma_bf16_ss(d_s, ad, bd, idesc_s, i != 0 ? 1u : 0u);
            }
            ptx::mma_commit(&ms->s_full);
          }
          __syncwarp();
          issued_any = true;
          ++t1;
          progressed = true;
        }
      }
      if (progressed) {
        idle_t0 = clock64();
      } else {
        __nanosleep(32);  // leave issue slots to the softmax warps on this SM sub-partition
        int stop = 0;
        if (lane == 0) {
          if (*abort) {
            stop = 1;
          } else if (clock64() - idle_t0 > kWaitBudget) {
            *abort = 1;
            report(p.status, MLA_DEVICE_WAIT_TIMEOUT);
            stop = 1;
          }
        }
        if (__shfl_sync(0xffffffffu, stop, 0)) ok = false;
      }
    }
    // every MMA this warp issued must retire before TMEM is released
    if (issued_any) {
      if (lane == 0) {
        ptx::mma_commit(&ms->mma_done);
        long long t0c = clock64();
        while (!ptx::mbar_try_wait(&ms->mma_done, 0) && clock64() - t0c < kWaitBudget) {
          if (*abort) break;  // the other MMA warps may not commit; the tensor core drains anyway
        }
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const SoftmaxArgs a{ms, sKv, sPt, tmem, warp & 3, lane, tid - 32 * (kMmaWarps + 1), nrows, qrow0, kv_begin, kv_end,
                        ntiles, part_row0, ctx, qlen, tok0, abort};
    if (nch == 1)
      softmax_role<1>(a, p);
    else if (nch == 2)
      softmax_role<2>(a, p);
    else
      softmax_role<3>(a, p);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ LSE merge
// One CTA per (packed row, quarter of the 512 value columns): 8 warps share the
// splits of the row. L = ln sum_s exp(L_s), O = sum_s exp(L_s - L) O_s; a split that
// a causal row cannot see has L_s = -inf and weight 0.
constexpr int kMergeThreads = 256;
constexpr int kMergeMaxSplits = 2048;

__global__ void __launch_bounds__(kMergeThreads) lse_merge_kernel(const uint8_t* plan, const float* part_o,
                                                                 const float* part_lse, __nv_bfloat16* out, float* lse) {
  ptx::pdl_wait_primary();
  __shared__ float w_s[kMergeMaxSplits];
  __shared__ float red[8][2];
  __shared__ float4 acc_s[8][32];
  const PlanHeader* ph = (const PlanHeader*)plan;
  const PlanMerge m = ((const PlanMerge*)(plan + ph->merge_off))[blockIdx.y];
  const int row = blockIdx.x >> 2, quarter = blockIdx.x & 3;
  if (row >= m.nrows) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ns = m.n_splits;  // the planner keeps this <= kMergeMaxSplits
  // 1. L over the splits
  float mx = -INFINITY;
  for (int s = threadIdx.x; s < ns; s += kMergeThreads) {
    const float v = part_lse[m.part_row0 + s * m.nrows + row];
    w_s[s] = v;
    mx = fmaxf(mx, v);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red[warp][0] = mx;
  __syncthreads();
  mx = red[0][0];
#pragma unroll
  for (int i = 1; i < 8; ++i) mx = fmaxf(mx, red[i][0]);
  float sum = 0.f;
  for (int s = threadIdx.x; s < ns; s += kMergeThreads) {
    const float v = w_s[s];
    sum += v == -INFINITY ? 0.f : __expf(v - mx);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) red[warp][1] = sum;
  __syncthreads();
  sum = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) sum += red[i][1];
  const float L = mx + __logf(sum);
  for (int s = threadIdx.x; s < ns; s += kMergeThreads) {
    const float v = w_s[s];
    w_s[s] = v == -INFINITY ? 0.f : __expf(v - L);
  }
  __syncthreads();
  // 2. weighted sum: warp w takes splits w, w+8, ...; each lane takes 4 consecutive columns
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int col = quarter * 128 + 4 * lane;
  int s = warp;
  for (; s + 8 < ns; s += 16) {
    const float4 a = *reinterpret_cast<const float4*>(part_o + (size_t)(m.part_row0 + s * m.nrows + row) * kDv + col);
    const float4 c = *reinterpret_cast<const float4*>(part_o + (size_t)(m.part_row0 + (s + 8) * m.nrows + row) * kDv + col);
    const float wa = w_s[s], wc = w_s[s + 8];
    acc.x += wa * a.x + wc * c.x; acc.y += wa * a.y + wc * c.y;
    acc.z += wa * a.z + wc * c.z; acc.w += wa * a.w + wc * c.w;
  }
  for (; s < ns; s += 8) {
    const float4 a = *reinterpret_cast<const float4*>(part_o + (size_t)(m.part_row0 + s * m.nrows + row) * kDv + col);
    const float wa = w_s[s];
    acc.x += wa * a.x; acc.y += wa * a.y; acc.z += wa * a.z; acc.w += wa * a.w;
  }
  acc_s[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
    float4 r = acc_s[0][lane];
#pragma unroll
    for (int i = 1; i < 8; ++i) {
      const float4 v = acc_s[i][lane];
      r.x += v.x; r.y += v.y; r.z += v.z; r.w += v.w;
    }
    const int qr = m.qrow0 + row;
    uint2 pk = make_uint2(pack_bf16(r.x, r.y), pack_bf16(r.z, r.w));
    *reinterpret_cast<uint2*>(out + (size_t)qr * kDv + col) = pk;
    if (lse && quarter == 0 && lane == 0) lse[qr] = L;
  }
}

int rows_cap_for(int kv_dtype) {
  (void)kv_dtype;
  return kRowsCap;
}

int max_splits_for_merge() { return kMergeMaxSplits; }

// ------------------------------------------------------------------ host side
size_t workspace_bytes_for(int n_part_rows);
int check_plan(const void* plan_host, size_t plan_bytes, const PlanHeader** out);

static PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
  });
  return fn;
}

struct DeviceInfo {
  bool checked = false, ok = false, attrs_set = false;
  int major = 0, minor = 0;
};
static DeviceInfo g_dev[64];
static std::mutex g_dev_mu;

static int prepare_device(int dev) {
  if (dev < 0 || dev >= 64) return set_error(MLA_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.checked) {
    cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
    d.ok = (d.major == 10 && d.minor == 3);
    d.checked = true;
  }
  if (!d.ok)
    return set_error(MLA_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a (GB300)", dev, d.major,
                     d.minor);
  if (!d.attrs_set) {
    cudaError_t e1 = cudaFuncSetAttribute(fold_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    cudaError_t e2 = cudaFuncSetAttribute(fold_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e1 != cudaSuccess || e2 != cudaSuccess)
      return set_error(MLA_ERR_CUDA, "cudaFuncSetAttribute failed: %s", cudaGetErrorString(e1 != cudaSuccess ? e1 : e2));
    d.attrs_set = true;
  }
  return MLA_OK;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Tensor map of a [rows, 576] matrix viewed as (64 columns, rows, 9 column chunks): one
// box of (64, box_rows, 9) lands in shared memory as [chunk][row][64 columns].
static CUresult encode_chunked(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, const void* base, bool fp8,
                               uint64_t rows, uint32_t box_rows) {
  const uint64_t esz = fp8 ? 1 : 2;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)kChunks};
  cuuint64_t strides[2] = {(cuuint64_t)(kDqk * esz), (cuuint64_t)(64 * esz)};
  cuuint32_t box[3] = {64, box_rows, (cuuint32_t)kChunks};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
             dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace mla

using namespace mla;

extern "C" int mla_decode_run(const void* plan_dev, const void* plan_host, size_t plan_bytes, const void* q,
                              const void* kv_cache, const int32_t* page_table, int page_table_stride, int num_pages,
                              const int32_t* seq_lens, const int32_t* q_lens, float sm_scale, float kv_scale, void* out,
                              float* lse, void* workspace, size_t workspace_bytes, int32_t* status_dev, void* stream) {
  clear_error();
  const PlanHeader* h = nullptr;
  int rc = check_plan(plan_host, plan_bytes, &h);
  if (rc != MLA_OK) return rc;
  if (!plan_dev || !q || !kv_cache || !page_table || !seq_lens || !q_lens || !out)
    return set_error(MLA_ERR_INVALID_ARG, "plan_dev, q, kv_cache, page_table, seq_lens, q_lens and out must not be NULL");
  if (!aligned16(plan_dev) || !aligned16(q) || !aligned16(kv_cache) || !aligned16(out))
    return set_error(MLA_ERR_INVALID_ARG, "plan_dev, q, kv_cache and out must be 16-byte aligned");
  if (((uintptr_t)page_table & 3u) || ((uintptr_t)seq_lens & 3u) || ((uintptr_t)q_lens & 3u) || ((uintptr_t)lse & 3u) ||
      ((uintptr_t)status_dev & 3u))
    return set_error(MLA_ERR_INVALID_ARG, "page_table, seq_lens, q_lens, lse and status_dev must be 4-byte aligned");
  if (num_pages < 1) return set_error(MLA_ERR_INVALID_ARG, "num_pages must be >= 1 (got %d)", num_pages);
  if (page_table_stride < h->max_pages)
    return set_error(MLA_ERR_INVALID_ARG, "page_table_stride %d is smaller than the %d pages of the longest request",
                     page_table_stride, h->max_pages);
  if (!(sm_scale > 0.f) || !(kv_scale > 0.f) || !isfinite(sm_scale) || !isfinite(kv_scale))
    return set_error(MLA_ERR_INVALID_ARG, "sm_scale and kv_scale must be finite and > 0");
  const size_t ws_need = workspace_bytes_for(h->n_part_rows);
  if (ws_need > 0 && (!workspace || workspace_bytes < ws_need))
    return set_error(MLA_ERR_BUFFER, "workspace needs %zu bytes (got %zu)", ws_need, workspace ? workspace_bytes : (size_t)0);
  if (ws_need > 0 && ((uintptr_t)workspace & 255u)) return set_error(MLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if ((long long)num_pages * kPage > 0xFFFFFFFFLL) return set_error(MLA_ERR_INVALID_ARG, "num_pages too large");
  if (h->n_units == 0) return MLA_OK;

  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return set_error(MLA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(ce));
  rc = prepare_device(dev);
  if (rc != MLA_OK) return rc;
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encoder();
  if (!enc) return set_error(MLA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");

  const bool fp8 = h->kv_dtype == MLA_KV_FP8_E4M3;
  alignas(64) CUtensorMap tq, tkv;
  CUresult r = encode_chunked(enc, &tq, q, false, (uint64_t)h->total_q * (uint64_t)h->num_heads, kRowsCap);
  if (r != CUDA_SUCCESS) return set_error(MLA_ERR_CUDA, "tensor map for q failed (CUresult %d)", (int)r);
  r = encode_chunked(enc, &tkv, kv_cache, fp8, (uint64_t)num_pages * kPage, kTileKeys);
  if (r != CUDA_SUCCESS) return set_error(MLA_ERR_CUDA, "tensor map for kv_cache failed (CUresult %d)", (int)r);

  Params prm;
  prm.plan = (const uint8_t*)plan_dev;
  prm.page_table = page_table;
  prm.pt_stride = page_table_stride;
  prm.num_pages = num_pages;
  prm.H = h->num_heads;
  prm.seq_lens = seq_lens;
  prm.q_lens = q_lens;
  const float ks = fp8 ? kv_scale : 1.0f;
  prm.score_scale_log2 = sm_scale * ks * 1.4426950408889634f;
  prm.out_scale = ks;
  prm.out = (__nv_bfloat16*)out;
  prm.lse = lse;
  prm.part_o = (float*)workspace;
  prm.part_lse = ws_need ? (float*)((uint8_t*)workspace + ((size_t)h->n_part_rows * kDv * sizeof(float) + 255) / 256 * 256)
                         : nullptr;
  prm.status = status_dev;
  cudaStream_t st = (cudaStream_t)stream;
  if (fp8)
    fold_decode_kernel<true><<<h->n_units, kThreads, kSmemBytes, st>>>(tq, tkv, prm);
  else
    fold_decode_kernel<false><<<h->n_units, kThreads, kSmemBytes, st>>>(tq, tkv, prm);
  ce = cudaGetLastError();
  if (ce != cudaSuccess) return set_error(MLA_ERR_CUDA, "fold kernel launch: %s", cudaGetErrorString(ce));
  if (h->n_merge > 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(h->rows_cap * 4), (unsigned)h->n_merge, 1);
    cfg.blockDim = dim3(kMergeThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    ce = cudaLaunchKernelEx(&cfg, lse_merge_kernel, (const uint8_t*)plan_dev, (const float*)prm.part_o,
                            (const float*)prm.part_lse, (__nv_bfloat16*)out, lse);
    if (ce != cudaSuccess) return set_error(MLA_ERR_CUDA, "merge kernel launch: %s", cudaGetErrorString(ce));
  }
  return MLA_OK;
}
