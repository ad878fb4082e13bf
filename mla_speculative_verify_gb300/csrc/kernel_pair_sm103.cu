// kernel_pair_sm103.cu -- the verify decode for fold groups of 49..96 packed rows with a
// bf16 cache, on clusters of two CTAs (sm_103a).
//
// A fold group of H * F packed rows (sglang PR #33650, "Why" paragraph: the q verify
// tokens folded into the rows) that is wider than one CTA's 48-row tile would otherwise
// stream every page through two CTAs, each holding the whole 72 KB page for its half of
// the rows. Here the two CTAs of a cluster split the page's COLUMNS instead (the wide
// kernel of flashinfer PR #5602, "What r52 changes", splits O between two CTAs; this is
// that split in the transposed orientation):
//
//   CTA c holds the latent columns [256 c, 256 c + 256) of every key (chunks 4c .. 4c+3)
//   and the 64 rope columns (chunk 8), i.e. 40 KB per page, so three page stages fit
//   beside its 96-row Q slice (61 KB). For all rows it computes the partial scores
//     S^T_c[key, row] = K[key, cols_c] . Q[row, cols_c]^T   (18 K-steps: 16 latent + 2 rope)
//   and sends them to the other CTA through distributed shared memory (st.async, whose
//   completion is counted on the receiver's mbarrier) one tile ahead of their use. Each
//   CTA adds the two partials (p0 + p1 in both: fp32 addition is commutative, so both
//   CTAs hold the same scores bit for bit) and runs the online softmax of all rows (the
//   lazy per-row reference of flashinfer PR #5602) itself, so the two CTAs take the same
//   decisions without exchanging P or row scales. Each then accumulates its half of the
//   values
//     O^T_c[dv, row] += V^T[dv in 256 c .. 256 c + 255, key] . P^T[key, row]
//   for all rows (two 128-row value blocks, N = rows) in tensor memory.
//
// Per page and CTA that is 18 S^T MMAs (N <= 96) and 8 O^T MMAs against 36 + 16 per
// 48-row tile in the single-CTA kernel, and every page is read by the pair once. The one
// exchange per tile is off the critical path: the partials of tile t + 1 leave while the
// softmax works on tile t (S^T is double-buffered in tensor memory).
//
// Warps (one CTA per SM, 11 warps): warp 0 the TMA producer (the Q slice once, then the
// 40 KB column half of each page into a three-stage ring, with an L2 prefetch of the page
// that enters the ring next); warp 1 issues S^T (18 K-steps per tile into buffer t % 2);
// warp 2 issues O^T (two value blocks) once the softmax has closed P^T(t); warps 3-10 the
// softmax (two per TMEM lane quadrant). Every accumulator has one writer, so a unit's
// results are the same bit for bit on every run. Every wait is bounded; waits on the other
// CTA acquire at cluster scope.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "decode_common.cuh"
#include "mla_decode.h"
#include "plan_format.h"
#include "ptx.cuh"
#include "status.h"

namespace mla {
namespace pair {

constexpr int kRows = 96;                        // packed rows of a unit (both CTAs)
constexpr int kHalf = 48;                        // rows whose LSE one CTA writes
constexpr int kChunks = 5;                       // 64-column chunks per CTA: 4 latent + rope
constexpr int kChunkBytes = 64 * 128;            // 64 keys x 64 bf16 columns (128-byte swizzle rows)
constexpr int kSlot = kChunks * kChunkBytes;     // 40960: one page's column half
constexpr int kStages = 3;
constexpr int kQChunkBytes = kRows * 128;        // 12288
constexpr int kQBytes = kChunks * kQChunkBytes;  // 61440
constexpr int kPtBytes = kRows * 128;            // P^T, K-major: [row][64 keys] bf16
constexpr int kXFloats = 24;                     // partial scores a softmax thread sends per tile (<= 6 chunks x 4)
constexpr int kXBytes = kSoftmaxThreads * kXFloats * 4;  // 24576
constexpr int kOffQ = 0;
constexpr int kOffKv = kOffQ + kQBytes;
constexpr int kOffPt = kOffKv + kStages * kSlot;
constexpr int kOffX = kOffPt + kPtBytes;
constexpr int kOffMisc = kOffX + kXBytes;
constexpr int kMiscBytes = 4096;
constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-CTA shared memory");
static_assert(kOffKv % 1024 == 0 && kOffPt % 1024 == 0 && kOffX % 1024 == 0 && kOffMisc % 1024 == 0,
              "1024-byte swizzle atoms");
constexpr int kSWarp = 1, kOWarp = 2;
constexpr int kFirstSoftmaxWarp = 3;
constexpr int kThreads = 32 * (kFirstSoftmaxWarp + kSoftmaxWarps);  // 352
// TMEM (512 columns): O^T value blocks 0 and 1 (this CTA's 256 value columns) at columns 0
// and 128, S^T buffer b at 256 + 128 b; N <= 96 columns each
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemS = 256;
constexpr float kRefSlack = 8.0f;  // octaves a score may exceed the row reference before it moves

struct Misc {
  uint64_t bar_q;
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], s_empty[2];
  uint64_t pt_empty;  // O^T(t) is done (P^T buffer free, O^T may be rescaled): one commit per tile
  uint64_t p_ready;   // the softmax warps closed P^T(t) (8 arrivals per tile)
  uint64_t x_full;    // the other CTA's partial scores of tile t arrived (1 arming arrival + bytes)
  uint64_t x_free;    // the other CTA read the partial scores this CTA sent (8 arrivals per tile)
  uint64_t mma_done[4];
  uint32_t tmem_base;
  int abort;
  int unit[12];
  alignas(16) float ref[kRows];
  alignas(16) float alpha[kRows];
  alignas(16) int lim[kRows];
  alignas(16) float colred[4][kRows];
  alignas(16) float oscale[kRows];  // output scale / l of every row
};
static_assert(sizeof(Misc) <= kMiscBytes, "misc block too small");

struct Args {
  Misc* ms;
  uint8_t* sKv;
  uint8_t* sPt;
  uint8_t* sX;
  uint32_t tmem;
  uint32_t crank, peer;
  int qd, grp, lane, sidx, nmma, nrows, qrow0, kv_begin, kv_end, ntiles, part_row0, b, ctx, qlen, tok0;
  volatile int* abort;
};

// Byte offset of P^T(row, key) in a K-major buffer of 128-byte rows, 128-byte swizzle.
__device__ __forceinline__ uint32_t pt_offset(int row, int key) {
  return (uint32_t)(row * 128 + ((((key >> 3) ^ row) & 7) << 4) + (key & 7) * 2);
}

// The 4 NM scores (columns 16 c + 8 grp + 4 half + j, c < NM, j < 4) of this thread's key
// from S^T buffer `buf`: lanes 0..15 read 8 columns of each 16 and hand the upper 4 to
// lanes 16..31.
template <int NM>
__device__ __forceinline__ void read_scores(uint32_t tmem, uint32_t lane_off, int grp, int lane, int buf, float* v) {
  const int half = lane >> 4;
  const uint32_t base = tmem + kTmemS + 128 * buf + lane_off + 8 * grp;
#pragma unroll
  for (int c = 0; c < NM; ++c) {
    float s[8];
    ptx::tmem_ld8(base + 16 * c, s);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float hi = __shfl_sync(0xffffffffu, s[4 + j], lane & 15);
      v[4 * c + j] = half ? hi : s[j];
    }
  }
}

// Softmax warps of one CTA for all 16 NM rows of the unit. Warp (qd, grp) owns the 16
// keys of TMEM lane quadrant qd and, of every 16 columns, the 8 columns 8 grp .. 8 grp + 7.
// Per tile t: take the other CTA's partials of tile t; send this CTA's partials of tile
// t + 1; add this CTA's partials of tile t; mask, vote on reference moves, P^T.
template <int NM>
__device__ __forceinline__ void softmax_role(const Args& a, const Params& p) {
  constexpr int NC = 4 * NM;
  constexpr float kMoveAbove = kRefSlack;
  Misc* ms = a.ms;
  const int lane = a.lane, qd = a.qd, grp = a.grp, sidx = a.sidx;
  const int half = lane >> 4;
  const int krow = qd * 16 + (lane & 15);
  const int col0 = 8 * grp + 4 * half;
  const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
  const int w8 = sidx >> 5;
  const int r0 = kHalf * (int)a.crank;
  volatile int* abort = a.abort;
  if (sidx == 0 && (p.seq_lens[a.b] != a.ctx || p.q_lens[a.b] != a.qlen)) {
    report(p.status, MLA_DEVICE_PLAN_MISMATCH);
    *a.abort = 1;
  }
  {
    // O^T starts at zero: this warp clears its lane quadrant of value block grp
    float z[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) ptx::tmem_st16(a.tmem + kTmemO + lane_off + 128 * grp + 16 * c, z);
    ptx::tmem_st_wait();
    ptx::tc_fence_before();
  }
  if (sidx < kRows) {
    int lim = 0;
    if (sidx < a.nrows) {
      const int i = (a.qrow0 + sidx) / p.H - a.tok0;  // verify token of this packed row
      lim = a.ctx - a.qlen + i + 1;
    }
    ms->lim[sidx] = lim;
    ms->ref[sidx] = -INFINITY;
    ms->alpha[sidx] = 1.f;
  }
  // the other CTA's copy of this thread's slot of the partial-score buffer, and its barriers
  const uint32_t x_dst = ptx::mapa(ptx::smem_addr(a.sX + (size_t)(w8 * 32 + lane) * kXFloats * 4), a.peer);
  const uint32_t x_full_peer = ptx::mapa(ptx::smem_addr(&ms->x_full), a.peer);
  const uint32_t x_free_peer = ptx::mapa(ptx::smem_addr(&ms->x_free), a.peer);
  const float* xsrc = reinterpret_cast<const float*>(a.sX + (size_t)(w8 * 32 + lane) * kXFloats * 4);
  constexpr uint32_t kXTx = kSoftmaxThreads * NM * 16;  // bytes of one tile's partials
  // phase 0 of x_full: one arming arrival plus the other CTA's bytes (which may land first)
  if (sidx == 0) ptx::mbar_arrive_expect_tx(&ms->x_full, kXTx);

  bool stop = softmax_any(*abort != 0);
  bool fail = false;
  int lim_min = a.kv_end;
  for (int n = 0; n < a.nrows; ++n) lim_min = min(lim_min, ms->lim[n]);
  float l_acc[NC];
#pragma unroll
  for (int i = 0; i < NC; ++i) l_acc[i] = 0.f;
  const float scale = p.score_scale_log2;
  // send this CTA's partials of tile u (buffer u % 2) to the other CTA
  auto send = [&](int u) {
    if (!fail) fail = !warp_wait(&ms->s_full[u & 1], (u >> 1) & 1, abort, p);
    if (fail) return;
    ptx::tc_fence_after();
    float y[NC];
    read_scores<NM>(a.tmem, lane_off, grp, lane, u & 1, y);
    // the other CTA has read the partials of tile u - 1 out of its single buffer
    if (u >= 1) fail = !warp_wait<true>(&ms->x_free, (u - 1) & 1, abort, p);
    if (fail) return;
#pragma unroll
    for (int c = 0; c < NM; ++c)
      ptx::st_async_v4f(x_dst + 16 * c, y[4 * c], y[4 * c + 1], y[4 * c + 2], y[4 * c + 3], x_full_peer);
  };
  if (!stop) send(0);
  for (int t = 0; !stop && t < a.ntiles; ++t) {
    float x[NC];
    bool need = false, unmasked = false;
    // ---- the other CTA's partials of tile t
    if (!fail) fail = !warp_wait<true>(&ms->x_full, t & 1, abort, p);
    if (!fail) {
#pragma unroll
      for (int c = 0; c < NM; ++c) {
        const float4 v = *reinterpret_cast<const float4*>(xsrc + 4 * c);
        x[4 * c] = v.x;
        x[4 * c + 1] = v.y;
        x[4 * c + 2] = v.z;
        x[4 * c + 3] = v.w;
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_remote(x_free_peer);
      if (sidx == 0 && t + 1 < a.ntiles) ptx::mbar_arrive_expect_tx(&ms->x_full, kXTx);  // arm phase t + 1
    }
    // ---- this CTA's partials of tile t + 1 leave now, one tile ahead of their use
    if (t + 1 < a.ntiles) send(t + 1);
    // ---- this CTA's partials of tile t: scores = (this CTA's) + (the other CTA's), in the
    // same order in both CTAs (p0 + p1 = p1 + p0 exactly)
    if (!fail) {
      ptx::tc_fence_after();
      float own[NC];
      read_scores<NM>(a.tmem, lane_off, grp, lane, t & 1, own);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&ms->s_empty[t & 1]);
#pragma unroll
      for (int i = 0; i < NC; ++i) x[i] = a.crank == 0 ? own[i] + x[i] : x[i] + own[i];
      const int key = a.kv_begin + t * 64 + krow;
      const int tile_last = a.kv_begin + t * 64 + 63;
      unmasked = tile_last < a.kv_end && tile_last < lim_min;
#pragma unroll
      for (int c = 0; c < NM; ++c) {
        const int n0 = 16 * c + col0;
        const float4 rr = *reinterpret_cast<const float4*>(&ms->ref[n0]);
        const float rrv[4] = {rr.x, rr.y, rr.z, rr.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float v = x[4 * c + j] * scale;
          if (!unmasked) v = (key < a.kv_end && key < ms->lim[n0 + j]) ? v : -INFINITY;
          x[4 * c + j] = v;
          need |= v > rrv[j] + kMoveAbove;
        }
      }
    }
    // ---- P^T(t) (K-major), written against the current references once O^T(t - 1) is done
    // with the buffer
    float pv[NC];
    auto make_p = [&]() {
#pragma unroll
      for (int c = 0; c < NM; ++c) {
        const float4 rr = *reinterpret_cast<const float4*>(&ms->ref[16 * c + col0]);
        const float rrv[4] = {rr.x, rr.y, rr.z, rr.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float v = x[4 * c + j];
          pv[4 * c + j] = (!unmasked && v == -INFINITY) ? 0.f : ex2(v - rrv[j]);
        }
      }
    };
    auto store_p = [&]() {
#pragma unroll
      for (int c = 0; c < NM; ++c)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<__nv_bfloat16*>(a.sPt + pt_offset(16 * c + col0 + j, krow)) = __float2bfloat16_rn(pv[4 * c + j]);
      const int key = a.kv_begin + t * 64 + krow;
      if (key >= a.kv_end) {
        // a cache slot past the key range: zero its value columns (this thread: value chunk
        // 2 grp + half of this CTA's four) so that P = 0 meets V = 0
        uint8_t* row = a.sKv + (t % kStages) * kSlot + (2 * grp + half) * kChunkBytes + krow * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(row + 16 * j) = make_uint4(0, 0, 0, 0);
      }
      ptx::fence_async_smem();
      ptx::tc_fence_before();
    };
    if (!fail) {
      make_p();
      if (t >= 1) fail = !warp_wait(&ms->pt_empty, (t - 1) & 1, abort, p);
    }
    if (!fail) store_p();
    // ---- one barrier closes P^T(t) and votes on reference moves
    if (softmax_any(need || fail || *abort != 0)) {
      if (softmax_any(fail || *abort != 0)) {
        stop = true;
        break;
      }
      // column maxima over the tile's keys, each row's reference up to its maximum, l and
      // O^T (tiles < t; O^T(t - 1) is done) rescaled by alpha, P^T(t) written again
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        float m = x[i];
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((lane & 15) == 0) ms->colred[qd][16 * (i / 4) + col0 + (i % 4)] = m;
      }
      softmax_sync();
      if (sidx < 16 * NM) {
        const float cm = fmaxf(fmaxf(ms->colred[0][sidx], ms->colred[1][sidx]), fmaxf(ms->colred[2][sidx], ms->colred[3][sidx]));
        const float old = ms->ref[sidx];
        const float nw = fmaxf(old, cm);
        ms->alpha[sidx] = (nw == old) ? 1.f : ex2(old - nw);
        ms->ref[sidx] = nw;
      }
      softmax_sync();
#pragma unroll
      for (int i = 0; i < NC; ++i) l_acc[i] *= ms->alpha[16 * (i / 4) + col0 + (i % 4)];
      if (t >= 1) {
        // this warp: value block grp of its lane quadrant, every row
        ptx::tc_fence_after();
        const uint32_t ta = a.tmem + kTmemO + 128 * grp + lane_off;
#pragma unroll
        for (int c = 0; c < NM; ++c) {
          float o[16];
          ptx::tmem_ld16(ta + 16 * c, o);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            const float4 al = *reinterpret_cast<const float4*>(&ms->alpha[16 * c + j]);
            o[j] *= al.x;
            o[j + 1] *= al.y;
            o[j + 2] *= al.z;
            o[j + 3] *= al.w;
          }
          ptx::tmem_st16(ta + 16 * c, o);
        }
        ptx::tmem_st_wait();
      }
      make_p();
      store_p();
      if (softmax_any(fail || *abort != 0)) {  // also closes the rewritten P^T(t)
        stop = true;
        break;
      }
    }
#pragma unroll
    for (int i = 0; i < NC; ++i) l_acc[i] += pv[i];
    // the O^T warp may multiply P^T(t)
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&ms->p_ready);
  }
  // ------------------------------------------------------------ epilogue
  if (!stop) {
#pragma unroll
    for (int i = 0; i < NC; ++i) {
      float s = l_acc[i];
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if ((lane & 15) == 0) ms->colred[qd][16 * (i / 4) + col0 + (i % 4)] = s;
    }
    softmax_sync();
    if (sidx < kRows) {
      float L = 0.f;
      if (sidx < a.nrows) {
        L = ms->colred[0][sidx] + ms->colred[1][sidx] + ms->colred[2][sidx] + ms->colred[3][sidx];
        if (sidx >= r0 && sidx < r0 + kHalf) {  // each CTA writes the LSE of half the rows
          const float lse_v = L > 0.f ? (ms->ref[sidx] + lg2(L)) * 0.69314718055994531f : -INFINITY;
          if (a.part_row0 < 0) {
            if (p.lse) p.lse[a.qrow0 + sidx] = lse_v;
          } else {
            p.part_lse[a.part_row0 + sidx] = lse_v;
          }
        }
      }
      ms->oscale[sidx] = L > 0.f ? p.out_scale / L : 0.f;
    }
    if (!fail) fail = !warp_wait(&ms->pt_empty, (a.ntiles - 1) & 1, abort, p);
    stop = softmax_any(fail || *abort != 0);  // also publishes oscale to all softmax warps
  }
  if (stop) return;
  ptx::tc_fence_after();
  // O(row, dv) = O^T(dv, row) * oscale(row): this thread holds dv = 256 crank + 128 grp +
  // 32 qd + lane, every row of the unit
  __nv_bfloat16* dst = a.part_row0 < 0 ? p.out + (size_t)a.qrow0 * kDv : p.part_o + (size_t)a.part_row0 * kDv;
  const int dv = 256 * (int)a.crank + 128 * grp + 32 * qd + lane;
#pragma unroll 1
  for (int c = 0; c < NM; ++c) {
    float o[16];
    ptx::tmem_ld16(a.tmem + kTmemO + 128 * grp + lane_off + 16 * c, o);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int n = 16 * c + j;
      if (n < a.nrows) dst[(size_t)n * kDv + dv] = __float2bfloat16_rn(o[j] * ms->oscale[n]);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    fold_pair_kernel(const __grid_constant__ CUtensorMap tq4, const __grid_constant__ CUtensorMap tq1,
                     const __grid_constant__ CUtensorMap tkv4, const __grid_constant__ CUtensorMap tkv1, Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base; the same offset in both CTAs of the cluster
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
  Misc* ms = (Misc*)(smem + kOffMisc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = ptx::cluster_ctarank(), peer = crank ^ 1u;
  volatile int* abort = &ms->abort;
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sKv = smem + kOffKv;
  uint8_t* sPt = smem + kOffPt;
  uint8_t* sX = smem + kOffX;
  constexpr int kUnitWords = (int)(sizeof(PlanUnit) / 4);
  const int unit_idx = blockIdx.x >> 1;

  ptx::pdl_launch_dependents();

  int pid_cur = 0, pid_next = 0;
  if (warp == 0) {
    if (lane == 0) {
      ms->abort = 0;
      ptx::mbar_init(&ms->bar_q, 1);
      for (int i = 0; i < kStages; ++i) {
        ptx::mbar_init(&ms->kv_full[i], 1);
        ptx::mbar_init(&ms->kv_empty[i], 1);  // the O^T warp's commit
      }
      for (int i = 0; i < 2; ++i) {
        ptx::mbar_init(&ms->s_full[i], 1);
        ptx::mbar_init(&ms->s_empty[i], kSoftmaxWarps);
      }
      ptx::mbar_init(&ms->pt_empty, 1);
      ptx::mbar_init(&ms->p_ready, kSoftmaxWarps);
      ptx::mbar_init(&ms->x_full, 1);
      ptx::mbar_init(&ms->x_free, kSoftmaxWarps);
      for (int i = 0; i < 4; ++i) ptx::mbar_init(&ms->mma_done[i], 1);
      ptx::fence_mbar_init();
    }
    int uw = 0;
    if (lane < kUnitWords) uw = reinterpret_cast<const int32_t*>(p.units + unit_idx)[lane];
    if (lane < kUnitWords) ms->unit[lane] = uw;
    const int ub = __shfl_sync(0xffffffffu, uw, 0), uq0 = __shfl_sync(0xffffffffu, uw, 1);
    const int ukb = __shfl_sync(0xffffffffu, uw, 3), uke = __shfl_sync(0xffffffffu, uw, 4);
    const int unt = (uke - ukb + 63) / 64;
    if (lane == 0) {
      ptx::prefetch_tmap(&tkv4);
      ptx::prefetch_tmap(&tkv1);
      ptx::prefetch_tmap(&tq4);
      ptx::prefetch_tmap(&tq1);
      ptx::mbar_arrive_expect_tx(&ms->bar_q, kQBytes);
      ptx::tma_load_3d(sQ, &tq4, &ms->bar_q, 0, uq0, 4 * (int)crank);
      ptx::tma_load_3d(sQ + 4 * kQChunkBytes, &tq1, &ms->bar_q, 0, uq0, 8);
    }
    const int32_t* pt_row = p.page_table + (size_t)ub * p.pt_stride + ukb / kPage;
    pid_cur = lane < unt ? pt_row[lane] : 0;
    pid_next = 32 + lane < unt ? pt_row[32 + lane] : 0;
  } else if (warp == 1) {
    ptx::tmem_alloc(&ms->tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // the other CTA's barriers are initialised before either CTA signals across the pair
  ptx::cluster_arrive();
  ptx::cluster_wait();

  const int b = ms->unit[0], qrow0 = ms->unit[1], nrows = ms->unit[2];
  const int kv_begin = ms->unit[3], kv_end = ms->unit[4], part_row0 = ms->unit[5];
  const int ctx = ms->unit[8], qlen = ms->unit[9], tok0 = ms->unit[10];
  const int ntiles = (kv_end - kv_begin + 63) / 64;
  const int nmma = (nrows + 15) & ~15;
  const uint32_t tmem = ms->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int issued = 0;
    const int32_t* pt_row = p.page_table + (size_t)b * p.pt_stride + kv_begin / kPage;
    auto checked = [&](int pid, int t) {
      if (t < ntiles && (pid < 0 || pid >= p.num_pages)) {
        report(p.status, MLA_DEVICE_BAD_PAGE);
        pid = 0;
      }
      return pid;
    };
    auto load_ids = [&](int t0) { return checked(t0 + lane < ntiles ? pt_row[t0 + lane] : 0, t0 + lane); };
    const bool read_once = (ms->unit[11] & kUnitKvReadOnce) != 0;
    const uint64_t pol = ptx::policy_evict_first();
    pid_cur = checked(pid_cur, lane);
    pid_next = checked(pid_next, 32 + lane);
    for (int t0 = 0; t0 < ntiles && !*abort; t0 += 32) {
      const int cnt = min(32, ntiles - t0);
      for (int i = 0; i < cnt; ++i) {
        const int page = __shfl_sync(0xffffffffu, pid_cur, i);
        const int tp = i + kStages;
        const int page_pf = __shfl_sync(0xffffffffu, tp < 32 ? pid_cur : pid_next, tp & 31);
        const int t = t0 + i, slot = t % kStages;
        // the slot of page t - S is free once O^T(t - S) is done (the whole warp waits)
        if (t >= kStages && !warp_wait(&ms->kv_empty[slot], ((t - kStages) / kStages) & 1, abort, p)) break;
        if (lane == 0 && !(blockIdx.x == 0 && t == p.skip_copy)) {
          uint8_t* dst = sKv + slot * kSlot;
          ptx::mbar_arrive_expect_tx(&ms->kv_full[slot], kSlot);
          if (read_once)
            ptx::tma_load_3d_hint(dst, &tkv4, &ms->kv_full[slot], 0, page * kPage, 4 * (int)crank, pol);
          else
            ptx::tma_load_3d(dst, &tkv4, &ms->kv_full[slot], 0, page * kPage, 4 * (int)crank);
          ptx::tma_load_3d(dst + 4 * kChunkBytes, &tkv1, &ms->kv_full[slot], 0, page * kPage, 8);
          if (t0 + tp < ntiles) {
            ptx::tma_prefetch_l2_3d(&tkv4, 0, page_pf * kPage, 4 * (int)crank);
            ptx::tma_prefetch_l2_3d(&tkv1, 0, page_pf * kPage, 8);
          }
        }
        __syncwarp();
        issued = t + 1;
      }
      pid_cur = pid_next;
      pid_next = (t0 + 64 < ntiles) ? load_ids(t0 + 64) : 0;
    }
    if (lane == 0) {
      // drain: every issued copy must land before the CTA may exit
      for (int t = max(0, issued - kStages); t < issued; ++t) {
        if (blockIdx.x == 0 && t == p.skip_copy) continue;
        long long t0c = clock64();
        while (!ptx::mbar_try_wait(&ms->kv_full[t % kStages], (t / kStages) & 1) && clock64() - t0c < p.wait_budget) {
        }
      }
      long long t0c = clock64();
      while (!ptx::mbar_try_wait(&ms->bar_q, 0) && clock64() - t0c < p.wait_budget) {
      }
    }
    __syncwarp();
  } else if (warp == kSWarp) {
    // ------------------------------------------------------------ S^T issue
    // K-steps 0..15 over this CTA's four latent chunks, then rope K-steps 2 crank and
    // 2 crank + 1 (the other CTA takes the other two), into buffer t % 2
    const uint32_t sq = ptx::smem_addr(sQ), skv = ptx::smem_addr(sKv);
    bool ok = !*abort && warp_wait(&ms->bar_q, 0, abort, p);
    bool issued = false;
    const uint32_t idesc_s = ptx::idesc_bf16(64, nmma, 0, 0);
    for (int t = 0; ok && t < ntiles; ++t) {
      ok = warp_wait(&ms->kv_full[t % kStages], (t / kStages) & 1, abort, p);
      if (ok && t >= 2) ok = warp_wait(&ms->s_empty[t & 1], ((t - 2) >> 1) & 1, abort, p);
      if (!ok) break;
      ptx::tc_fence_after();
      if (lane == 0) {
        const uint32_t a0 = skv + (t % kStages) * kSlot;
        const uint32_t d = tmem + kTmemS + 128 * (t & 1);
#pragma unroll
        for (int ks = 0; ks < 18; ++ks) {
          const int c = ks < 16 ? ks >> 2 : 4;
          const int k = ks < 16 ? ks & 3 : 2 * (int)crank + (ks - 16);
          const uint64_t ad = ptx::smem_desc(a0 + c * kChunkBytes + 32 * k, 16, 1024, ptx::kSwizzle128B);
          const uint64_t bd = ptx::smem_desc(sq + c * kQChunkBytes + 32 * k, 16, 1024, ptx::kSwizzle128B);
          ptx::mma_bf16_ss(d, ad, bd, idesc_s, ks != 0 ? 1u : 0u);
        }
        ptx::mma_commit(&ms->s_full[t & 1]);
      }
      __syncwarp();
      issued = true;
    }
    if (issued) {
      if (lane == 0) drain_mmas(&ms->mma_done[0], p.wait_budget);
      __syncwarp();
    }
  } else if (warp == kOWarp) {
    // ------------------------------------------------------------ O^T issue
    // O^T(t) += V^T . P^T(t) for this CTA's two value blocks once the softmax closed P^T(t)
    const uint32_t skv = ptx::smem_addr(sKv), spt = ptx::smem_addr(sPt);
    const uint32_t idesc_o = ptx::idesc_bf16(128, nmma, 1, 0);
    bool ok = true, issued = false;
    for (int t = 0; ok && t < ntiles; ++t) {
      ok = warp_wait(&ms->p_ready, t & 1, abort, p);
      if (!ok) break;
      ptx::tc_fence_after();
      if (lane == 0) {
        const uint32_t v0 = skv + (t % kStages) * kSlot;
#pragma unroll
        for (int blk = 0; blk < 2; ++blk)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t ad = ptx::smem_desc(v0 + 2 * blk * kChunkBytes + 2048 * k, kChunkBytes, 1024,
                                               ptx::kSwizzle128B);
            const uint64_t bd = ptx::smem_desc(spt + 32 * k, 16, 1024, ptx::kSwizzle128B);
            ptx::mma_bf16_ss(tmem + kTmemO + 128 * blk, ad, bd, idesc_o, 1u);
          }
        ptx::mma_commit(&ms->kv_empty[t % kStages]);
        ptx::mma_commit(&ms->pt_empty);
      }
      __syncwarp();
      issued = true;
    }
    if (issued) {
      if (lane == 0) drain_mmas(&ms->mma_done[1], p.wait_budget);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int sw = warp - kFirstSoftmaxWarp;
    const Args a{ms, sKv, sPt, sX, tmem, crank, peer, warp & 3, sw >> 2, lane, tid - 32 * kFirstSoftmaxWarp, nmma,
                 nrows, qrow0, kv_begin, kv_end, ntiles, part_row0, b, ctx, qlen, tok0, abort};
    if (nmma == 64)
      softmax_role<4>(a, p);
    else if (nmma == 80)
      softmax_role<5>(a, p);
    else
      softmax_role<6>(a, p);
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  // neither CTA leaves while the other may still write into its shared memory
  ptx::cluster_arrive();
  ptx::cluster_wait();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace pair

int pair_rows_cap() { return pair::kRows; }

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();  // defined next to the single-CTA kernel

// Tensor map of a bf16 [rows, 576] matrix viewed as (64 columns, rows, 9 column chunks)
// whose box is (64, box_rows, box_chunks): [chunk][row][64 columns] in shared memory.
static CUresult encode_box(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, const void* base, uint64_t rows,
                           uint32_t box_rows, uint32_t box_chunks) {
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, 9};
  cuuint64_t strides[2] = {(cuuint64_t)(kDqk * 2), 128};
  cuuint32_t box[3] = {64, box_rows, box_chunks};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

static std::mutex g_pair_mu;
static bool g_pair_attr[64];

static int set_pair_attrs(int dev) {
  if (dev < 0 || dev >= 64) return set_error(MLA_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_pair_mu);
  if (!g_pair_attr[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(pair::fold_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, pair::kSmemBytes);
    if (e != cudaSuccess) return set_error(MLA_ERR_CUDA, "cudaFuncSetAttribute (pair kernel): %s", cudaGetErrorString(e));
    g_pair_attr[dev] = true;
  }
  return MLA_OK;
}

static cudaLaunchConfig_t pair_config(unsigned grid, cudaStream_t st, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(pair::kThreads, 1, 1);
  cfg.dynamicSmemBytes = pair::kSmemBytes;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

int launch_pair_kernel(int dev, const PlanHeader* h, const void* q, const void* kv_cache, int num_pages,
                       const Params& prm, cudaStream_t st) {
  int rc = set_pair_attrs(dev);
  if (rc != MLA_OK) return rc;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return set_error(MLA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  alignas(64) CUtensorMap tq4, tq1, tkv4, tkv1;
  const uint64_t qrows = (uint64_t)h->total_q * (uint64_t)h->num_heads;
  const uint64_t kvrows = (uint64_t)num_pages * kPage;
  CUresult r = encode_box(enc, &tq4, q, qrows, pair::kRows, 4);
  if (r == CUDA_SUCCESS) r = encode_box(enc, &tq1, q, qrows, pair::kRows, 1);
  if (r == CUDA_SUCCESS) r = encode_box(enc, &tkv4, kv_cache, kvrows, 64, 4);
  if (r == CUDA_SUCCESS) r = encode_box(enc, &tkv1, kv_cache, kvrows, 64, 1);
  if (r != CUDA_SUCCESS) return set_error(MLA_ERR_CUDA, "tensor maps for the pair kernel failed (CUresult %d)", (int)r);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config((unsigned)(2 * h->n_units), st, attr);
  cudaError_t ce = cudaLaunchKernelEx(&cfg, pair::fold_pair_kernel, tq4, tq1, tkv4, tkv1, prm);
  if (ce != cudaSuccess) return set_error(MLA_ERR_CUDA, "pair kernel launch: %s", cudaGetErrorString(ce));
  return MLA_OK;
}

// Clusters of two CTAs of the pair kernel that the device runs at once.
int pair_slots_on_device(int dev, int* slots) {
  int rc = set_pair_attrs(dev);
  if (rc != MLA_OK) return rc;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config(2, 0, attr);
  int n = 0;
  cudaError_t e = cudaOccupancyMaxActiveClusters(&n, (void*)pair::fold_pair_kernel, &cfg);
  if (e != cudaSuccess) return set_error(MLA_ERR_CUDA, "cudaOccupancyMaxActiveClusters: %s", cudaGetErrorString(e));
  *slots = n;
  return MLA_OK;
}

}  // namespace mla
