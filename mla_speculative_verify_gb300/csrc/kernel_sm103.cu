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
// One thread issues a tcgen05.mma only every ~65-125 cycles (the form and the operand
// layouts), whatever the MMA's N, while an N = 16..96 MMA needs 8..48 cycles of tensor time,
// so the products of a page are issued from several threads, each into accumulators no
// other thread writes (so a unit's result is the same bit for bit on every run). O^T is
// zeroed in tensor memory at the start of the unit, so every O^T MMA accumulates.
//   bf16 cache:  three MMA warps each issue a third of the 36 S^T K-steps into a partial
//                accumulator of their own (the softmax adds the three); one S^T buffer, so
//                the next page's product starts as soon as the softmax has read this one.
//                O^T is issued by four of the softmax warps, one value block each.
//   e4m3 cache:  each S^T K-step multiplies the page by Q_hi and Q_lo at once (N = 2 nmma);
//                two MMA warps take alternate pages into two S^T buffers; O^T value blocks
//                0-1 come from an O^T warp, blocks 2-3 from the producer warp.
//
// Warp roles (one CTA per SM):
//   warp 0     TMA producer: the Q tile once (bf16 cache), then one page per stage
//              (two bf16 stages, or four e4m3 stages, in the same ring), each copy with
//              an L2 prefetch of the page that enters the ring next (bf16: those of the
//              first S copies leave once page 0 has landed); e4m3: also O^T blocks 2-3
//   warps 1-3  MMA warps (above)
//   warps 4-11 softmax: warp (quadrant qd, group grp) owns the 16 keys of TMEM lane
//              quadrant qd and 8 of every 16 columns; a 16-lane TMEM load gives each
//              thread 2 keys x 2 columns. Online softmax with a lazy per-row reference:
//              the reference moves, and O^T is rescaled in TMEM, only when a score exceeds
//              it by a few octaves (the conditional rescale of flashinfer PR #5602); then
//              the epilogue: O / l to bf16 out and LSE, or bf16 partials for the merge
//              kernel. The eight warps agree on every decision through OR-reducing named
//              barriers. For a bf16 cache P^T(t) is written with the current references
//              first, so that one barrier per tile both votes on reference moves and closes
//              P^T(t) (a move rewrites it); after it four of the warps each issue one value
//              block of O^T(t) += V^T P^T(t). (On the critical path of the two-stage bf16
//              page ring this saves a wake-up; the e4m3 softmax is already the busiest role,
//              so there other warps do it.)
//
// For an e4m3 cache the products run on kind::f8f6f4 MMAs straight from the cached
// codes: each Q row is scaled by a power of two and split into two e4m3 parts (hi and
// lo), and P into two e4m3 parts as well, so no page is ever expanded to bf16 and the
// only rounding beyond fp32 accumulation is that of the lo parts (~2^-8 relative).
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

#include <algorithm>
#include <mutex>

#include "mla_decode.h"
#include "plan_format.h"
#include "decode_common.cuh"
#include "ptx.cuh"
#include "status.h"

namespace mla {

// ------------------------------------------------------------------ tile geometry
constexpr int kRowsCap = 48;                       // packed rows per CTA (shared-memory bound)
constexpr int kTileKeys = 64;                      // keys per stage = one page
constexpr int kChunks = 9;                         // 576 = 9 x 64 columns (128-byte swizzle rows)
constexpr int kQChunkBytes = kRowsCap * 128;       // 6144
constexpr int kQBytes = kChunks * kQChunkBytes;    // 55296
// e4m3 path: per 64-column chunk, the Q_hi rows and then the Q_lo rows (<= 2 x 48 rows of
// 64 bytes, 64-byte swizzle), so that one MMA with N = 2 nmma multiplies K by both parts
constexpr int kQ8ChunkBytes = 2 * kRowsCap * 64;   // 6144
static_assert(kChunks * kQ8ChunkBytes <= kQBytes, "e4m3 Q fits the Q region");
constexpr int kKvChunkBytes = kTileKeys * 128;     // 8192 (bf16 page chunk: 64 keys x 64 columns)
constexpr int kSlotBytes = kChunks * kKvChunkBytes;  // 73728 (bf16 page)
constexpr int kKvBytes = 2 * kSlotBytes;           // page ring: two bf16 stages or four e4m3 stages
constexpr int kPtBytes = kTileKeys * 128;          // P^T tile: 64 keys x (<= 64 rows) bf16, or e4m3 hi + lo
constexpr int kOffQ = 0;
constexpr int kOffKv = kOffQ + kQBytes;
constexpr int kOffPt = kOffKv + kKvBytes;
constexpr int kOffMisc = kOffPt + 2 * kPtBytes;
constexpr int kMiscBytes = 4096;
constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-CTA shared memory");
static_assert(kOffKv % 1024 == 0 && kOffPt % 1024 == 0 && kOffMisc % 1024 == 0, "1024-byte swizzle atoms");

// Per cache dtype: a bf16 page is 128-byte rows per 64-column chunk (128-byte swizzle), an
// e4m3 page 64-byte rows (64-byte swizzle), so the same ring holds two or four pages.
template <bool kFp8>
struct Geo {
  static constexpr int kStages = kFp8 ? 4 : 2;
  static constexpr int kRowBytes = kFp8 ? 64 : 128;           // bytes of one key in one chunk
  static constexpr int kChunkBytes = kTileKeys * kRowBytes;   // 4096 / 8192
  static constexpr int kSlot = kChunks * kChunkBytes;         // 36864 / 73728
  static_assert(kStages * kSlot == kKvBytes, "ring size");
};


// Warps: producer, MMA warps, softmax. Every accumulator is written by one thread in
// program order, so a unit's result is the same bit for bit on every run.
//   bf16:  three S^T warps, each a third of the K-steps into a partial accumulator of its
//          own (the softmax adds the three); O^T is issued by four of the softmax warps,
//          one value block each (it is on the critical path of the two-stage page ring)
//   e4m3:  two S^T warps that take alternate pages (all K-steps of a page each); value
//          blocks 0 and 1 of O^T come from an O^T warp, blocks 2 and 3 from the producer
//          warp, just before it waits for the page's slot to refill it (the softmax warps
//          are the busiest role there, and twelve warps keep ~170 registers per thread)
template <bool kFp8>
struct Roles {
  static constexpr int kSWarps = kFp8 ? 2 : 3;
  static constexpr int kOWarps = kFp8 ? 1 : 0;
  static constexpr int kMmaWarps = kSWarps + kOWarps;
  static constexpr int kThreads = 32 * (1 + kMmaWarps + kSoftmaxWarps);
};
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;       // O^T block b at columns 64 b (N <= 64)
// S^T: bf16: one buffer, partial p of the three at columns 256 + 64 p (N <= 48);
//       e4m3: two buffers, buffer b at columns 256 + 128 b (Q_hi and Q_lo products, 2 N <= 96)
constexpr uint32_t kTmemS = 256;
constexpr float kRefSlack = 8.0f;    // octaves a score may exceed the row reference before it moves
// e4m3 path: a smaller slack (p <= 16) so that P can be stored times 2^4 (<= 256 < 448,
// the largest e4m3); probabilities down to 2^-10 of the reference stay in e4m3's normal
// range, smaller ones keep an absolute error below 2^-14. The 2^4 is applied by keeping
// the stored reference kPShiftFp8 octaves below the row's reference, so exp2(s - ref) is
// already P times 2^4; l carries the same factor, which cancels in O / l and in the LSE.
constexpr float kRefSlackFp8 = 4.0f;
constexpr float kPShiftFp8 = 4.0f;
struct Misc {
  uint64_t bar_q;
  uint64_t kv_full[4], kv_empty[4];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[2], pt_empty[2];  // p_full: e4m3 only (the O^T warp waits on it)
  uint64_t mma_done[8];  // MMA warps 0..2, producer 3, softmax O^T issuers 4..7
  uint32_t tmem_base;
  int abort;
  int unit[12];  // this CTA's PlanUnit
  alignas(16) float ref[64];  // read as float4
  alignas(16) float alpha[64];
  alignas(16) int lim[64];
  alignas(16) float colred[4][64];  // per TMEM lane quadrant, per packed row
  alignas(16) float oscale[64];  // per packed row: output scale / l (0 for padding rows)
  alignas(16) float colscale[64];  // e4m3 path: score scale of each row (its Q split scale folded in)
};
static_assert(offsetof(Misc, ref) % 16 == 0, "float4 reads of ref need 16-byte alignment");
static_assert(sizeof(Misc) <= kMiscBytes, "misc block too small");

// An fp32 rounded to the precision of e4m3 (4 significant bits, round to nearest even),
// still as fp32; exact for magnitudes in e4m3's normal range.
__device__ __forceinline__ float round_to_e4m3_precision(float x) {
  const uint32_t u = __float_as_uint(x);
  return __uint_as_float((u + 0x7FFFFu + ((u >> 20) & 1u)) & 0xFFF00000u);
}
// Two fp32 -> two e4m3 codes (round to nearest even, saturating), first in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}
// Two fp32 values (<= 448) -> hi and lo e4m3 pairs with hi + lo ~ the values: through f16x2
// (11 significant bits, more than hi + lo keep), hi = the e4m3 rounding, lo = the e4m3
// rounding of the f16 remainder. Each result holds the first value in its low byte.
__device__ __forceinline__ void split_e4m3x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 w = __floats2half2_rn(a, b);
  const __nv_fp8x2_storage_t h = __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&w), __NV_SATFINITE,
                                                           __NV_E4M3);
  const __half2_raw hb = __nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3);
  const __half2 r = __hsub2(w, *reinterpret_cast<const __half2*>(&hb));
  hi = (uint32_t)h;
  lo = (uint32_t)__nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&r), __NV_SATFINITE, __NV_E4M3);
}
// Byte offset of (row, column) in a 64-byte-swizzled e4m3 region with 64-byte rows.
__device__ __forceinline__ int sw64_offset(int row, int col) {
  return row * 64 + ((((col >> 4) ^ (row >> 1)) & 3) << 4) + (col & 15);
}

// O^T is zeroed in tensor memory before the first tile, so every O^T MMA accumulates and
// the MMAs of one value block may come from different threads in any order.
// bf16: O^T += V^T . P^T(t) for value block blk (MN-major V^T from page t's ring slot,
// MN-major P^T), the block's four K-steps, issued by one lane.
__device__ __forceinline__ void issue_ot_block_bf16(uint32_t tmem, uint32_t skv, uint32_t spt, int t, int nmma,
                                                    int blk) {
  using G = Geo<false>;
  const uint32_t idesc_o = ptx::idesc_bf16(128, nmma, 1, 1);
  const uint32_t pt0 = spt + (t & 1) * kPtBytes;
  // value columns [128 blk, 128 blk + 128) = chunks 2 blk, 2 blk + 1 of the page
  const uint32_t v0 = skv + (t % G::kStages) * G::kSlot + 2 * blk * G::kChunkBytes;
  const uint32_t d = tmem + kTmemO + 64 * blk;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint64_t ad = ptx::smem_desc(v0 + 2048 * k, G::kChunkBytes, 1024, ptx::kSwizzle128B);
    uint64_t bd = ptx::smem_desc(pt0 + 2048 * k, 8192, 1024, ptx::kSwizzle128B);
    ptx::mma_bf16_ss(d, ad, bd, idesc_o, 1u);
  }
}
// e4m3: one MMA of O^T += V^T . P^T(t): value block blk, K-step k (32 keys), P^T part
// (0 = hi, 1 = lo; each 64 keys x 64 bytes).
__device__ __forceinline__ void issue_ot_mma_e4m3(uint32_t tmem, uint32_t skv, uint32_t spt, int t, int nmma, int blk,
                                                  int k, int part) {
  using G = Geo<true>;
  const uint32_t idesc_o = ptx::idesc_e4m3(128, nmma, 1, 1);
  const uint32_t pt0 = spt + (t & 1) * kPtBytes;
  const uint32_t v0 = skv + (t % G::kStages) * G::kSlot + 2 * blk * G::kChunkBytes;
  const uint64_t ad = ptx::smem_desc(v0 + 2048 * k, G::kChunkBytes, 512, ptx::kSwizzle64B);
  const uint64_t bd = ptx::smem_desc(pt0 + part * (kTileKeys * 64) + 2048 * k, 4096, 512, ptx::kSwizzle64B);
  ptx::mma_e4m3_ss(tmem + kTmemO + 64 * blk, ad, bd, idesc_o, 1u);
}

struct SoftmaxArgs {
  Misc* ms;
  uint8_t* sQ;
  uint8_t* sKv;
  uint8_t* sPt;
  uint32_t tmem, skv, spt;
  int qd, grp, lane, sidx, nmma, b, nrows, qrow0, kv_begin, kv_end, ntiles, part_row0, ctx, qlen, tok0;
  volatile int* abort;
};

// Softmax warps for a tile of 16 NCH packed rows. Warp (qd, grp) owns the 16 key rows of
// TMEM lane quadrant qd (the M = 64 accumulator uses 16 lanes per quadrant) and, of every
// 16 columns, the 8 columns 8 grp .. 8 grp + 7, which one 16-lane TMEM load (16x256b)
// spreads over all 32 threads: thread t holds keys kr0 = 16 qd + t / 4 and kr0 + 8 at columns
// 16 c + cp and 16 c + cp + 1, cp = 8 grp + 2 (t % 4). Element x[4 c + j] is key kr0 + 8 (j / 2),
// column 16 c + cp + j % 2 (c < NCH, j < 4).
// Returns whether this thread issued O^T MMAs (lane 0 of softmax warps 0..3).
template <int NCH, bool kFp8>
__device__ __forceinline__ bool softmax_role(const SoftmaxArgs& a, const Params& p) {
  constexpr int NC = 4 * NCH;
  using G = Geo<kFp8>;
  constexpr float kPShift = kFp8 ? kPShiftFp8 : 0.f;
  constexpr float kMoveAbove = (kFp8 ? kRefSlackFp8 : kRefSlack) + kPShift;  // score - stored ref
  Misc* ms = a.ms;
  const int lane = a.lane, qd = a.qd, grp = a.grp, sidx = a.sidx;
  const int kr0 = qd * 16 + (lane >> 2);  // this thread's first key row in the 64-key tile (second: kr0 + 8)
  const int cp = 8 * grp + 2 * (lane & 3);  // first of this thread's 2 columns in each 16-column chunk
  const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
  const int w8 = sidx >> 5;              // softmax warp 0..7; warps 0..3 issue O^T block w8
  bool issued_ot = false;
  volatile int* abort = a.abort;
  if (sidx == 0 && (p.seq_lens[a.b] != a.ctx || p.q_lens[a.b] != a.qlen)) {
    // the device lengths differ from those the plan was built for: stop the unit
    report(p.status, MLA_DEVICE_PLAN_MISMATCH);
    *a.abort = 1;
  }
  {
    // O^T starts at zero (every O^T MMA accumulates): this warp clears the lanes of its
    // quadrant in columns [128 grp, 128 grp + 128) of the O^T region
    float z[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) ptx::tmem_st16(a.tmem + kTmemO + lane_off + 128 * grp + 16 * c, z);
    ptx::tmem_st_wait();
    ptx::tc_fence_before();
  }
  if (sidx < 64) {
    int lim = 0;
    if (sidx < a.nrows) {
      const int i = (a.qrow0 + sidx) / p.H - a.tok0;  // verify token of this packed row
      lim = a.ctx - a.qlen + i + 1;
    }
    ms->lim[sidx] = lim;
    ms->ref[sidx] = -INFINITY;
  }
  if constexpr (kFp8) {
    // Q tile -> e4m3 hi rows [0, nmma) and lo rows [nmma, 2 nmma) (64-byte swizzle,
    // K-major) for the e4m3 S^T MMAs, whose N = 2 nmma columns hold K Q_hi^T and then
    // K Q_lo^T. Row r is scaled by 2^e_r so that its largest |q| lands in [128, 256);
    // hi = q 2^e_r rounded to e4m3, lo = the remainder in e4m3: hi + lo reproduces the
    // bf16 row to ~2^-17 of its largest entry. 2^-e_r goes into the row's score scale.
    // This warp's rows r = w8 + 8 k: all of their loads go out first (one round trip).
    const float base = p.score_scale_log2;
    constexpr int kRowsPerWarp = 16 * NCH / kSoftmaxWarps;
    uint32_t raw[kRowsPerWarp][9];
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      const int grow = a.qrow0 + w8 + kSoftmaxWarps * k;
      const uint32_t* src = reinterpret_cast<const uint32_t*>(p.q + (size_t)grow * kDqk + 18 * lane);
#pragma unroll
      for (int j = 0; j < 9; ++j) raw[k][j] = grow < p.q_rows ? src[j] : 0u;
    }
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      const int r = w8 + kSoftmaxWarps * k;
      float v[18];
#pragma unroll
      for (int j = 0; j < 9; ++j) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw[k][j]));
        v[2 * j] = f.x;
        v[2 * j + 1] = f.y;
      }
      float mx = 0.f;
#pragma unroll
      for (int j = 0; j < 18; ++j) mx = fmaxf(mx, fabsf(v[j]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      int e = 0;
      if (mx > 0.f && mx < INFINITY) e = max(-100, min(100, 7 - ((int)((__float_as_uint(mx) >> 23) & 0xFF) - 127)));
      const float sc = __uint_as_float((uint32_t)(e + 127) << 23);  // 2^e
#pragma unroll
      for (int j = 0; j < 18; j += 2) {
        const float w0 = v[j] * sc, w1 = v[j + 1] * sc;
        const float h0 = round_to_e4m3_precision(w0), h1 = round_to_e4m3_precision(w1);
        const int col = 18 * lane + j;  // even: the pair stays in one 16-byte piece
        uint8_t* chunk = a.sQ + (col >> 6) * kQ8ChunkBytes;
        *reinterpret_cast<uint16_t*>(chunk + sw64_offset(r, col & 63)) = (uint16_t)e4m3x2(h0, h1);
        *reinterpret_cast<uint16_t*>(chunk + sw64_offset(16 * NCH + r, col & 63)) = (uint16_t)e4m3x2(w0 - h0, w1 - h1);
      }
      if (lane == 0) ms->colscale[r] = base * __uint_as_float((uint32_t)(127 - e) << 23);
    }
    ptx::fence_async_smem();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&ms->bar_q);
  }
  // `stop` only ever changes through a barrier's reduction, so it is the same in all
  // softmax warps; `fail` is this warp's own: one of its bounded waits gave up.
  bool stop = softmax_any(*abort != 0);
  bool fail = false;
  int lim_min = a.kv_end;
  for (int n = 0; n < a.nrows; ++n) lim_min = min(lim_min, ms->lim[n]);
  constexpr int NP = 2 * NCH;  // this thread's columns (rows of the tile): 16 c + cp + k, index 2 c + k
  float l_acc[NC];
  // e4m3: this thread's copies of its columns' references (they change only when a row
  // moves), so the shared-memory pipe, which the e4m3 path fills, serves fewer loads; the
  // bf16 path reads them from shared memory (its registers are spoken for)
  float rref[kFp8 ? NP : 1];
#pragma unroll
  for (int i = 0; i < NC; ++i) l_acc[i] = 0.f;
#pragma unroll
  for (int i = 0; i < (kFp8 ? NP : 1); ++i) rref[i] = -INFINITY;
  // e4m3: the columns' score scales (fixed for the unit; the barrier above published them)
  float csr[kFp8 ? NP : 1];
#pragma unroll
  for (int i = 0; i < (kFp8 ? NP : 1); ++i) csr[i] = kFp8 ? ms->colscale[16 * (i / 2) + cp + (i % 2)] : 0.f;
  // the references of chunk c's two columns, r[j] for element 4 c + j
  auto ref4 = [&](int c, float* r) {
    if constexpr (kFp8) {
      r[0] = r[2] = rref[2 * c];
      r[1] = r[3] = rref[2 * c + 1];
    } else {
      const float2 rr = *reinterpret_cast<const float2*>(&ms->ref[16 * c + cp]);
      r[0] = r[2] = rr.x;
      r[1] = r[3] = rr.y;
    }
  };
  const float scale = p.score_scale_log2;
  for (int t = 0; !stop && t < a.ntiles; ++t) {
    const int sb = t & 1;
    float x[NC];
    bool need = false;
    bool unmasked = false;  // this tile: every key visible to every row
    // S^T(t): e4m3 buffer t % 2; bf16 the one buffer (its phase flips every tile)
    const int s_buf = kFp8 ? sb : 0;
    if (!fail) fail = !warp_wait(&ms->s_full[s_buf], kFp8 ? ((t >> 1) & 1) : (t & 1), abort, p);
    if (!fail) {
      ptx::tc_fence_after();
      // S^T: e4m3: the sum of the Q_hi and Q_lo column blocks of buffer t % 2; bf16: the
      // sum of the three partials. All loads are issued before the one wait
      const uint32_t sbase = a.tmem + kTmemS + (kFp8 ? 128 * sb : 0) + lane_off + 8 * grp;
      float s1[NC];
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        ptx::tmem_ld_16x256b(sbase + 16 * c, &x[4 * c]);
        ptx::tmem_ld_16x256b(sbase + (kFp8 ? 16 * NCH : 64) + 16 * c, &s1[4 * c]);
      }
      if constexpr (kFp8) {
        ptx::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < NC; ++i) x[i] += s1[i];
      } else {
        float s2[NC];
#pragma unroll
        for (int c = 0; c < NCH; ++c) ptx::tmem_ld_16x256b(sbase + 128 + 16 * c, &s2[4 * c]);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < NC; ++i) x[i] = (x[i] + s1[i]) + s2[i];
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&ms->s_empty[s_buf]);
      const int key0 = a.kv_begin + t * kTileKeys + kr0;  // and key0 + 8
      const int tile_last = a.kv_begin + t * kTileKeys + kTileKeys - 1;
      unmasked = tile_last < a.kv_end && tile_last < lim_min;  // tile-uniform fast path
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const int n0 = 16 * c + cp;
        float rrv[4];
        ref4(c, rrv);
        float csv[4] = {scale, scale, scale, scale};
        if constexpr (kFp8) {
          csv[0] = csv[2] = csr[2 * c];
          csv[1] = csv[3] = csr[2 * c + 1];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float v = x[4 * c + j] * csv[j];
          const int key = key0 + 8 * (j >> 1);
          if (!unmasked) v = (key < a.kv_end && key < ms->lim[n0 + (j & 1)]) ? v : -INFINITY;
          x[4 * c + j] = v;
          need |= v > rrv[j] + kMoveAbove;
        }
      }
    }
    // Moving the references (rare once a row has seen its largest scores): column maxima
    // over this tile's keys (the quadrant's 16 keys: 2 per thread, 8 threads per column),
    // each row's reference up to its maximum, l and O^T (tiles < t, once PV(t-1) is done)
    // rescaled by alpha.
    auto move_refs = [&]() {
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        const int c = i >> 1, k = i & 1;
        float m = fmaxf(x[4 * c + k], x[4 * c + k + 2]);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((lane >> 2) == 0) ms->colred[qd][16 * c + cp + k] = m;
      }
      softmax_sync();
      if (sidx < 16 * NCH) {
        const float cm = fmaxf(fmaxf(ms->colred[0][sidx], ms->colred[1][sidx]), fmaxf(ms->colred[2][sidx], ms->colred[3][sidx]));
        const float old = ms->ref[sidx];
        const float nw = fmaxf(old, cm - kPShift);
        ms->alpha[sidx] = (nw == old) ? 1.f : ex2(old - nw);
        ms->ref[sidx] = nw;
      }
      softmax_sync();
#pragma unroll
      for (int i = 0; i < NC; ++i) l_acc[i] *= ms->alpha[16 * (i / 4) + cp + (i & 1)];
      if constexpr (kFp8) {
#pragma unroll
        for (int i = 0; i < NP; ++i) rref[i] = ms->ref[16 * (i / 2) + cp + (i % 2)];
      }
      if (t >= 1) {
        // this warp: value blocks 2 grp and 2 grp + 1 of its lane quadrant
        fail = !warp_wait(&ms->pt_empty[(t - 1) & 1], ((t - 1) >> 1) & 1, abort, p);
        if (!fail) {
          ptx::tc_fence_after();
#pragma unroll 1
          for (int blk = 2 * grp; blk < 2 * grp + 2; ++blk) {
            const uint32_t ta = a.tmem + kTmemO + 64 * blk + lane_off;
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
              float o[16];
              ptx::tmem_ld16(ta + 16 * c, o);
              ptx::tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 16; j += 4) {
                const float4 al = *reinterpret_cast<const float4*>(&ms->alpha[16 * c + j]);
                o[j] *= al.x; o[j + 1] *= al.y; o[j + 2] *= al.z; o[j + 3] *= al.w;
              }
              ptx::tmem_st16(ta + 16 * c, o);
            }
          }
          ptx::tmem_st_wait();
        }
      }
    };
    // probabilities relative to the current references (pv, kept until l takes them),
    // packed to bf16, or for the e4m3 path times 2^4 and split into hi + lo e4m3 parts
    float pv[NC];
    uint32_t pk[NC / 2];           // bf16: pk[2 c + k] = the 2 columns of key kr0 + 8 k in chunk c
    uint32_t ph[NC / 2], pl[NC / 2];  // e4m3: the same pairs as hi and lo bytes (low 16 bits)
    auto make_p = [&]() {
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        float rrv[4];
        ref4(c, rrv);
        if (unmasked) {  // no masked score (a reference may still be -inf: then a move follows)
#pragma unroll
          for (int j = 0; j < 4; ++j) pv[4 * c + j] = ex2(x[4 * c + j] - rrv[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float v = x[4 * c + j];
            pv[4 * c + j] = v == -INFINITY ? 0.f : ex2(v - rrv[j]);
          }
        }
        if constexpr (kFp8) {
          split_e4m3x2(pv[4 * c], pv[4 * c + 1], ph[2 * c], pl[2 * c]);
          split_e4m3x2(pv[4 * c + 2], pv[4 * c + 3], ph[2 * c + 1], pl[2 * c + 1]);
        } else {
          pk[2 * c] = pack_bf16(pv[4 * c], pv[4 * c + 1]);
          pk[2 * c + 1] = pack_bf16(pv[4 * c + 2], pv[4 * c + 3]);
        }
      }
    };
    auto store_p = [&]() {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int kr = kr0 + 8 * k;
        if constexpr (kFp8) {
          // e4m3 P^T hi and lo, MN-major with 64-byte rows (64-byte swizzle): key kr's row
          uint8_t* line_hi = a.sPt + sb * kPtBytes + kr * 64;
          uint8_t* line_lo = line_hi + kTileKeys * 64;
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            const int off = (((c ^ (kr >> 1)) & 3) << 4) + cp;
            *reinterpret_cast<uint16_t*>(line_hi + off) = (uint16_t)ph[2 * c + k];
            *reinterpret_cast<uint16_t*>(line_lo + off) = (uint16_t)pl[2 * c + k];
          }
        } else {
          uint8_t* line = a.sPt + sb * kPtBytes + kr * 128;
#pragma unroll
          for (int c = 0; c < NCH; ++c)
            *reinterpret_cast<uint32_t*>(line + ((((2 * c + grp) ^ (kr & 7)) & 7) << 4) + 4 * (lane & 3)) = pk[2 * c + k];
        }
        if (a.kv_begin + t * kTileKeys + kr >= a.kv_end) {
          // a cache slot past the key range: zero its value columns so P = 0 meets V = 0 (the
          // 8 threads holding key kr take one of its 8 value chunks each: 4 grp + t % 4)
          uint8_t* row = a.sKv + (t % G::kStages) * G::kSlot + kr * G::kRowBytes + (4 * grp + (lane & 3)) * G::kChunkBytes;
#pragma unroll
          for (int j = 0; j < G::kRowBytes / 16; ++j) *reinterpret_cast<uint4*>(row + 16 * j) = make_uint4(0, 0, 0, 0);
        }
      }
      ptx::fence_async_smem();
      ptx::tc_fence_before();
    };
    if constexpr (kFp8) {
      // e4m3: the vote comes first, then P^T; the O^T warp issues O^T(t) once all softmax
      // warps have arrived (a warp that gave up a wait leaves the loop with the others at
      // the next tile's vote)
      if (softmax_any(need || fail)) {
        if (softmax_any(fail || *abort != 0)) {
          stop = true;
          break;
        }
        move_refs();
      }
      if (!fail) {
        make_p();
        if (t >= 2) fail = !warp_wait(&ms->pt_empty[sb], ((t - 2) >> 1) & 1, abort, p);
      }
      if (!fail) {
#pragma unroll
        for (int i = 0; i < NC; ++i) l_acc[i] += pv[i];
        store_p();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&ms->p_full[sb]);
      }
      continue;
    }
    // bf16: P^T(t) is written with the current references before the vote, so that in the
    // usual tile (no reference moves) one barrier both votes and closes P^T(t); if a row
    // must move, the references move and P^T(t) is written again. The barriers also end the
    // loop in all warps together if one of them gave up a wait. Then warps 0..3 each issue
    // one value block of O^T(t) and release the page slot and the P^T buffer.
    if (!fail) {
      make_p();
      if (t >= 2) fail = !warp_wait(&ms->pt_empty[sb], ((t - 2) >> 1) & 1, abort, p);
    }
    if (!fail) store_p();
    if (softmax_any(need || fail || *abort != 0)) {
      if (softmax_any(fail || *abort != 0)) {
        stop = true;
        break;
      }
      move_refs();
      if (!fail) {
        make_p();
        store_p();
      }
      if (softmax_any(fail || *abort != 0)) {
        stop = true;
        break;
      }
    }
#pragma unroll
    for (int i = 0; i < NC; ++i) l_acc[i] += pv[i];
    if (w8 < 4) {
      ptx::tc_fence_after();
      if (lane == 0) {
        issue_ot_block_bf16(a.tmem, a.skv, a.spt, t, a.nmma, w8);
        ptx::mma_commit(&ms->kv_empty[t % G::kStages]);
        ptx::mma_commit(&ms->pt_empty[sb]);
        issued_ot = true;
      }
      __syncwarp();
    }
  }
  // ------------------------------------------------------------ epilogue
  // Row sums, LSE and the per-row output scale first: they need only l, so they overlap
  // the last tile's O^T MMAs. The wait for those MMAs and the abort vote come after.
  if (!stop) {
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const int c = i >> 1, k = i & 1;
      float s = l_acc[4 * c + k] + l_acc[4 * c + k + 2];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if ((lane >> 2) == 0) ms->colred[qd][16 * c + cp + k] = s;
    }
    softmax_sync();
    if (sidx < 64) {
      float L = 0.f;
      if (sidx < a.nrows) {
        L = ms->colred[0][sidx] + ms->colred[1][sidx] + ms->colred[2][sidx] + ms->colred[3][sidx];
        const float lse_v = L > 0.f ? (ms->ref[sidx] + lg2(L)) * 0.69314718055994531f : -INFINITY;
        if (a.part_row0 < 0) {
          if (p.lse) p.lse[a.qrow0 + sidx] = lse_v;
        } else {
          p.part_lse[a.part_row0 + sidx] = lse_v;
        }
      }
      ms->oscale[sidx] = L > 0.f ? p.out_scale / L : 0.f;  // one division per row
    }
    if (!fail) fail = !warp_wait(&ms->pt_empty[(a.ntiles - 1) & 1], ((a.ntiles - 1) >> 1) & 1, abort, p);
    // this barrier also publishes oscale to all softmax warps
    stop = softmax_any(fail || *abort != 0);
  }
  if (stop) return issued_ot;
  ptx::tc_fence_after();
  // O^T(dv, row) / l(row): this thread holds dv = 128 blk + 32 qd + lane of value blocks
  // 2 grp, 2 grp + 1; a warp's stores of one row cover 32 consecutive dv (bf16 out, or
  // the bf16 split partial)
  __nv_bfloat16* dst = a.part_row0 < 0 ? p.out + (size_t)a.qrow0 * kDv : p.part_o + (size_t)a.part_row0 * kDv;
  const int dv_in_blk = qd * 32 + lane;
#pragma unroll 1
  for (int blk = 2 * grp; blk < 2 * grp + 2; ++blk) {
    const int dv = blk * 128 + dv_in_blk;
    float o[NCH][16];
#pragma unroll
    for (int c = 0; c < NCH; ++c) ptx::tmem_ld16(a.tmem + kTmemO + 64 * blk + lane_off + 16 * c, o[c]);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
#pragma unroll
      for (int j = 0; j < 16; j += 4) {
        const float4 sc = *reinterpret_cast<const float4*>(&ms->oscale[16 * c + j]);
        const float v4[4] = {o[c][j] * sc.x, o[c][j + 1] * sc.y, o[c][j + 2] * sc.z, o[c][j + 3] * sc.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int n = 16 * c + j + u;
          if (n < a.nrows) dst[(size_t)n * kDv + dv] = __float2bfloat16_rn(v4[u]);
        }
      }
    }
  }
  return issued_ot;
}

template <bool kFp8>
__global__ void __launch_bounds__(Roles<kFp8>::kThreads, 1)
    fold_decode_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_kv, Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base (the 128-byte swizzle atoms), kept in the shared window
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
  Misc* ms = (Misc*)(smem + kOffMisc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort = &ms->abort;

  ptx::pdl_launch_dependents();

  // Prologue. Warp 0 reads this CTA's unit record (one round trip), issues the Q copy and
  // reads the first page ids before the CTA-wide barrier, so that the first page copies
  // leave as early as possible. The device copies of seq_lens / q_lens are checked
  // against the plan by the softmax warps afterwards.
  constexpr int kUnitWords = (int)(sizeof(PlanUnit) / 4);
  using G = Geo<kFp8>;
  constexpr int S = G::kStages;
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sKv = smem + kOffKv;
  uint8_t* sPt = smem + kOffPt;
  int pid_cur = 0, pid_next = 0;  // producer: page ids of 32 consecutive pages, and of the next 32
  if (warp == 0) {
    if (lane == 0) {
      ms->abort = 0;
      ptx::mbar_init(&ms->bar_q, kFp8 ? kSoftmaxWarps : 1);  // e4m3: the softmax warps convert Q themselves
    constexpr int kOtIssuers = kFp8 ? 2 : 4;  // e4m3: the O^T warp and the producer; bf16: four softmax warps
    for (int i = 0; i < 4; ++i) {
      ptx::mbar_init(&ms->kv_full[i], 1);
      ptx::mbar_init(&ms->kv_empty[i], kOtIssuers);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&ms->s_full[i], kFp8 ? 1 : Roles<kFp8>::kSWarps);  // the S^T warp(s) of a tile
      ptx::mbar_init(&ms->s_empty[i], kSoftmaxWarps);
      ptx::mbar_init(&ms->pt_empty[i], kOtIssuers);
      ptx::mbar_init(&ms->p_full[i], kSoftmaxWarps);
    }
    for (int i = 0; i < 8; ++i) ptx::mbar_init(&ms->mma_done[i], 1);
    ptx::fence_mbar_init();
    }
    int uw = 0;
    if (lane < kUnitWords) uw = reinterpret_cast<const int32_t*>(p.units + blockIdx.x)[lane];
    if (lane < kUnitWords) ms->unit[lane] = uw;
    const int ub = __shfl_sync(0xffffffffu, uw, 0), uq0 = __shfl_sync(0xffffffffu, uw, 1);
    const int ukb = __shfl_sync(0xffffffffu, uw, 3), uke = __shfl_sync(0xffffffffu, uw, 4);
    const int unt = (uke - ukb + kTileKeys - 1) / kTileKeys;
    if (lane == 0) {
      ptx::prefetch_tmap(&tmap_kv);
      if (!kFp8) {
        ptx::prefetch_tmap(&tmap_q);
        ptx::mbar_arrive_expect_tx(&ms->bar_q, kQBytes);
        ptx::tma_load_3d(sQ, &tmap_q, &ms->bar_q, 0, uq0, 0);
      }
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

  const int b = ms->unit[0], qrow0 = ms->unit[1], nrows = ms->unit[2];
  const int kv_begin = ms->unit[3], kv_end = ms->unit[4], part_row0 = ms->unit[5];
  const int ctx = ms->unit[8], qlen = ms->unit[9], tok0 = ms->unit[10];
  const int ntiles = (kv_end - kv_begin + kTileKeys - 1) / kTileKeys;
  const int nmma = (nrows + 15) & ~15;   // MMA N (rows rounded up to 16)
  const int nch = nmma / 16;             // 16-column chunks of S^T / O^T
  const uint32_t tmem = ms->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int issued = 0;
    bool ot_issued = false;  // e4m3: lane 0 issued O^T MMAs
    const bool q_issued = !kFp8;
    {
      const int32_t* pt_row = p.page_table + (size_t)b * p.pt_stride + kv_begin / kPage;
      // page ids 32 at a time (one per lane), the next batch read one batch ahead. An id
      // outside the cache is reported and replaced by page 0. With the copy of page t the
      // producer also asks L2 for page t + S, the next one to enter the ring, so that its
      // copy (issued once O^T(t) frees the slot) is served by L2; for a bf16 cache the
      // first S of these wait until page 0 has landed. (Prefetching four pages beyond the
      // ring measured slower: those requests queue in front of the ring's own.)
      auto checked = [&](int pid, int t) {
        if (t < ntiles && (pid < 0 || pid >= p.num_pages)) {
          report(p.status, MLA_DEVICE_BAD_PAGE);
          pid = 0;
        }
        return pid;
      };
      auto load_ids = [&](int t0) { return checked(t0 + lane < ntiles ? pt_row[t0 + lane] : 0, t0 + lane); };
      // e4m3: O^T(u) += V^T . P^T(u) for value blocks 2 and 3, once P^T(u) is written (the
      // whole warp waits, lane 0 issues)
      auto producer_ot = [&](int u) -> int {
        if (!warp_wait(&ms->p_full[u & 1], (u >> 1) & 1, abort, p)) return 0;
        ptx::tc_fence_after();
        if (lane == 0) {
          const uint32_t skv = ptx::smem_addr(sKv), spt = ptx::smem_addr(sPt);
#pragma unroll
          for (int blk = 2; blk < 4; ++blk)
#pragma unroll
            for (int k = 0; k < 2; ++k)
#pragma unroll
              for (int part = 0; part < 2; ++part) issue_ot_mma_e4m3(tmem, skv, spt, u, nmma, blk, k, part);
          ptx::mma_commit(&ms->kv_empty[u % S]);
          ptx::mma_commit(&ms->pt_empty[u & 1]);
          ot_issued = true;
        }
        __syncwarp();
        return 1;
      };
      // a page that only this row tile reads may leave L2 first once it is in shared
      // memory, which keeps the plan, the page table and the split partials there
      const bool read_once = (ms->unit[11] & kUnitKvReadOnce) != 0;
      const uint64_t pol = ptx::policy_evict_first();
      pid_cur = checked(pid_cur, lane);
      pid_next = checked(pid_next, 32 + lane);
      for (int t0 = 0; t0 < ntiles && !*abort; t0 += 32) {
        const int cnt = min(32, ntiles - t0);
        for (int i = 0; i < cnt; ++i) {
          const int page = __shfl_sync(0xffffffffu, pid_cur, i);
          const int tp = i + S;  // the page after the ring (index relative to t0)
          const int page_pf = __shfl_sync(0xffffffffu, tp < 32 ? pid_cur : pid_next, tp & 31);
          const int t = t0 + i, slot = t % S;
          // e4m3: this warp also issues value blocks 2 and 3 of O^T(t - S), the page whose
          // slot the copy of page t reuses (blocks 0 and 1 come from the O^T warp). The
          // waits are the whole warp's; lane 0 issues.
          bool ok = true;
          if (kFp8 && t >= S) ok = producer_ot(t - S) != 0;
          if (ok && t >= S) ok = warp_wait(&ms->kv_empty[slot], ((t - S) / S) & 1, abort, p);
          if (!ok) break;
          if (lane == 0 && !(blockIdx.x == 0 && t == p.skip_copy)) {
            ptx::mbar_arrive_expect_tx(&ms->kv_full[slot], G::kSlot);
            if (read_once)
              ptx::tma_load_3d_hint(sKv + slot * G::kSlot, &tmap_kv, &ms->kv_full[slot], 0, page * kPage, 0, pol);
            else
              ptx::tma_load_3d(sKv + slot * G::kSlot, &tmap_kv, &ms->kv_full[slot], 0, page * kPage, 0);
            if ((kFp8 || t >= S) && t0 + tp < ntiles) ptx::tma_prefetch_l2_3d(&tmap_kv, 0, page_pf * kPage, 0);
          }
          __syncwarp();
          issued = t + 1;
          if (!kFp8 && t == S - 1) {
            // bf16: the prefetches that go with the first S copies leave once page 0 has
            // landed, so that the first pages do not share HBM with them
            int pf[S];
#pragma unroll
            for (int k = 0; k < S; ++k) pf[k] = __shfl_sync(0xffffffffu, pid_cur, S + k);
            if (warp_wait(&ms->kv_full[0], 0, abort, p) && lane == 0) {
#pragma unroll
              for (int k = 0; k < S; ++k)
                if (S + k < ntiles) ptx::tma_prefetch_l2_3d(&tmap_kv, 0, pf[k] * kPage, 0);
            }
            __syncwarp();
          }
        }
        pid_cur = pid_next;
        pid_next = (t0 + 64 < ntiles) ? load_ids(t0 + 64) : 0;
      }
      // e4m3: blocks 2 and 3 of O^T for the last S pages (no copy follows them)
      if (kFp8 && issued == ntiles) {
        int ok = 1;
        for (int u = max(0, ntiles - S); ok && u < ntiles; ++u) ok = producer_ot(u);
      }
    }
    // Drain: every issued copy must land before the CTA may exit (at most the last S
    // pages can still be in flight; earlier ones were consumed by the MMAs).
    if (lane == 0) {
      for (int t = max(0, issued - S); t < issued; ++t) {
        if (blockIdx.x == 0 && t == p.skip_copy) continue;  // never issued (timeout test)
        long long t0c = clock64();
        while (!ptx::mbar_try_wait(&ms->kv_full[t % S], (t / S) & 1) && clock64() - t0c < p.wait_budget) {
        }
      }
      if (q_issued) {
        long long t0c = clock64();
        while (!ptx::mbar_try_wait(&ms->bar_q, 0) && clock64() - t0c < p.wait_budget) {
        }
      }
      // and the O^T MMAs this lane issued must retire before TMEM is released
      if (ot_issued) drain_mmas(&ms->mma_done[3], p.wait_budget);
    }
    __syncwarp();
  } else if (warp <= Roles<kFp8>::kMmaWarps) {
    // ------------------------------------------------------------ MMA issue
    // One thread issues a tcgen05.mma only every ~100 cycles, so several warps issue the
    // products of a page, each into accumulators that no other thread writes.
    const int mi = warp - 1;
    const uint32_t sq = ptx::smem_addr(sQ), skv = ptx::smem_addr(sKv), spt = ptx::smem_addr(sPt);
    bool ok = !*abort && warp_wait(&ms->bar_q, 0, abort, p);
    bool issued = false;
    if (mi < Roles<kFp8>::kSWarps) {
      const uint32_t idesc_s = kFp8 ? ptx::idesc_e4m3(64, 2 * nmma, 0, 0) : ptx::idesc_bf16(64, nmma, 0, 0);
      for (int t = 0; ok && t < ntiles; ++t) {
        // e4m3: warp mi takes the pages with t % 2 == mi; bf16: every page
        if (kFp8 && (t & 1) != mi) continue;
        ok = warp_wait(&ms->kv_full[t % S], (t / S) & 1, abort, p);
        // the softmax must have read the previous S^T out of this buffer (e4m3: of t - 2 in
        // buffer t % 2; bf16: of t - 1 in the one buffer)
        if constexpr (kFp8) {
          if (ok && t >= 2) ok = warp_wait(&ms->s_empty[t & 1], ((t - 2) >> 1) & 1, abort, p);
        } else {
          if (ok && t >= 1) ok = warp_wait(&ms->s_empty[0], (t - 1) & 1, abort, p);
        }
        if (!ok) break;
        ptx::tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = skv + (t % S) * G::kSlot;
          if constexpr (kFp8) {
            // S^T(t) = K . [Q_hi | Q_lo]^T into buffer t % 2: all 18 K-steps (32 columns each)
            const uint32_t d = tmem + kTmemS + 128 * (t & 1);
#pragma unroll
            for (int ks = 0; ks < 18; ++ks) {
              const int c = ks >> 1, kk = ks & 1;
              const uint64_t ad = ptx::smem_desc(a0 + c * G::kChunkBytes + 32 * kk, 16, 512, ptx::kSwizzle64B);
              const uint64_t bd = ptx::smem_desc(sq + c * kQ8ChunkBytes + 32 * kk, 16, 512, ptx::kSwizzle64B);
              ptx::mma_e4m3_ss(d, ad, bd, idesc_s, ks != 0 ? 1u : 0u);
            }
            ptx::mma_commit(&ms->s_full[t & 1]);
          } else {
            // partial mi of S^T(t) = K . Q^T: K-steps [12 mi, 12 mi + 12) of the 36 (16 columns each)
            const uint32_t d = tmem + kTmemS + 64 * mi;
#pragma unroll
            for (int i = 0; i < 12; ++i) {
              const int ks = 12 * mi + i, c = ks >> 2, k = ks & 3;
              const uint64_t ad = ptx::smem_desc(a0 + c * G::kChunkBytes + 32 * k, 16, 1024, ptx::kSwizzle128B);
              const uint64_t bd = ptx::smem_desc(sq + c * kQChunkBytes + 32 * k, 16, 1024, ptx::kSwizzle128B);
              ptx::mma_bf16_ss(d, ad, bd, idesc_s, i != 0 ? 1u : 0u);
            }
            ptx::mma_commit(&ms->s_full[0]);
          }
        }
        __syncwarp();
        issued = true;
      }
    } else if constexpr (kFp8) {
      // e4m3: O^T(t) += V^T . P^T(t) for value blocks 0 and 1 (the producer issues 2 and 3),
      // once the softmax warps have written P^T(t)
      const int ow = mi - Roles<kFp8>::kSWarps;  // 0
      for (int t = 0; ok && t < ntiles; ++t) {
        ok = warp_wait(&ms->p_full[t & 1], (t >> 1) & 1, abort, p);
        if (!ok) break;
        ptx::tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int blk = 2 * ow; blk < 2 * ow + 2; ++blk)
#pragma unroll
            for (int k = 0; k < 2; ++k)
#pragma unroll
              for (int part = 0; part < 2; ++part) issue_ot_mma_e4m3(tmem, skv, spt, t, nmma, blk, k, part);
          ptx::mma_commit(&ms->kv_empty[t % S]);
          ptx::mma_commit(&ms->pt_empty[t & 1]);
        }
        __syncwarp();
        issued = true;
      }
    }
    // every MMA this warp issued must retire before TMEM is released
    if (issued) {
      if (lane == 0) drain_mmas(&ms->mma_done[mi], p.wait_budget);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    constexpr int kMma = Roles<kFp8>::kMmaWarps;
    const SoftmaxArgs a{ms, sQ, sKv, sPt, tmem, ptx::smem_addr(sKv), ptx::smem_addr(sPt), warp & 3,
                        (warp - 1 - kMma) >> 2, lane, tid - 32 * (kMma + 1), nmma, b, nrows, qrow0,
                        kv_begin, kv_end, ntiles, part_row0, ctx, qlen, tok0, abort};
    bool issued_ot;
    if (nch == 1)
      issued_ot = softmax_role<1, kFp8>(a, p);
    else if (nch == 2)
      issued_ot = softmax_role<2, kFp8>(a, p);
    else
      issued_ot = softmax_role<3, kFp8>(a, p);
    // the O^T MMAs this lane issued must retire before TMEM is released
    if (issued_ot) drain_mmas(&ms->mma_done[4 + (warp - 1 - kMma)], p.wait_budget);
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ LSE merge
// One CTA per (packed row, slice of the 512 value columns: SL = 4 slices of 128 columns, or
// 8 of 64 when the merge has few rows, so that more SMs share its loads): its W warps (4, 8
// or 16, enough for all splits at kMergeBatch loads per lane) share the splits of the row;
// fewer warps per CTA let more CTAs share an SM. L = ln sum_s exp(L_s),
// O = sum_s exp(L_s - L) O_s.
constexpr int kMergeThreads = 512;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kMergeBatch = 10;  // partial-O loads in flight per lane (16 warps x 10 = 160 splits per round trip)
constexpr int kMergeMaxSplits = 2048;
constexpr long long kMergeWideSlicesMaxCtas = 200;  // 8 slices per row up to this many merge CTAs

// Four bf16 partial-O values (8 bytes, streamed: read once) as fp32.
__device__ __forceinline__ float4 load_part4(const __nv_bfloat16* ptr) {
  const uint2 raw = __ldcs(reinterpret_cast<const uint2*>(ptr));
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// 64 registers per thread (the minimum-blocks bound): two 16-warp CTAs per SM, so the
// merge CTAs of a 48-row tile with ~150 splits (192 of them) run in one wave.
template <int W, int SL>
__global__ void __launch_bounds__(32 * W, 1024 / (32 * W)) lse_merge_kernel(const PlanMerge* merges, const __nv_bfloat16* part_o,
                                                                 const float* part_lse, __nv_bfloat16* out, float* lse) {
  static_assert(SL == 4 || SL == 8, "4 or 8 column slices per row");
  constexpr int kCols = kDv / SL / 32;  // value columns per lane: 4 or 2
  __shared__ float m_s[W], l_s[W];
  __shared__ float4 acc_s[W][32];
  // the merge item is plan data, written before the fold kernel ran: read it while the
  // fold kernel finishes, then wait for the partials
  const PlanMerge m = merges[blockIdx.y];
  ptx::pdl_wait_primary();
  const int row = blockIdx.x / SL, slice = blockIdx.x % SL;
  if (row >= m.nrows) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ns = m.n_splits;  // the planner keeps this <= kMergeMaxSplits
  const int col = slice * (kDv / SL) + kCols * lane;
  const __nv_bfloat16* base = part_o + (size_t)(m.part_row0 + row) * kDv + col;
  const size_t split_stride = (size_t)m.nrows * kDv;
  // Warp w folds its splits w, w + W, ... into a running (max M_w, sum l_w = sum_s e^(L_s -
  // M_w), acc_w = sum_s e^(L_s - M_w) O_s), kMergeBatch splits per round trip (their
  // partial O and LSE loads issued together); one barrier then combines the W warps:
  // L = M + ln l, O = acc / l. A split that the row cannot see has L_s = -inf: weight 0.
  float mw = -INFINITY, lw = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = warp; s0 < ns; s0 += W * kMergeBatch) {
    uint2 v[kMergeBatch];  // kCols bf16 partial-O values each, unpacked when used
    float x[kMergeBatch];
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const int s = s0 + W * u;
      if constexpr (kCols == 4) {
        v[u] = s < ns ? __ldcs(reinterpret_cast<const uint2*>(base + (size_t)s * split_stride)) : make_uint2(0u, 0u);
      } else {
        v[u].x = s < ns ? __ldcs(reinterpret_cast<const unsigned int*>(base + (size_t)s * split_stride)) : 0u;
        v[u].y = 0u;
      }
      x[u] = s < ns ? part_lse[m.part_row0 + s * m.nrows + row] : -INFINITY;
    }
    float mb = mw;
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) mb = fmaxf(mb, x[u]);
    if (mb == -INFINITY) continue;  // nothing visible so far
    const float sc = mw == -INFINITY ? 0.f : __expf(mw - mb);
    lw *= sc;
    acc.x *= sc; acc.y *= sc; acc.z *= sc; acc.w *= sc;
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const float w = x[u] == -INFINITY ? 0.f : __expf(x[u] - mb);
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v[u].x));
      lw += w;
      acc.x += w * a.x; acc.y += w * a.y;
      if constexpr (kCols == 4) {
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v[u].y));
        acc.z += w * b.x; acc.w += w * b.y;
      }
    }
    mw = mb;
  }
  if (lane == 0) {
    m_s[warp] = mw;
    l_s[warp] = lw;
  }
  acc_s[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
    // lane i < W holds warp i's (M_i, l_i): maximum and weights across the lanes
    const float mi = lane < W ? m_s[lane] : -INFINITY;
    float M = mi;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float fi = mi == -INFINITY ? 0.f : __expf(mi - M);
    float l = lane < W ? fi * l_s[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < W; ++i) {
      const float f = __shfl_sync(0xffffffffu, fi, i);
      const float4 a = acc_s[i][lane];
      r.x += f * a.x; r.y += f * a.y; r.z += f * a.z; r.w += f * a.w;
    }
    const float inv = 1.f / l;
    const int qr = m.qrow0 + row;
    if constexpr (kCols == 4)
      *reinterpret_cast<uint2*>(out + (size_t)qr * kDv + col) =
          make_uint2(pack_bf16(r.x * inv, r.y * inv), pack_bf16(r.z * inv, r.w * inv));
    else
      *reinterpret_cast<uint32_t*>(out + (size_t)qr * kDv + col) = pack_bf16(r.x * inv, r.y * inv);
    if (lse && slice == 0 && lane == 0) lse[qr] = M + __logf(l);
  }
}

// The same merge for plans whose row tiles have at most kMergeSmallSplits splits (ragged
// batches cut into many short units): one warp per (packed row, quarter of the value
// columns), all of its partial-O loads issued at once, the LSE reduction done across the
// warp's lanes (lane s holds split s). A CTA of 8 warps covers two rows.
constexpr int kMergeSmallSplits = 16;
constexpr int kMergeSmallWarps = 8;

__global__ void __launch_bounds__(32 * kMergeSmallWarps) lse_merge_small_kernel(const PlanMerge* merges,
                                                                                const __nv_bfloat16* part_o,
                                                                                const float* part_lse,
                                                                                __nv_bfloat16* out, float* lse) {
  const PlanMerge m = merges[blockIdx.y];  // plan data: read before the wait, as above
  ptx::pdl_wait_primary();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int idx = blockIdx.x * kMergeSmallWarps + warp;
  const int row = idx >> 2, quarter = idx & 3;
  if (row >= m.nrows) return;
  const int ns = m.n_splits;  // <= kMergeSmallSplits (checked on the host)
  const int col = quarter * 128 + 4 * lane;
  const __nv_bfloat16* base = part_o + (size_t)(m.part_row0 + row) * kDv + col;
  const size_t split_stride = (size_t)m.nrows * kDv;
  float4 v[kMergeSmallSplits];
#pragma unroll
  for (int s = 0; s < kMergeSmallSplits; ++s)
    v[s] = s < ns ? load_part4(base + (size_t)s * split_stride) : make_float4(0.f, 0.f, 0.f, 0.f);
  const float x = lane < ns ? part_lse[m.part_row0 + lane * m.nrows + row] : -INFINITY;
  float mx = x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = x == -INFINITY ? 0.f : __expf(x - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float L = mx + __logf(sum);
  const float w = x == -INFINITY ? 0.f : __expf(x - L);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int s = 0; s < kMergeSmallSplits; ++s) {
    const float ws = __shfl_sync(0xffffffffu, w, s);
    if (s < ns) {
      acc.x += ws * v[s].x; acc.y += ws * v[s].y; acc.z += ws * v[s].z; acc.w += ws * v[s].w;
    }
  }
  const int qr = m.qrow0 + row;
  *reinterpret_cast<uint2*>(out + (size_t)qr * kDv + col) = make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
  if (lse && quarter == 0 && lane == 0) lse[qr] = L;
}

int rows_cap_for(int kv_dtype) {
  (void)kv_dtype;
  return kRowsCap;
}

int max_splits_for_merge() { return kMergeMaxSplits; }

// ------------------------------------------------------------------ host side
size_t workspace_bytes_for(int n_part_rows);
int check_plan(const void* plan_host, size_t plan_bytes, const PlanHeader** out);
int launch_pair_kernel(int dev, const PlanHeader* h, const void* q, const void* kv_cache, int num_pages,
                       const Params& prm, cudaStream_t st);
int pair_slots_on_device(int dev, int* slots);

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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
             fp8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return set_error(MLA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");

  const bool fp8 = h->kv_dtype == MLA_KV_FP8_E4M3;
  alignas(64) CUtensorMap tq, tkv;
  CUresult r = encode_chunked(enc, &tq, q, false, (uint64_t)h->total_q * (uint64_t)h->num_heads, kRowsCap);
  if (r != CUDA_SUCCESS) return set_error(MLA_ERR_CUDA, "tensor map for q failed (CUresult %d)", (int)r);
  r = encode_chunked(enc, &tkv, kv_cache, fp8, (uint64_t)num_pages * kPage, kTileKeys);
  if (r != CUDA_SUCCESS) return set_error(MLA_ERR_CUDA, "tensor map for kv_cache failed (CUresult %d)", (int)r);

  Params prm;
  prm.units = (const PlanUnit*)((const uint8_t*)plan_dev + h->units_off);
  prm.q = (const __nv_bfloat16*)q;
  prm.q_rows = h->total_q * h->num_heads;
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
  prm.part_o = (__nv_bfloat16*)workspace;
  prm.part_lse =
      ws_need ? (float*)((uint8_t*)workspace + ((size_t)h->n_part_rows * kDv * kPartOElemBytes + 255) / 256 * 256) : nullptr;
  prm.status = status_dev;
  prm.wait_budget = h->debug_skip_copy > 0 ? kWaitBudgetTest : kWaitBudget;
  prm.skip_copy = h->debug_skip_copy - 1;
  cudaStream_t st = (cudaStream_t)stream;
  if (h->cta_pair) {
    if (fp8) return set_error(MLA_ERR_PLAN, "a two-CTA plan needs a bf16 cache");
    rc = launch_pair_kernel(dev, h, q, kv_cache, num_pages, prm, st);
    if (rc != MLA_OK) return rc;
  } else {
    if (fp8)
      fold_decode_kernel<true><<<h->n_units, Roles<true>::kThreads, kSmemBytes, st>>>(tq, tkv, prm);
    else
      fold_decode_kernel<false><<<h->n_units, Roles<false>::kThreads, kSmemBytes, st>>>(tq, tkv, prm);
    ce = cudaGetLastError();
    if (ce != cudaSuccess) return set_error(MLA_ERR_CUDA, "fold kernel launch: %s", cudaGetErrorString(ce));
  }
  if (h->n_merge > 0) {
    // the warp-per-row merge when every row tile has few splits, else the CTA-per-row one
    const PlanMerge* mh = (const PlanMerge*)((const uint8_t*)plan_host + h->merge_off);
    int max_ns = 0;
    for (int i = 0; i < h->n_merge; ++i) max_ns = max(max_ns, mh[i].n_splits);
    const bool small = max_ns <= kMergeSmallSplits;
    // CTA-per-row merge: 8 column slices per row while that keeps the CTAs within about
    // two-thirds of the SMs (a 12- or 24-row merge: its loads spread over twice the SMs),
    // else 4 (more CTAs than that queue for SMs and cost more than they spread)
    const int slices = (long long)h->rows_cap * 8 * h->n_merge <= kMergeWideSlicesMaxCtas ? 8 : 4;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = small ? dim3((unsigned)((h->rows_cap * 4 + kMergeSmallWarps - 1) / kMergeSmallWarps), (unsigned)h->n_merge, 1)
                        : dim3((unsigned)(h->rows_cap * slices), (unsigned)h->n_merge, 1);
    // CTA-per-row merge: just enough warps for one round trip of loads (fewer registers per
    // CTA, so more of them fit on an SM as the fold kernel's CTAs leave)
    const int large_warps = max_ns <= 4 * kMergeBatch ? 4 : max_ns <= 8 * kMergeBatch ? 8 : kMergeWarps;
    cfg.blockDim = dim3(small ? 32 * kMergeSmallWarps : 32 * large_warps, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    auto merge_fn = small ? lse_merge_small_kernel
                    : slices == 8 ? (large_warps == 4   ? lse_merge_kernel<4, 8>
                                     : large_warps == 8 ? lse_merge_kernel<8, 8>
                                                        : lse_merge_kernel<kMergeWarps, 8>)
                                  : (large_warps == 4   ? lse_merge_kernel<4, 4>
                                     : large_warps == 8 ? lse_merge_kernel<8, 4>
                                                        : lse_merge_kernel<kMergeWarps, 4>);
    ce = cudaLaunchKernelEx(&cfg, merge_fn, (const PlanMerge*)((const uint8_t*)plan_dev + h->merge_off),
                            (const __nv_bfloat16*)prm.part_o, (const float*)prm.part_lse, (__nv_bfloat16*)out, lse);
    if (ce != cudaSuccess) return set_error(MLA_ERR_CUDA, "merge kernel launch: %s", cudaGetErrorString(ce));
  }
  return MLA_OK;
}

extern "C" int mla_device_pair_slots(int device, int* slots) {
  clear_error();
  if (!slots) return set_error(MLA_ERR_INVALID_ARG, "slots must not be NULL");
  int rc = prepare_device(device);
  if (rc != MLA_OK) return rc;
  int cur = 0;
  cudaError_t ce = cudaGetDevice(&cur);
  if (ce != cudaSuccess) return set_error(MLA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(ce));
  if (cur != device && (ce = cudaSetDevice(device)) != cudaSuccess)
    return set_error(MLA_ERR_CUDA, "cudaSetDevice: %s", cudaGetErrorString(ce));
  rc = pair_slots_on_device(device, slots);
  if (cur != device) cudaSetDevice(cur);
  return rc;
}
