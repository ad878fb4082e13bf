// plan_format.h -- binary layout of a decode plan, shared by the host planner and
// the kernels. A plan is one contiguous byte block: header, request table, work
// units, merge items. The same bytes live in host memory (launch sizing) and in
// device memory (read by the kernels).
#pragma once
#include <stdint.h>

namespace mla {

constexpr uint32_t kPlanMagic = 0x564C4D41u;  // "AMLV"
constexpr uint32_t kPlanVersion = 5;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kPage = 64;
// Split partials of O are stored as bf16 (each split's O is already normalised by its
// own l, so bf16 adds at most 2^-9 relative error before the merge's weighted sum).
constexpr int kPartOElemBytes = 2;
// PlanUnit.flags: the request's cache pages are read by this row tile only (one fold
// group, one tile), so a page can leave L2 right after its copy into shared memory.
constexpr int32_t kUnitKvReadOnce = 1;

struct PlanHeader {
  uint32_t magic, version;
  int32_t batch, num_heads, kv_dtype, total_q;
  int32_t n_units, n_merge;
  int32_t rows_cap;      // largest packed-row tile any unit uses
  int32_t n_part_rows;   // rows of partial (O, LSE) in the workspace
  int32_t max_pages;     // pages of the longest request
  int32_t req_off, units_off, merge_off;  // byte offsets from the plan start
  int32_t total_bytes;
  int32_t debug_skip_copy;  // mla_plan_options.debug_skip_copy (0 in production plans)
  int32_t cta_pair;         // 1: every unit is one fold group of 49..96 rows for a cluster of two CTAs
  int32_t reserved[3];
};
static_assert(sizeof(PlanHeader) == 80, "plan header is 80 bytes");

// One request: ctx keys (verify tokens included), q verify tokens, first global token.
struct PlanRequest {
  int32_t ctx, q, tok0, fold;
};

// One work unit: a tile of packed rows of one fold group over one key range, for one CTA
// (or, in a cta_pair plan, for a cluster of two CTAs that split the tile's columns).
// Packed rows are global Q rows qrow0 .. qrow0 + nrows - 1 (row = token * H + head).
struct PlanUnit {
  int32_t b;           // request
  int32_t qrow0;       // first global Q row of the tile
  int32_t nrows;       // rows in the tile (<= rows_cap)
  int32_t kv_begin;    // first key (multiple of 64)
  int32_t kv_end;      // one past the last key (<= ctx)
  int32_t part_row0;   // first workspace partial row, or -1: write out/lse directly
  int32_t split;       // split index within the row tile
  int32_t n_splits;    // splits of this row tile
  int32_t ctx, q, tok0;  // the request's fields, repeated so that a CTA reads one record
  int32_t flags;         // kUnitKv* bits
};
static_assert(sizeof(PlanUnit) == 48, "plan unit is 48 bytes");

// One merge item: nrows rows whose n_splits partials sit at part_row0 + s * nrows.
struct PlanMerge {
  int32_t qrow0, nrows, part_row0, n_splits;
};

}  // namespace mla
