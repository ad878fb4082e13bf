// plan.cpp -- host-only split-KV work partition for MLA verify decode.
//
// The planner works from host-known scalars only (seq_lens, q_lens, H, the SM
// count), as the host plan of flashinfer PR #5588 ("What was measured" table,
// host-plan row) does. Steps:
//   1. fold_sq (sglang PR #33650, "Why" paragraph): F = largest divisor of q with
//      H * F <= 128; the q tokens form q / F groups of F * H packed rows
//      (row = token * H + head, contiguous in Q and in the output).
//   2. A group's packed rows are cut into CTA row tiles of at most rows_cap rows
//      (the shared-memory budget of one CTA, see kernel_sm103.cu). The tiles of
//      one group are adjacent in the unit list, so they stream the same pages at
//      the same time and the second read is served by L2.
//   3. Each group's key range [0, ctx) is cut into page-aligned splits of about the
//      per-SM share of the work; split units write partial (O, LSE) rows that the
//      merge kernel combines.
#include <algorithm>
#include <functional>
#include <queue>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "mla_decode.h"
#include "plan_format.h"
#include "status.h"

namespace mla {

int rows_cap_for(int kv_dtype);  // defined next to the kernel
int max_splits_for_merge();       // defined next to the merge kernel
int pair_rows_cap();              // defined next to the two-CTA kernel

static int fold_factor(int q, int H) {
  int best = 1;
  for (int f = 1; f <= q; ++f)
    if (q % f == 0 && (long long)H * f <= 128) best = f;
  return best;
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t workspace_bytes_for(int n_part_rows) {
  if (n_part_rows <= 0) return 0;
  return align_up((size_t)n_part_rows * kDv * kPartOElemBytes, 256) + align_up((size_t)n_part_rows * sizeof(float), 256);
}

}  // namespace mla

using namespace mla;

extern "C" int mla_decode_plan_ex(const int32_t* seq_lens_h, const int32_t* q_lens_h, int batch, int num_heads,
                                  int page_size, int kv_dtype, int num_sms, const mla_plan_options* opts,
                                  void* plan_buf, size_t plan_buf_bytes, size_t* plan_bytes_out,
                                  size_t* workspace_bytes_out) {
  clear_error();
  if (!seq_lens_h || !q_lens_h) return set_error(MLA_ERR_INVALID_ARG, "seq_lens_h and q_lens_h must not be NULL");
  if (batch < 1) return set_error(MLA_ERR_INVALID_ARG, "batch must be >= 1 (got %d)", batch);
  if (num_heads < 1 || num_heads > MLA_MAX_HEADS)
    return set_error(MLA_ERR_UNSUPPORTED, "num_heads must be in [1, %d] (got %d)", MLA_MAX_HEADS, num_heads);
  if (page_size != kPage) return set_error(MLA_ERR_UNSUPPORTED, "only page_size 64 is supported (got %d)", page_size);
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3)
    return set_error(MLA_ERR_INVALID_ARG, "kv_dtype must be MLA_KV_BF16 or MLA_KV_FP8_E4M3 (got %d)", kv_dtype);
  if (num_sms < 1) return set_error(MLA_ERR_INVALID_ARG, "num_sms must be >= 1 (got %d)", num_sms);
  mla_plan_options o{};
  if (opts) o = *opts;
  int cap = rows_cap_for(kv_dtype);
  if (o.max_rows_per_cta > 0) {
    if (o.max_rows_per_cta % 16 != 0 || o.max_rows_per_cta > cap)
      return set_error(MLA_ERR_INVALID_ARG, "max_rows_per_cta must be a multiple of 16 and <= %d (got %d)", cap,
                       o.max_rows_per_cta);
    cap = o.max_rows_per_cta;
  }
  if (o.force_splits < 0 || o.min_pages_per_split < 0 || o.force_fold < 0 || o.unit_pages < 0 || o.cta_pair < 0 ||
      o.pair_slots < 0 || o.debug_skip_copy < 0)
    return set_error(MLA_ERR_INVALID_ARG, "plan options must be >= 0");
  if (o.force_splits > 0 && o.unit_pages > 0)
    return set_error(MLA_ERR_INVALID_ARG, "force_splits and unit_pages exclude each other");

  long long total_q = 0;
  int max_pages = 0;
  for (int b = 0; b < batch; ++b) {
    int ctx = seq_lens_h[b], q = q_lens_h[b];
    if (q < 1) return set_error(MLA_ERR_INVALID_ARG, "q_lens[%d] = %d must be >= 1", b, q);
    if (ctx < q) return set_error(MLA_ERR_INVALID_ARG, "seq_lens[%d] = %d is smaller than q_lens[%d] = %d", b, ctx, b, q);
    if (o.force_fold > 0 && q % o.force_fold != 0)
      return set_error(MLA_ERR_INVALID_ARG, "force_fold %d does not divide q_lens[%d] = %d", o.force_fold, b, q);
    total_q += q;
    max_pages = std::max(max_pages, (ctx + kPage - 1) / kPage);
  }
  if (total_q * num_heads > (1LL << 30)) return set_error(MLA_ERR_INVALID_ARG, "too many query rows");

  // On request (cta_pair), a bf16 cache whose every fold group has 49..96 packed rows runs
  // on clusters of two CTAs, one unit per fold group and key piece: each CTA streams half
  // of every page's columns, so the page enters the pair once instead of once per 48-row
  // tile. (Off by default: on GB300 the 48-row single-CTA tiles are faster.)
  bool pair = kv_dtype == MLA_KV_BF16 && o.cta_pair > 0 && o.max_rows_per_cta == 0;
  for (int b = 0; pair && b < batch; ++b) {
    const int F = o.force_fold > 0 ? o.force_fold : fold_factor(q_lens_h[b], num_heads);
    const int R = F * num_heads;
    pair = R > cap && R <= pair_rows_cap();
  }
  if (pair) cap = pair_rows_cap();
  const int slots = pair ? (o.pair_slots > 0 ? o.pair_slots : std::max(1, num_sms / 2)) : num_sms;

  // --- row tiles ----------------------------------------------------------------------
  struct RowTile { int b, qrow0, nrows, pages; };
  std::vector<RowTile> tiles;
  std::vector<PlanRequest> reqs(batch);
  int tok0 = 0;
  for (int b = 0; b < batch; ++b) {
    int ctx = seq_lens_h[b], q = q_lens_h[b];
    int F = o.force_fold > 0 ? o.force_fold : fold_factor(q, num_heads);
    reqs[b] = PlanRequest{ctx, q, tok0, F};
    int R = F * num_heads;                       // packed rows per fold group
    int n_rt = (R + cap - 1) / cap;
    int T = ((R + n_rt - 1) / n_rt + 15) / 16 * 16;
    if (T > cap) T = cap;
    int pages = (ctx + kPage - 1) / kPage;
    for (int g = 0; g < q / F; ++g) {
      int grow0 = (tok0 + g * F) * num_heads;
      for (int r0 = 0; r0 < R; r0 += T) {
        tiles.push_back(RowTile{b, grow0 + r0, std::min(T, R - r0), pages});
      }
    }
    tok0 += q;
  }

  // --- fold groups ------------------------------------------------------------------
  // tiles [t0, t1) of one fold group: consecutive, same request, qrow0 contiguous
  struct Group { size_t t0, t1; int b, pages, n_split, cap; };  // cap: piece length in pages (0: equal pieces)
  std::vector<Group> groups;
  for (size_t i = 0; i < tiles.size();) {
    size_t j = i;
    int grp_rows = 0;
    const int b = tiles[i].b;
    const int R = reqs[b].fold * num_heads;
    while (j < tiles.size() && tiles[j].b == b && grp_rows < R) { grp_rows += tiles[j].nrows; ++j; }
    groups.push_back(Group{i, j, b, tiles[i].pages, 1, 1});
    i = j;
  }

  // --- splits ----------------------------------------------------------------------
  // Each group is cut into pieces of T pages (the last one shorter); all row tiles of the
  // group are cut at the same boundaries. The units are ordered longest first (below), so
  // the full-length units fill the SMs and the short tails run back to back on the SMs
  // left over. T is the per-SM share of the tile-pages divided by k, for the k whose
  // schedule ends first in a model of the hardware's in-order CTA dispatch: a unit costs
  // a start-up of kStart page-times (its prologue, first copies and Q preparation, the
  // epilogue and its split partial) plus its pages, each weighted by its row tile's cost
  // (a tile of <= 32 rows of an e4m3 cache takes less than a 48-row tile). The model's
  // constants were fitted to measured call times over forced piece lengths on GB300
  // (bf16: a unit start ~ 6 page-times; e4m3: ~ 16). It sees each request's q, so a batch
  // of ragged query lengths, whose fold groups differ in tile count, gets other piece
  // lengths than a uniform one of the same total work. A split keeps at least min_pages
  // pages.
  const int min_pages = o.min_pages_per_split > 0 ? o.min_pages_per_split : 4;
  const int max_splits = max_splits_for_merge();
  const bool fp8 = kv_dtype == MLA_KV_FP8_E4M3;
  const double start_cost = fp8 ? 16.0 : 6.0;
  auto row_cost = [&](int nrows) { return (fp8 && nrows <= 32) ? 0.9 : 1.0; };
  long long tile_pages = 0;
  for (const Group& g : groups) tile_pages += (long long)(g.t1 - g.t0) * g.pages;
  auto assign = [&](long long T) {
    for (auto& g : groups) {
      long long n = o.force_splits > 0 ? o.force_splits : (g.pages + T - 1) / T;
      g.n_split = (int)std::max<long long>(1, std::min<long long>(std::min<long long>(n, g.pages), max_splits));
      // pieces of T pages, unless the split count was capped or forced: then equal pieces
      g.cap = (o.force_splits <= 0 && (long long)g.n_split == (g.pages + T - 1) / T) ? (int)T : 0;
    }
  };
  auto piece_pages = [](const Group& g, int s) {
    if (g.cap > 0) return std::min(g.pages, (s + 1) * g.cap) - s * g.cap;
    return (int)((long long)g.pages * (s + 1) / g.n_split - (long long)g.pages * s / g.n_split);
  };
  long long best_T = std::max<long long>(min_pages, (tile_pages + slots - 1) / slots);
  if (o.unit_pages > 0) best_T = o.unit_pages;
  if (o.force_splits <= 0 && o.unit_pages <= 0) {
    double best_end = -1;
    std::vector<std::pair<int, double>> lens;  // (pages, per-page cost) of every unit
    // candidates: the per-SM share divided by 1, 1.25, ... 8, and the longest group's
    // pages divided into 1 .. 64 equal pieces
    std::vector<long long> cands;
    for (int k4 : {4, 5, 6, 8, 10, 12, 16, 20, 24, 32})
      cands.push_back((4 * tile_pages + (long long)slots * k4 - 1) / ((long long)slots * k4));
    int longest = 0;
    for (const Group& g : groups) longest = std::max(longest, g.pages);
    for (int n = 1; n <= 64; ++n) cands.push_back((longest + n - 1) / n);
    std::sort(cands.begin(), cands.end());
    cands.erase(std::unique(cands.begin(), cands.end()), cands.end());
    for (long long c : cands) {
      const long long T = std::max<long long>(min_pages, c);
      // more than 16 waves of units (beyond one unit per row tile) never pays for its
      // start-up costs; skipping those keeps the search cheap for very long batches
      long long n_units = 0;
      for (const Group& g : groups) n_units += (long long)(g.t1 - g.t0) * ((g.pages + T - 1) / T);
      if (n_units > std::max<long long>(16LL * slots, (long long)tiles.size()) && !cands.empty() && c != cands.back())
        continue;
      assign(T);
      lens.clear();
      for (const Group& g : groups)
        for (int s = 0; s < g.n_split; ++s)
          for (size_t t = g.t0; t < g.t1; ++t) lens.emplace_back(piece_pages(g, s), row_cost(tiles[t].nrows));
      std::stable_sort(lens.begin(), lens.end(),
                       [](const std::pair<int, double>& a, const std::pair<int, double>& b) { return a.first > b.first; });
      std::priority_queue<double, std::vector<double>, std::greater<double>> sm;
      for (int i = 0; i < slots; ++i) sm.push(0.0);
      double end = 0;
      for (const auto& L : lens) {
        const double t = sm.top() + start_cost + L.first * L.second;
        sm.pop();
        sm.push(t);
        end = std::max(end, t);
      }
      if (best_end < 0 || end < best_end - 1e-9) {
        best_end = end;
        best_T = T;
      }
    }
  }
  assign(best_T);

  std::vector<PlanUnit> units;
  std::vector<PlanMerge> merges;
  int part_rows = 0;
  for (const Group& g : groups) {
    const int b = g.b, n_split = g.n_split, pages = g.pages;
    std::vector<int> part0(g.t1 - g.t0, -1);
    if (n_split > 1) {
      for (size_t t = g.t0; t < g.t1; ++t) {
        part0[t - g.t0] = part_rows;
        merges.push_back(PlanMerge{tiles[t].qrow0, tiles[t].nrows, part_rows, n_split});
        part_rows += n_split * tiles[t].nrows;
      }
    }
    for (int s = 0; s < n_split; ++s) {
      int p_begin, p_end;
      if (g.cap > 0) {  // pieces of T = g.cap pages, the last one shorter
        p_begin = s * g.cap;
        p_end = std::min(pages, (s + 1) * g.cap);
      } else {
        p_begin = (int)((long long)pages * s / n_split);
        p_end = (int)((long long)pages * (s + 1) / n_split);
      }
      int kb = p_begin * kPage, ke = std::min(reqs[b].ctx, p_end * kPage);
      for (size_t t = g.t0; t < g.t1; ++t) {
        PlanUnit u;
        u.b = b; u.qrow0 = tiles[t].qrow0; u.nrows = tiles[t].nrows;
        u.kv_begin = kb; u.kv_end = ke;
        u.part_row0 = n_split > 1 ? part0[t - g.t0] + s * tiles[t].nrows : -1;
        u.split = s; u.n_splits = n_split;
        u.ctx = reqs[b].ctx; u.q = reqs[b].q; u.tok0 = reqs[b].tok0;
        // pages read by one row tile only: the request is a single fold group of one tile
        u.flags = (reqs[b].q / reqs[b].fold == 1 && g.t1 - g.t0 == 1) ? kUnitKvReadOnce : 0;
        units.push_back(u);
      }
    }
  }
  // Longest units first: when the grid needs more than one wave, the SMs that finish
  // early pick up the short units. (Stable, so the tiles of a group stay adjacent.)
  if ((long long)units.size() > slots)
    std::stable_sort(units.begin(), units.end(), [](const PlanUnit& a, const PlanUnit& c) {
      return a.kv_end - a.kv_begin > c.kv_end - c.kv_begin;
    });

  size_t req_off = sizeof(PlanHeader);
  size_t units_off = align_up(req_off + sizeof(PlanRequest) * batch, 32);
  size_t merge_off = align_up(units_off + sizeof(PlanUnit) * units.size(), 32);
  size_t total = align_up(merge_off + sizeof(PlanMerge) * merges.size(), 64);
  if (total > (size_t)INT32_MAX) return set_error(MLA_ERR_INVALID_ARG, "plan too large");
  if (plan_bytes_out) *plan_bytes_out = total;
  if (workspace_bytes_out) *workspace_bytes_out = workspace_bytes_for(part_rows);
  if (!plan_buf || plan_buf_bytes < total)
    return set_error(MLA_ERR_BUFFER, "plan buffer needs %zu bytes (got %zu)", total, plan_buf ? plan_buf_bytes : (size_t)0);

  uint8_t* base = (uint8_t*)plan_buf;
  memset(base, 0, total);
  PlanHeader h{};
  h.magic = kPlanMagic; h.version = kPlanVersion;
  h.batch = batch; h.num_heads = num_heads; h.kv_dtype = kv_dtype; h.total_q = (int32_t)total_q;
  h.n_units = (int32_t)units.size(); h.n_merge = (int32_t)merges.size();
  int used_cap = 0;
  for (auto& u : units) used_cap = std::max(used_cap, u.nrows);
  h.rows_cap = used_cap; h.n_part_rows = part_rows; h.max_pages = max_pages;
  h.req_off = (int32_t)req_off; h.units_off = (int32_t)units_off; h.merge_off = (int32_t)merge_off;
  h.total_bytes = (int32_t)total;
  h.debug_skip_copy = o.debug_skip_copy;
  h.cta_pair = pair ? 1 : 0;
  memcpy(base, &h, sizeof h);
  memcpy(base + req_off, reqs.data(), sizeof(PlanRequest) * batch);
  if (!units.empty()) memcpy(base + units_off, units.data(), sizeof(PlanUnit) * units.size());
  if (!merges.empty()) memcpy(base + merge_off, merges.data(), sizeof(PlanMerge) * merges.size());
  return MLA_OK;
}

extern "C" int mla_decode_plan(const int32_t* seq_lens_h, const int32_t* q_lens_h, int batch, int num_heads,
                               int page_size, int kv_dtype, int num_sms, void* plan_buf, size_t plan_buf_bytes,
                               size_t* plan_bytes_out, size_t* workspace_bytes_out) {
  return mla_decode_plan_ex(seq_lens_h, q_lens_h, batch, num_heads, page_size, kv_dtype, num_sms, nullptr, plan_buf,
                            plan_buf_bytes, plan_bytes_out, workspace_bytes_out);
}

namespace mla {

int check_plan(const void* plan_host, size_t plan_bytes, const PlanHeader** out) {
  if (!plan_host) return set_error(MLA_ERR_INVALID_ARG, "plan_host must not be NULL");
  if (plan_bytes < sizeof(PlanHeader)) return set_error(MLA_ERR_PLAN, "plan is %zu bytes, smaller than its header", plan_bytes);
  const PlanHeader* h = (const PlanHeader*)plan_host;
  if (h->magic != kPlanMagic || h->version != kPlanVersion)
    return set_error(MLA_ERR_PLAN, "plan bytes were not written by this library version");
  if ((size_t)h->total_bytes != plan_bytes)
    return set_error(MLA_ERR_PLAN, "plan_bytes %zu differs from the plan's size %d", plan_bytes, h->total_bytes);
  *out = h;
  return MLA_OK;
}

}  // namespace mla

extern "C" int mla_decode_plan_info(const void* plan_host, size_t plan_bytes, int* n_units, int* n_merge,
                                    int* total_q, int* num_heads, int* kv_dtype) {
  clear_error();
  const PlanHeader* h = nullptr;
  int rc = check_plan(plan_host, plan_bytes, &h);
  if (rc != MLA_OK) return rc;
  if (n_units) *n_units = h->n_units;
  if (n_merge) *n_merge = h->n_merge;
  if (total_q) *total_q = h->total_q;
  if (num_heads) *num_heads = h->num_heads;
  if (kv_dtype) *kv_dtype = h->kv_dtype;
  return MLA_OK;
}
