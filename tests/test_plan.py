"""Host-side tests of the C-ABI library: exports, planner invariants, argument checks.
No GPU needed: the planner is host-only and mla_decode_run validates every argument
before it touches the CUDA runtime."""
import ctypes

import numpy as np
import pytest

from mla_speculative_verify_gb300 import binding, inputs
from tests.plan_reader import read_plan

KV = binding.MLA_KV_BF16


def test_library_exports_every_declared_symbol():
    lib = binding.load()
    names = binding.declared_functions()
    assert set(names) >= {"mla_decode_plan", "mla_decode_plan_ex", "mla_decode_plan_info", "mla_decode_run",
                          "mla_last_error", "mla_version"}
    for name in names:
        assert hasattr(lib, name), name
    assert set(binding.SIGNATURES) == set(names)
    assert lib.mla_version() >= 100


def _fold(q, H):
    return max(f for f in range(1, q + 1) if q % f == 0 and H * f <= 128)


CASES = [
    ([4096], [2], 12), ([131072], [1], 12), ([131072], [8], 12), ([1 << 20], [8], 12), ([32768], [8], 96),
    ([131072], [1], 96), ([20000, 17000, 30000, 16384], [1, 2, 3, 4], 48), ([25000] * 5, [4] * 5, 128),
    ([1], [1], 1), ([8], [8], 12), ([65], [3], 7), ([64 * 5 + 1], [6], 20),
]


@pytest.mark.parametrize("seq_lens,q_lens,H", CASES)
@pytest.mark.parametrize("num_sms", [152, 7])
def test_plan_invariants(seq_lens, q_lens, H, num_sms):
    buf, ws = binding.plan(seq_lens, q_lens, H, KV, num_sms)
    p = read_plan(buf)
    hd = p["header"]
    assert hd["batch"] == len(seq_lens) and hd["num_heads"] == H and hd["total_q"] == sum(q_lens)
    cu = np.concatenate([[0], np.cumsum(q_lens)])
    # every (global row, key) pair is covered exactly once by the units
    cover = {}
    for u in p["units"]:
        b = u["b"]
        ctx = seq_lens[b]
        assert 0 <= u["kv_begin"] < u["kv_end"] <= ctx
        assert u["kv_begin"] % 64 == 0
        assert u["kv_end"] % 64 == 0 or u["kv_end"] == ctx
        assert 1 <= u["nrows"] <= (96 if hd["cta_pair"] else 48)
        # the request fields repeated in the unit record match the request table
        req = p["requests"][b]
        assert (u["ctx"], u["q"], u["tok0"]) == (req["ctx"], req["q"], req["tok0"]) == (ctx, q_lens[b], cu[b])
        r0, r1 = u["qrow0"], u["qrow0"] + u["nrows"]
        assert cu[b] * H <= r0 and r1 <= cu[b + 1] * H, "a unit's rows stay inside its request"
        for r in range(r0, r1, max(1, (r1 - r0) // 3)):
            cover.setdefault(r, []).append((u["kv_begin"], u["kv_end"]))
    for r, spans in cover.items():
        spans.sort()
        b = int(np.searchsorted(cu, r // H, side="right") - 1)
        assert spans[0][0] == 0 and spans[-1][1] == seq_lens[b]
        for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
            assert a1 == b0
    # fold groups: a unit's rows never straddle two fold groups
    for u in p["units"]:
        b = u["b"]
        F = _fold(q_lens[b], H)
        g0 = (u["qrow0"] // H - cu[b]) // F
        g1 = ((u["qrow0"] + u["nrows"] - 1) // H - cu[b]) // F
        assert g0 == g1
        assert p["requests"][b]["fold"] == F
    # merge items point at exactly the split units' partial rows
    parts = sorted((u["part_row0"], u["nrows"]) for u in p["units"] if u["part_row0"] >= 0)
    covered = sum(n for _, n in parts)
    assert covered == hd["n_part_rows"]
    for m in p["merges"]:
        assert m["n_splits"] >= 2
    # partial layout: split s of a row tile writes its rows at merge part_row0 + s * nrows + r,
    # and every workspace partial row is written by exactly one unit
    by_tile = {m["qrow0"]: m for m in p["merges"]}
    written = []
    for u in p["units"]:
        if u["part_row0"] < 0:
            assert u["n_splits"] == 1
            continue
        m = by_tile[u["qrow0"]]
        assert m["nrows"] == u["nrows"] and m["n_splits"] == u["n_splits"]
        assert u["part_row0"] == m["part_row0"] + u["split"] * u["nrows"]
        written += [u["part_row0"] + r for r in range(u["nrows"])]
    assert sorted(written) == list(range(hd["n_part_rows"]))
    # bf16 partial O rows (1 KB each) and fp32 partial LSE, each block 256-byte aligned
    assert ws == (0 if hd["n_part_rows"] == 0 else
                  ((hd["n_part_rows"] * 512 * 2 + 255) // 256 * 256 + (hd["n_part_rows"] * 4 + 255) // 256 * 256))
    # the read-once flag: set exactly when the request is one fold group of one row tile
    for u in p["units"]:
        F = p["requests"][u["b"]]["fold"]
        one_tile = q_lens[u["b"]] == F and (H * F <= 48 or hd["cta_pair"])
        assert u["flags"] == (1 if one_tile else 0)
    # clusters of two CTAs only on request
    assert hd["cta_pair"] == 0
    # the units fill the SMs without leaving most of them idle
    total_pages = sum(-(-s // 64) for s in seq_lens)
    if total_pages >= 4 * num_sms:
        assert len(p["units"]) * (2 if hd["cta_pair"] else 1) >= num_sms // 2


def test_plan_forced_splits_and_fold():
    opts = binding.PlanOptions(force_splits=5, max_rows_per_cta=16, min_pages_per_split=0, force_fold=1)
    buf, _ = binding.plan([1000], [4], 12, KV, 152, opts)
    p = read_plan(buf)
    assert all(u["nrows"] <= 16 for u in p["units"])
    assert all(u["n_splits"] == 5 for u in p["units"])
    assert p["requests"][0]["fold"] == 1
    assert len(p["units"]) == 5 * 4  # 4 tokens x 12 heads = 4 tiles of 12 rows, 5 splits each


@pytest.mark.parametrize("args,code", [
    (dict(seq_lens=[10], q_lens=[11], H=12), binding.MLA_ERR_INVALID_ARG),
    (dict(seq_lens=[10], q_lens=[0], H=12), binding.MLA_ERR_INVALID_ARG),
    (dict(seq_lens=[10], q_lens=[1], H=0), binding.MLA_ERR_UNSUPPORTED),
    (dict(seq_lens=[10], q_lens=[1], H=129), binding.MLA_ERR_UNSUPPORTED),
    (dict(seq_lens=[10], q_lens=[1], H=12, page_size=32), binding.MLA_ERR_UNSUPPORTED),
    (dict(seq_lens=[10], q_lens=[1], H=12, kv_dtype=7), binding.MLA_ERR_INVALID_ARG),
    (dict(seq_lens=[10], q_lens=[1], H=12, num_sms=0), binding.MLA_ERR_INVALID_ARG),
])
def test_plan_rejects(args, code):
    with pytest.raises(binding.MlaError) as e:
        binding.plan(args["seq_lens"], args["q_lens"], args["H"], args.get("kv_dtype", KV), args.get("num_sms", 152),
                     page_size=args.get("page_size", 64))
    assert e.value.code == code
    assert binding.last_error()


def test_plan_buffer_too_small():
    lib = binding.load()
    s = np.array([100], np.int32)
    q = np.array([2], np.int32)
    nb, ws = ctypes.c_size_t(0), ctypes.c_size_t(0)
    small = np.zeros(16, np.uint8)
    rc = lib.mla_decode_plan(s.ctypes.data_as(binding._I32P), q.ctypes.data_as(binding._I32P), 1, 12, 64, KV, 152,
                             small.ctypes.data_as(ctypes.c_void_p), 16, ctypes.byref(nb), ctypes.byref(ws))
    assert rc == binding.MLA_ERR_BUFFER and nb.value > 16


def _run_args(plan, **over):
    a = dict(plan_dev=0x10000, plan_host=plan, q=0x20000, kv=0x30000, pt=0x40000, stride=4, num_pages=8,
             seq=0x50000, ql=0x60000, sm=0.07, kvs=1.0, out=0x70000, lse=0x80000, ws=None, ws_bytes=0, status=None)
    a.update(over)
    return a


def _call_run(a):
    lib = binding.load()
    P = ctypes.c_void_p
    ph = a["plan_host"]
    return lib.mla_decode_run(P(a["plan_dev"]) if a["plan_dev"] else None, ph.ctypes.data_as(P), ph.nbytes,
                              P(a["q"]) if a["q"] else None, P(a["kv"]), P(a["pt"]), a["stride"], a["num_pages"],
                              P(a["seq"]), P(a["ql"]), a["sm"], a["kvs"], P(a["out"]),
                              P(a["lse"]) if a["lse"] else None, P(a["ws"]) if a["ws"] else None, a["ws_bytes"],
                              P(a["status"]) if a["status"] else None, None)


@pytest.mark.parametrize("over,code", [
    (dict(plan_dev=0), binding.MLA_ERR_INVALID_ARG),
    (dict(q=0), binding.MLA_ERR_INVALID_ARG),
    (dict(q=0x20008), binding.MLA_ERR_INVALID_ARG),          # misaligned for TMA
    (dict(lse=0x80002), binding.MLA_ERR_INVALID_ARG),
    (dict(stride=1), binding.MLA_ERR_INVALID_ARG),            # shorter than the longest request
    (dict(num_pages=0), binding.MLA_ERR_INVALID_ARG),
    (dict(sm=0.0), binding.MLA_ERR_INVALID_ARG),
    (dict(kvs=float("nan")), binding.MLA_ERR_INVALID_ARG),
])
def test_run_rejects_bad_arguments_before_any_launch(over, code):
    plan, ws = binding.plan([200], [2], 12, KV, 152, binding.PlanOptions(force_splits=1))
    assert ws == 0
    assert _call_run(_run_args(plan, **over)) == code


def test_run_rejects_small_workspace_and_foreign_plan():
    plan, ws = binding.plan([20000], [2], 12, KV, 152)
    assert ws > 0
    assert _call_run(_run_args(plan, stride=400, ws=None, ws_bytes=0)) == binding.MLA_ERR_BUFFER
    assert _call_run(_run_args(plan, stride=400, ws=0x100000, ws_bytes=ws - 1)) == binding.MLA_ERR_BUFFER
    bad = plan.copy()
    bad[:4] = 0
    assert _call_run(_run_args(bad, stride=400)) == binding.MLA_ERR_PLAN


def _lpt_makespan(lens, num_sms, start_cost=2):
    """End of an in-order dispatch of units (each SM takes the next unit when free)."""
    import heapq

    sms = [0] * num_sms
    for n in lens:
        t = heapq.heappop(sms)
        heapq.heappush(sms, t + n + start_cost)
    return max(sms)


@pytest.mark.parametrize("q", [1, 2, 4, 8])
def test_plan_single_long_request_fits_one_wave(q):
    """One long request: at most one unit per SM, and no unit much longer than the per-SM
    share of the tile-pages."""
    buf, _ = binding.plan([131072], [q], 12, KV, 152)
    p = read_plan(buf)
    units = p["units"]
    slots = 76 if p["header"]["cta_pair"] else 152  # q = 8: 96-row groups on clusters of two CTAs
    assert len(units) <= slots
    pages = [-(-(u["kv_end"] - u["kv_begin"]) // 64) for u in units]
    assert max(pages) <= -(-sum(pages) // slots) + 1


@pytest.mark.parametrize("H", [48, 96, 128])
def test_plan_balances_ragged_batches(H):
    """A ragged batch whose row tiles do not divide evenly over the SMs: units come longest
    first and an in-order dispatch ends within 15 % of the even share."""
    g = np.random.default_rng(7 + H)
    q_lens = g.integers(1, 5, size=32)
    seq_lens = g.integers(16384, 32769, size=32)
    buf, _ = binding.plan(seq_lens, q_lens, H, 1, 152)
    units = read_plan(buf)["units"]
    pages = [-(-(u["kv_end"] - u["kv_begin"]) // 64) for u in units]
    assert pages == sorted(pages, reverse=True)
    assert _lpt_makespan(pages, 152) <= 1.15 * (sum(pages) / 152 + 2)


def test_plan_carries_the_timeout_test_option_only_when_asked():
    buf, _ = binding.plan([4096], [2], 12, KV, 152)
    assert read_plan(buf)["header"]["debug_skip_copy"] == 0
    buf, _ = binding.plan([4096], [2], 12, KV, 152, binding.PlanOptions(debug_skip_copy=3))
    assert read_plan(buf)["header"]["debug_skip_copy"] == 3
    with pytest.raises(binding.MlaError):
        binding.plan([4096], [2], 12, KV, 152, binding.PlanOptions(debug_skip_copy=-1))


def _max_piece(plan_buf):
    return max(-(-(u["kv_end"] - u["kv_begin"]) // 64) for u in read_plan(plan_buf)["units"])


@pytest.mark.parametrize("H,pattern,best", [(48, "ragged", 212), (48, "uniform", 342), (128, "ragged", 318),
                                            (128, "uniform", 342)])
def test_planner_picks_the_piece_length_measured_fastest(H, pattern, best):
    """The B=32 MTP-3 batches (e4m3, ctx 16k-32k, both patterns on the same context lengths).
    On GB300 every piece length the planner can choose was timed (mla_decode_run, graph
    replay); the fastest were 212 / 342 pages (H=48 ragged 279.0 us, uniform 434.2 us) and
    318 / 342 pages (H=128 ragged 742.6 us, uniform 1164.7 us), against 290.1 / 436.9 /
    762.8 / 1193.7 us for the earlier start-up cost of 2 page-times. The planner's dispatch
    model must keep choosing those lengths."""
    seq_lens, q_lens = inputs.ragged_lengths(pattern)
    buf, _ = binding.plan(seq_lens, q_lens, H, binding.MLA_KV_FP8_E4M3, 152)
    assert _max_piece(buf) == best


def test_ragged_and_uniform_batches_of_equal_work_get_different_pieces():
    """flashinfer #5588 ("What was measured", host-plan row) found that unit sizes good for
    ragged query lengths lose on uniform ones of the same geometry, and that a plan built
    from host scalars alone could not tell the two apart. This planner receives every
    request's q: a ragged (MTP-3) and a uniform (q = 4) H=128 batch of the same total
    tile-pages (the uniform batch's contexts scaled down) get different piece lengths and
    unit counts, because their row tiles (48- and 32-row) fall into fold groups differently."""
    sl_r, ql_r = inputs.ragged_lengths("ragged")
    sl_u, ql_u = inputs.ragged_lengths("uniform")
    sl_u = np.maximum(64, (sl_u * (ql_r.sum() / ql_u.sum())).astype(np.int64))
    kv = binding.MLA_KV_FP8_E4M3
    br, _ = binding.plan(sl_r, ql_r, 128, kv, 152)
    bu, _ = binding.plan(sl_u, ql_u, 128, kv, 152)
    work = [sum(-(-(x["kv_end"] - x["kv_begin"]) // 64) for x in read_plan(b)["units"]) for b in (br, bu)]
    assert abs(work[0] - work[1]) <= 0.02 * work[0]
    assert _max_piece(br) != _max_piece(bu)
    assert len(read_plan(br)["units"]) != len(read_plan(bu)["units"])


def test_unit_pages_option_forces_the_piece_length():
    buf, _ = binding.plan([131072], [1], 12, KV, 152, binding.PlanOptions(unit_pages=20))
    pages = sorted({-(-(u["kv_end"] - u["kv_begin"]) // 64) for u in read_plan(buf)["units"]})
    assert pages == [8, 20]  # 2048 pages = 102 x 20 + 8
    with pytest.raises(binding.MlaError):
        binding.plan([4096], [2], 12, KV, 152, binding.PlanOptions(unit_pages=8, force_splits=2))


@pytest.mark.parametrize("seq_lens,q_lens,H", [([131072], [8], 12), ([3000, 5000], [8, 16], 12), ([700], [1], 80),
                                               ([900], [6], 16), ([700], [4], 12), ([700], [1], 128)])
def test_cta_pair_plans(seq_lens, q_lens, H):
    """With cta_pair, a bf16 plan whose every fold group has 49..96 rows gets one unit per
    fold group and key piece (rows up to 96), sized for num_sms / 2 clusters; other plans
    (48 rows, 128 rows, an e4m3 cache) stay on single CTAs."""
    rows = [_fold(q, H) * H for q in q_lens]
    eligible = all(48 < r <= 96 for r in rows)
    for kv in (KV, binding.MLA_KV_FP8_E4M3):
        buf, _ = binding.plan(seq_lens, q_lens, H, kv, 152, binding.PlanOptions(cta_pair=1))
        p = read_plan(buf)
        assert p["header"]["cta_pair"] == int(eligible and kv == KV)
        if p["header"]["cta_pair"]:
            assert {u["nrows"] for u in p["units"]} == set(rows)
            if len(seq_lens) == 1 and q_lens[0] * H == rows[0]:
                assert len(p["units"]) <= 76
