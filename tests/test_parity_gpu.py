"""GPU parity: the sm_103a path (through the C entry points) against the float64 oracle
on the same seeded inputs, element by element, at sizes that span several pages,
several splits and a ragged tail, plus the full-size workloads on sampled tokens."""
import numpy as np
import pytest
import torch

from mla_speculative_verify_gb300 import inputs
from mla_speculative_verify_gb300.binding import PlanOptions
from tests.gpu_util import assert_close, oracle_rows, run_gpu, run_oracle, sub_problem, to_device, token_rows

pytestmark = pytest.mark.gpu

BF16, FP8 = inputs.KV_BF16, inputs.KV_FP8


def _check(prob, options=None):
    out, lse, _ = run_gpu(prob, options)
    o_ref, l_ref = run_oracle(prob)
    return assert_close(out, lse, o_ref, l_ref)


def test_contiguous_h12_q2_ctx4096():
    """The small contiguous workload at full size."""
    _check(inputs.workload_contiguous_small())


@pytest.mark.parametrize("q", [1, 2, 4, 8])
@pytest.mark.parametrize("kv", [BF16, FP8])
def test_h12_sweep_reduced_ctx(q, kv):
    prob = inputs.make_problem(12, [9000 + 37], [q], kv, seed=2000 + q, poison_tail=True)
    _check(prob)


@pytest.mark.parametrize("q", [1, 8])
@pytest.mark.parametrize("kv", [BF16, FP8])
def test_h96_reduced_ctx(q, kv):
    prob = inputs.make_problem(96, [3000 + 5], [q], kv, seed=2100 + q, poison_tail=True)
    _check(prob)


@pytest.mark.parametrize("H", [48, 128])
@pytest.mark.parametrize("pattern", ["ragged", "uniform"])
def test_ragged_batch_fp8_reduced(H, pattern):
    prob = inputs.workload_ragged(H, pattern, B=32, ctx_lo=300, ctx_hi=900, seed=2200)
    _check(prob)


@pytest.mark.parametrize("seq,q,H", [([1], [1], 12), ([8], [8], 12), ([64], [3], 12), ([65], [2], 20),
                                     ([130], [6], 7), ([200], [5], 128)])
def test_edge_shapes(seq, q, H):
    """ctx == q (only verify keys), one key, exactly one page, one key past a page,
    odd head counts, H = 128."""
    for kv in (BF16, FP8):
        _check(inputs.make_problem(H, seq, q, kv, seed=2300 + seq[0], poison_tail=True))


def test_fp8_zero_and_subnormal_codes():
    """Zero (both signs) and subnormal e4m3 codes in visible keys, and one page of zero
    codes, go straight into the e4m3 tensor-core products."""
    prob = inputs.make_problem(12, [64 * 5 + 9], [4], FP8, seed=2450)
    g = torch.Generator().manual_seed(3)
    rows = prob.kv.shape[0]
    idx = torch.randint(0, rows * 576, (4000,), generator=g)
    codes = torch.tensor([0x00, 0x80, 0x01, 0x87, 0x05, 0x83], dtype=torch.uint8)
    prob.kv.view(-1)[idx] = codes[torch.randint(0, len(codes), (4000,), generator=g)]
    prob.kv[64:128] = 0  # one whole page of zero codes
    _check(prob)


def test_fp8_query_rows_of_very_different_magnitude():
    """The e4m3 path scales each query row by its own power of two before splitting it
    into two e4m3 parts: rows from 2^-14 to 2^3 times the usual size, an all-zero row and
    a row with one large entry must all come out right."""
    prob = inputs.make_problem(12, [64 * 9 + 17], [4], FP8, seed=2460)
    q = prob.q.float()
    rows = q.reshape(-1, 576)
    for r in range(rows.shape[0]):
        rows[r] *= 2.0 ** (-14 + (r * 7) % 18)
    rows[5] = 0
    rows[11] = 0
    rows[11, 300] = 6.0
    prob.q = rows.reshape(prob.q.shape).to(torch.bfloat16)
    _check(prob)


@pytest.mark.parametrize("splits", [16, 17, 40])
@pytest.mark.parametrize("kv", [BF16, FP8])
def test_both_merge_kernels(splits, kv):
    """Up to 16 splits per row tile the warp-per-row merge runs, above it the CTA-per-row
    merge; both against the oracle on a 96-row fold group (two 48-row tiles)."""
    prob = inputs.make_problem(12, [64 * 45 + 21], [8], kv, seed=2470 + splits, poison_tail=True)
    _check(prob, PlanOptions(force_splits=splits))


def test_many_splits_with_empty_causal_partials():
    """One page per split: the last split holds keys that early verify rows may not see."""
    prob = inputs.make_problem(12, [64 * 6 + 3], [8], BF16, seed=2400, poison_tail=True)
    _check(prob, PlanOptions(force_splits=7))


@pytest.mark.parametrize("kv", [BF16, FP8])
def test_fold_less_mode_matches_fold(kv):
    """F = 1 (one token per CTA tile) against the folded plan: same numbers within rounding."""
    prob = inputs.make_problem(12, [5000], [4], kv, seed=2500)
    o1, l1, _ = run_gpu(prob)
    o2, l2, _ = run_gpu(prob, PlanOptions(force_fold=1))
    o_ref, l_ref = run_oracle(prob)
    assert_close(o1, l1, o_ref, l_ref)
    assert_close(o2, l2, o_ref, l_ref)


def test_unsplit_rows_are_bitwise_reproducible():
    prob = inputs.make_problem(12, [3000], [4], BF16, seed=2600)
    opts = PlanOptions(force_splits=1)
    a = run_gpu(prob, opts)
    b = run_gpu(prob, opts)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_split_replay_spread_is_small():
    prob = inputs.make_problem(12, [20000], [8], BF16, seed=2700)
    a = run_gpu(prob)
    b = run_gpu(prob)
    assert np.abs(a[0] - b[0]).max() <= 1e-3 and np.abs(a[1] - b[1]).max() <= 1e-5


def test_graph_replay_with_changed_page_table():
    """Capture one call in a CUDA graph, then permute the pages (cache and table
    together) and replay: same result, no re-plan."""
    from mla_speculative_verify_gb300.decoder import VerifyDecoder

    prob = inputs.make_problem(12, [4000], [4], BF16, seed=2800, extra_pages=8)
    dec = VerifyDecoder(prob.seq_lens, prob.q_lens, prob.H, prob.kv_dtype)
    q, kv, pt = to_device(prob)
    out = torch.zeros((prob.total_q, prob.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((prob.total_q, prob.H), dtype=torch.float32, device="cuda")
    dec.run(q, kv, pt, out, lse, prob.sm_scale)  # warm-up (sets kernel attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            dec.run(q, kv, pt, out, lse, prob.sm_scale)
    g.replay()
    torch.cuda.synchronize()
    o_ref, l_ref = run_oracle(prob)
    assert_close(out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref)
    # move every page to a new physical slot
    n = prob.num_pages
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(5))
    new_kv = torch.empty_like(kv)
    new_kv.view(n, 64, 576)[perm.to("cuda")] = kv.view(n, 64, 576)
    kv.copy_(new_kv)
    pt.copy_(perm.to("cuda")[pt.long()].to(torch.int32))
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert_close(out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref)


def test_plan_mismatch_is_reported_not_faulted():
    from mla_speculative_verify_gb300.binding import MLA_DEVICE_PLAN_MISMATCH

    prob = inputs.make_problem(12, [1000], [2], BF16, seed=2900)
    from mla_speculative_verify_gb300.decoder import VerifyDecoder

    dec = VerifyDecoder(prob.seq_lens, prob.q_lens, prob.H, prob.kv_dtype)
    q, kv, pt = to_device(prob)
    out = torch.zeros((prob.total_q, prob.H, 512), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wrong = torch.tensor([999], dtype=torch.int32, device="cuda")
    dec.run(q, kv, pt, out, None, prob.sm_scale, 1.0, status, seq_lens_dev=wrong)
    torch.cuda.synchronize()
    assert int(status.item()) & MLA_DEVICE_PLAN_MISMATCH
    # the context stays usable
    out2, lse2, st = run_gpu(prob)
    assert st == 0


# ---------------------------------------------------------------- full sizes, sampled tokens
@pytest.mark.parametrize("q", [1, 2, 4, 8])
@pytest.mark.parametrize("kv", [BF16, FP8])
def test_full_size_h12_131k_sampled(q, kv):
    prob = inputs.workload_sweep_131k(q, kv_dtype=kv)
    out, lse, _ = run_gpu(prob)
    toks = sorted({0, q - 1})
    o_ref, l_ref = oracle_rows(prob, toks)
    assert_close(out[toks], lse[toks], o_ref, l_ref)


@pytest.mark.parametrize("q", [2, 4])
@pytest.mark.parametrize("kv", [BF16, FP8])
def test_full_size_h12_512k_sampled(q, kv):
    prob = inputs.workload_sweep_131k(q, ctx=1 << 19, kv_dtype=kv)
    out, lse, _ = run_gpu(prob)
    toks = [0, q - 1]
    o_ref, l_ref = oracle_rows(prob, toks)
    assert_close(out[toks], lse[toks], o_ref, l_ref)


@pytest.mark.parametrize("kv", [BF16, FP8])
def test_full_size_h12_1m_sampled(kv):
    prob = inputs.workload_long(kv)
    out, lse, _ = run_gpu(prob)
    toks = [0, 7]
    o_ref, l_ref = oracle_rows(prob, toks)
    assert_close(out[toks], lse[toks], o_ref, l_ref)


def test_closed_form_golden_fixture_gpu():
    """The hand-worked call of tests/golden/closed_form_h1_q2_ctx3.json through the C ABI:
    its page stored as physical page 1 of two, NaN in every other cache row."""
    from mla_speculative_verify_gb300.decoder import VerifyDecoder
    from tests import golden_fixture
    g = golden_fixture.load("closed_form_h1_q2_ctx3.json", page_size=64, page_order=[1])
    dec = VerifyDecoder(g["seq_lens"], g["q_lens"], g["H"], "bf16", "cuda")
    out = torch.full((2, 1, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((2, 1), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dec.run(g["q"].cuda(), g["kv"].cuda(), torch.from_numpy(g["page_table"]).cuda(), out, lse,
            g["sm_scale"], 1.0, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out.float().cpu().numpy(), lse.cpu().numpy(), g["out"], g["lse"])


@pytest.mark.parametrize("q,ctx,kv", [(8, 131072, BF16), (8, 131072, FP8), (1, 131072, BF16), (1, 32768, FP8)])
def test_full_size_h96_sampled(q, ctx, kv):
    """H = 96 (fold F = 1: every token is a group of its own) at the full context, in
    the plan the library makes for it; the first and last verify tokens against the
    oracle."""
    prob = inputs.workload_h96(q, ctx, kv)
    out, lse, _ = run_gpu(prob)
    toks = sorted({0, q - 1})
    o_ref, l_ref = oracle_rows(prob, toks)
    assert_close(out[toks], lse[toks], o_ref, l_ref)


@pytest.mark.parametrize("H", [48, 128])
@pytest.mark.parametrize("pattern", ["ragged", "uniform"])
def test_full_size_ragged_batch_sampled(H, pattern):
    """The B = 32 fp8 batches at their full contexts (16k-32k keys per request), in the
    plan the library makes for the whole batch (its piece lengths and merge layout);
    three requests (first, middle, last) against the oracle, each on its own."""
    prob = inputs.workload_ragged(H, pattern)
    out, lse, _ = run_gpu(prob)
    for b in (0, prob.batch // 2, prob.batch - 1):
        o_ref, l_ref = run_oracle(sub_problem(prob, b))
        rows = token_rows(prob, b)
        assert_close(out[rows], lse[rows], o_ref, l_ref)


def test_bad_page_id_is_reported_not_faulted():
    """A page id outside [0, num_pages) (one too large, one negative) in one request's
    page table: the kernel reports MLA_DEVICE_BAD_PAGE, reads page 0 in its place (in
    bounds), and the other request's output still matches the oracle."""
    from mla_speculative_verify_gb300.binding import MLA_DEVICE_BAD_PAGE

    prob = inputs.make_problem(12, [700, 900], [2, 4], BF16, seed=2950)
    prob.page_table = prob.page_table.copy()
    prob.page_table[0, 3] = prob.num_pages + 5
    prob.page_table[0, 7] = -1
    out, lse, st = run_gpu(prob, check_status=False)
    assert st & MLA_DEVICE_BAD_PAGE
    o_ref, l_ref = run_oracle(sub_problem(prob, 1))
    rows = token_rows(prob, 1)
    assert_close(out[rows], lse[rows], o_ref, l_ref)
    # the context stays usable
    good = inputs.make_problem(12, [700], [2], BF16, seed=2951)
    o2, l2, st2 = run_gpu(good)
    assert st2 == 0
    o_ref2, l_ref2 = run_oracle(good)
    assert_close(o2, l2, o_ref2, l_ref2)


@pytest.mark.parametrize("kv", [BF16, FP8])
def test_wait_timeout_is_reported_not_hung(kv):
    """The device timeout path, made to run without any fault or hang: a plan whose
    test-only option makes the first work unit never issue the copy of its page 2 and
    shortens every bounded wait to ~2 ms. The warps that wait for that page give up, the
    unit stops (in-flight copies drained, MMAs retired, tensor memory freed), the call
    reports MLA_DEVICE_WAIT_TIMEOUT, and the next call on the same context is exact."""
    from mla_speculative_verify_gb300.binding import MLA_DEVICE_WAIT_TIMEOUT

    prob = inputs.make_problem(12, [64 * 40 + 7], [4], kv, seed=2980)
    out, lse, st = run_gpu(prob, PlanOptions(force_splits=4, debug_skip_copy=3), check_status=False)
    assert st & MLA_DEVICE_WAIT_TIMEOUT
    o2, l2, st2 = run_gpu(prob)
    assert st2 == 0
    o_ref, l_ref = run_oracle(prob)
    assert_close(o2, l2, o_ref, l_ref)


@pytest.mark.parametrize("H,q,ctx,kv", [(96, 64, 3000, BF16), (12, 512, 4000, FP8), (12, 2048, 3100, BF16)])
def test_long_q_prefill_reduced_ctx(H, q, ctx, kv):
    """Long verify / prefill chunks through the same kernel: q in {64, 512, 2048} tokens
    (fold F = largest divisor of q with H F <= 128: 1 for H = 96, 8 for H = 12), every
    token with its own causal key range (the earliest of the 2048 sees ctx - 2047 keys),
    whole call against the oracle."""
    _check(inputs.make_problem(H, [ctx], [q], kv, seed=3100 + q, poison_tail=True))


@pytest.mark.parametrize("H,kv", [(12, BF16), (12, FP8), (96, BF16)])
def test_full_size_prefill_sampled(H, kv):
    """The prefill workload at its full size (q = 2048 tokens against ctx = 131072, the
    earliest token seeing 129025 keys): sampled tokens at the first, an inner and the last
    position (inner fold groups and row tiles; for H = 12 token 777 is the second of its
    8-token fold group), each against the oracle over its causal key prefix."""
    prob = inputs.make_problem(H, [131072], [2048], kv, seed=1006)
    out, lse, _ = run_gpu(prob)
    toks = [0, 777, 2047]
    o_ref, l_ref = oracle_rows(prob, toks)
    assert_close(out[toks], lse[toks], o_ref, l_ref)
