"""GPU parity of the two-CTA (cluster) decode: with the cta_pair plan option, fold groups
of 49..96 packed rows with a bf16 cache run on pairs of CTAs that split each page's columns and exchange partial
scores and P^T through distributed shared memory. Element by element against the
float64 oracle, with the single-CTA path on the same inputs as a second witness."""
import numpy as np
import pytest
import torch

from mla_speculative_verify_gb300 import binding, inputs
from mla_speculative_verify_gb300.binding import PlanOptions
from mla_speculative_verify_gb300.decoder import VerifyDecoder
from tests.gpu_util import assert_close, run_gpu, run_oracle
from tests.plan_reader import read_plan

pytestmark = pytest.mark.gpu

BF16 = inputs.KV_BF16


PAIR = PlanOptions(cta_pair=1)


def _is_pair(prob, options=PAIR):
    dec = VerifyDecoder(prob.seq_lens, prob.q_lens, prob.H, prob.kv_dtype, options=options)
    return read_plan(dec.plan_host)["header"]["cta_pair"] == 1


@pytest.mark.parametrize("H,q,ctx", [(12, 8, 64), (12, 8, 65), (12, 8, 200), (12, 8, 3000 + 7), (96, 1, 1000 + 3),
                                     (80, 1, 700), (50, 1, 700), (16, 6, 900), (7, 10, 1300), (12, 64, 2000)])
def test_pair_against_oracle(H, q, ctx):
    """Row counts 96, 80 (the second CTA owns 32 rows), 50 (2 rows), 70; one page, one key
    past a page, ragged tails (NaN in unused cache slots); eight fold groups per request."""
    prob = inputs.make_problem(H, [ctx], [q], BF16, seed=3000 + H + q + ctx, poison_tail=True)
    assert _is_pair(prob)
    out, lse, _ = run_gpu(prob, PAIR)
    o_ref, l_ref = run_oracle(prob)
    assert_close(out, lse, o_ref, l_ref)
    # the single-CTA path on the same inputs
    o2, l2, _ = run_gpu(prob, None)
    assert_close(o2, l2, o_ref, l_ref)


@pytest.mark.parametrize("splits", [1, 2, 5, 17])
def test_pair_splits_and_merge(splits):
    prob = inputs.make_problem(12, [64 * 40 + 11], [8], BF16, seed=3100 + splits, poison_tail=True)
    out, lse, _ = run_gpu(prob, PlanOptions(cta_pair=1, force_splits=splits))
    o_ref, l_ref = run_oracle(prob)
    assert_close(out, lse, o_ref, l_ref)


def test_pair_batch_of_requests():
    """Two requests of 96-row groups with different contexts and one of eight groups."""
    prob = inputs.make_problem(12, [3000, 5000, 2500], [8, 8, 16], BF16, seed=3200, poison_tail=True)
    assert _is_pair(prob)
    out, lse, _ = run_gpu(prob, PAIR)
    o_ref, l_ref = run_oracle(prob)
    assert_close(out, lse, o_ref, l_ref)


def test_pair_unsplit_rows_are_bitwise_reproducible():
    prob = inputs.make_problem(12, [3000], [8], BF16, seed=3300)
    opts = PlanOptions(cta_pair=1, force_splits=1)
    a = run_gpu(prob, opts)
    b = run_gpu(prob, opts)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_pair_large_score_range_moves_references():
    """Scores spread over tens of octaves force reference moves in both CTAs of the pair,
    in many tiles (each CTA rescales its value columns of the other CTA's rows too). Only
    the rope columns of the keys are scaled, by 1 .. 33 across the cache rows, so the
    values, and the output's size, stay as drawn."""
    prob = inputs.make_problem(12, [64 * 20 + 5], [8], BF16, seed=3400)
    k = prob.kv.float()
    pos = torch.arange(k.shape[0], dtype=torch.float32)
    k[:, 512:] *= 1.0 + (pos[:, None] % 1300) / 40.0
    prob.kv = k.to(prob.kv.dtype)
    o_ref, l_ref = run_oracle(prob)
    out, lse, _ = run_gpu(prob, PAIR)
    assert_close(out, lse, o_ref, l_ref)
    o2, l2, _ = run_gpu(prob, None)
    assert_close(o2, l2, o_ref, l_ref)


def test_device_reports_pair_slots():
    n = binding.device_pair_slots(0)
    assert 1 <= n <= 76


def test_pair_wait_timeout_is_reported_not_hung():
    """The test-only plan option on a two-CTA plan: CTA 0 of the first cluster never
    issues the copy of its page 2 and every bounded wait shrinks to ~2 ms. Its own waits
    give up first; the other CTA of the pair gives up waiting for partial sums that never
    come; both stop at a tile boundary, drain their copies and MMAs, meet at the final
    cluster barrier and free tensor memory. The call reports MLA_DEVICE_WAIT_TIMEOUT and
    the next call on the same context is exact."""
    from mla_speculative_verify_gb300.binding import MLA_DEVICE_WAIT_TIMEOUT

    prob = inputs.make_problem(12, [64 * 40 + 7], [8], BF16, seed=3500)
    assert _is_pair(prob, PlanOptions(cta_pair=1, force_splits=4, debug_skip_copy=3))
    out, lse, st = run_gpu(prob, PlanOptions(cta_pair=1, force_splits=4, debug_skip_copy=3), check_status=False)
    assert st & MLA_DEVICE_WAIT_TIMEOUT
    o2, l2, st2 = run_gpu(prob, PAIR)
    assert st2 == 0
    o_ref, l_ref = run_oracle(prob)
    assert_close(o2, l2, o_ref, l_ref)
