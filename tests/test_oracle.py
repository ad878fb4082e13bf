"""Pins of the float64 oracle against things other than itself (CPU only).

The pages print no input/output values for this operation, so every pin is a
brute-force evaluation, a library routine, a closed form or an invariant:
  * brute force: numpy, the fully materialised masked score matrix;
  * library: torch float64 scaled_dot_product_attention (unmasked q=1, and an
    explicit bottom-right causal mask for q>1) and torch's float8_e4m3fn cast;
  * closed forms: constant value rows, identical key rows, and a hand-worked call
    (tests/golden/closed_form_h1_q2_ctx3.json) through a permuted paged layout;
  * invariants: the causal rule, fold == direct, split + merge == direct, and
    the kv_scale homogeneity of an fp8 cache.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from mla_speculative_verify_gb300 import inputs

RTOL, ATOL = 1e-11, 1e-12


def _f64_q(prob):
    return prob.q.to(torch.float64).numpy()


def _f64_kv(prob):
    if prob.kv_dtype == inputs.KV_BF16:
        return prob.kv.to(torch.float64).numpy()
    return prob.kv.view(torch.float8_e4m3fn).to(torch.float64).numpy() * prob.kv_scale


def brute_force(prob):
    """Materialise every masked score; numpy only, independent of the oracle."""
    qf, kvf = _f64_q(prob), _f64_kv(prob)
    P = prob.page_size
    outs, lses = [], []
    t0 = 0
    for b in range(prob.batch):
        ctx, q = int(prob.seq_lens[b]), int(prob.q_lens[b])
        rows = np.array([prob.page_table[b, j // P] * P + j % P for j in range(ctx)], dtype=np.int64)
        K = kvf[rows]                      # [ctx, 576]
        V = K[:, :512]
        Qb = qf[t0:t0 + q]                 # [q, H, 576]
        S = prob.sm_scale * np.einsum("ihd,jd->ihj", Qb, K)
        allowed = np.arange(ctx)[None, :] < (ctx - q + np.arange(q)[:, None] + 1)
        S = np.where(allowed[:, None, :], S, -np.inf)
        m = S.max(-1, keepdims=True)
        W = np.exp(S - m)
        l = W.sum(-1, keepdims=True)
        outs.append(np.einsum("ihj,jd->ihd", W, V) / l)
        lses.append((m + np.log(l))[..., 0])
        t0 += q
    return np.concatenate(outs), np.concatenate(lses)


def run_oracle(prob, mode=oracle.MODE_DIRECT, split_bounds=None, lib=None):
    kvd = oracle.KV_BF16 if prob.kv_dtype == inputs.KV_BF16 else oracle.KV_FP8_E4M3
    return oracle.decode(prob.q_bits(), prob.kv_bits(), kvd, prob.kv_scale, prob.page_table,
                         prob.page_size, prob.seq_lens, prob.q_lens, prob.H, prob.sm_scale,
                         mode=mode, split_bounds=split_bounds, lib=lib)


def tiny_cases():
    return [
        inputs.make_problem(2, [5], [3], inputs.KV_BF16, seed=11, page_size=2),
        inputs.make_problem(3, [7, 4, 9], [1, 4, 2], inputs.KV_BF16, seed=12, page_size=2),
        inputs.make_problem(2, [6, 11], [2, 3], inputs.KV_FP8, seed=13, page_size=4),
        inputs.make_problem(5, [70, 130], [4, 1], inputs.KV_BF16, seed=14, page_size=64),
        inputs.make_problem(12, [200], [8], inputs.KV_FP8, seed=15, page_size=64),
    ]


@pytest.mark.parametrize("idx", range(5))
@pytest.mark.parametrize("mode", [oracle.MODE_DIRECT, oracle.MODE_FOLDED])
def test_brute_force(idx, mode):
    prob = tiny_cases()[idx]
    o_ref, l_ref = brute_force(prob)
    o, l = run_oracle(prob, mode)
    np.testing.assert_allclose(o, o_ref, rtol=RTOL, atol=ATOL)
    np.testing.assert_allclose(l, l_ref, rtol=RTOL, atol=ATOL)


def test_e4m3_decode_every_code():
    """All 256 codes against torch's float8_e4m3fn and a few hand values."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib_vals = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    nan = np.isnan(lib_vals)
    assert np.array_equal(nan, np.isnan(ours))
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(ours[~nan], lib_vals[~nan])
    assert ours[0x00] == 0.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6
    assert ours[0x38] == 1.0 and ours[0x7E] == 448.0 and ours[0xFE] == -448.0


def test_fold_factor_table():
    # F = largest divisor of q with H*F <= 128
    table = {(8, 12): 8, (4, 12): 4, (2, 12): 2, (1, 12): 1, (3, 48): 1, (4, 48): 2, (2, 48): 2,
             (2, 96): 1, (8, 96): 1, (1, 128): 1, (6, 20): 6, (7, 20): 1, (4, 200): 1, (12, 12): 6, (16, 12): 8, (10, 16): 5}
    for (q, H), F in table.items():
        assert oracle.fold_factor(q, H) == F, (q, H)


def test_sdpa_unmasked_q1():
    """q = 1: the plain softmax attention of torch's float64 SDPA (library routine)."""
    prob = inputs.make_problem(6, [300], [1], inputs.KV_BF16, seed=21)
    o, l = run_oracle(prob)
    Q = torch.from_numpy(_f64_q(prob))[None].transpose(1, 2)         # [1, H, 1, 576]
    rows = [prob.page_table[0, j // 64] * 64 + j % 64 for j in range(300)]
    K = torch.from_numpy(_f64_kv(prob)[rows])[None, None]             # [1, 1, ctx, 576]
    ref = torch.nn.functional.scaled_dot_product_attention(
        Q, K.expand(1, 6, -1, -1), K[..., :512].expand(1, 6, -1, -1), scale=prob.sm_scale)
    np.testing.assert_allclose(o, ref.transpose(1, 2)[0].numpy(), rtol=1e-10, atol=1e-12)
    lse_ref = torch.logsumexp(prob.sm_scale * (Q @ K.transpose(-1, -2)), -1)
    np.testing.assert_allclose(l, lse_ref[0, :, 0].numpy()[None], rtol=1e-12, atol=1e-12)


def test_sdpa_bottom_right_mask():
    """q > 1: SDPA with an explicit bottom-right causal boolean mask."""
    prob = inputs.make_problem(4, [129], [5], inputs.KV_FP8, seed=22)
    o, l = run_oracle(prob, oracle.MODE_FOLDED)
    ctx, q = 129, 5
    Q = torch.from_numpy(_f64_q(prob)).transpose(0, 1)[None]          # [1, H, q, 576]
    rows = [prob.page_table[0, j // 64] * 64 + j % 64 for j in range(ctx)]
    K = torch.from_numpy(_f64_kv(prob)[rows])[None, None].expand(1, 4, -1, -1)
    mask = torch.arange(ctx)[None, :] <= (ctx - q + torch.arange(q)[:, None])
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, K[..., :512], attn_mask=mask, scale=prob.sm_scale)
    np.testing.assert_allclose(o, ref[0].transpose(0, 1).numpy(), rtol=1e-10, atol=1e-12)


def test_causal_rows_match_shorter_q1_calls():
    """Row i of a q-token call equals a q=1 call over the first ctx-q+i+1 keys;
    the last row therefore sees every key."""
    prob = inputs.make_problem(3, [150], [6], inputs.KV_BF16, seed=23)
    o, l = run_oracle(prob, oracle.MODE_FOLDED)
    for i in range(6):
        sub = inputs.Problem(H=3, seq_lens=np.array([150 - 6 + i + 1], np.int32), q_lens=np.array([1], np.int32),
                             page_table=prob.page_table, q=prob.q[i:i + 1].clone(), kv=prob.kv,
                             kv_dtype=prob.kv_dtype, kv_scale=prob.kv_scale)
        o1, l1 = run_oracle(sub)
        np.testing.assert_allclose(o[i:i + 1], o1, rtol=RTOL, atol=ATOL)
        np.testing.assert_allclose(l[i:i + 1], l1, rtol=RTOL, atol=ATOL)


@pytest.mark.parametrize("seed", [31, 32, 33])
def test_split_merge_equals_direct(seed):
    """Random chunkings: 1-key chunks, empty chunks and chunks a causal row cannot see."""
    prob = inputs.make_problem(4, [97, 64, 33], [7, 3, 1], inputs.KV_BF16 if seed % 2 else inputs.KV_FP8,
                               seed=seed)
    rng = np.random.default_rng(seed)
    bounds = []
    for ctx in prob.seq_lens:
        cuts = sorted(set(rng.integers(0, ctx + 1, size=6).tolist()) | {0, int(ctx), int(ctx) - 1, int(ctx) - 2})
        cuts = [c for c in cuts if 0 <= c <= ctx]
        cuts.insert(2, cuts[1])          # an empty chunk
        bounds.append(cuts)
    o_d, l_d = run_oracle(prob)
    o_s, l_s = run_oracle(prob, oracle.MODE_SPLIT, bounds)
    np.testing.assert_allclose(o_s, o_d, rtol=RTOL, atol=ATOL)
    np.testing.assert_allclose(l_s, l_d, rtol=RTOL, atol=ATOL)


def test_fold_equals_direct_wide():
    prob = inputs.make_problem(48, [260, 200], [4, 3], inputs.KV_FP8, seed=41)
    o_d, l_d = run_oracle(prob)
    o_f, l_f = run_oracle(prob, oracle.MODE_FOLDED)
    np.testing.assert_allclose(o_f, o_d, rtol=RTOL, atol=ATOL)
    np.testing.assert_allclose(l_f, l_d, rtol=RTOL, atol=ATOL)


def test_constant_value_rows():
    """Every key row holds the same 512 value columns (rope columns random): O == v."""
    prob = inputs.make_problem(5, [90], [3], inputs.KV_BF16, seed=51)
    v = prob.kv[7, :512].clone()
    prob.kv[:, :512] = v
    for mode in (oracle.MODE_DIRECT, oracle.MODE_FOLDED):
        o, _ = run_oracle(prob, mode)
        np.testing.assert_allclose(o, np.broadcast_to(v.to(torch.float64).numpy(), o.shape), rtol=1e-13, atol=1e-13)


def test_identical_key_rows():
    """All keys equal: O = that row's value part, LSE = s + ln n with n visible keys."""
    prob = inputs.make_problem(2, [40], [4], inputs.KV_BF16, seed=52)
    prob.kv[:] = prob.kv[3].clone()
    o, l = run_oracle(prob)
    k = prob.kv[3].to(torch.float64).numpy()
    for i in range(4):
        n = 40 - 4 + i + 1
        for h in range(2):
            s = prob.sm_scale * float(prob.q[i, h].to(torch.float64).numpy() @ k)
            assert abs(l[i, h] - (s + math.log(n))) < 1e-12
            np.testing.assert_allclose(o[i, h], k[:512], rtol=1e-13, atol=1e-13)


def test_fp8_scale_homogeneity():
    """For an fp8 cache, kv_scale=c equals kv_scale=1 with sm_scale*c, O times c."""
    prob = inputs.make_problem(3, [77], [2], inputs.KV_FP8, seed=53)
    c = prob.kv_scale
    o, l = run_oracle(prob)
    prob1 = inputs.Problem(H=3, seq_lens=prob.seq_lens, q_lens=prob.q_lens, page_table=prob.page_table,
                           q=prob.q, kv=prob.kv, kv_dtype=prob.kv_dtype, kv_scale=1.0,
                           sm_scale=prob.sm_scale * c)
    o1, l1 = run_oracle(prob1)
    np.testing.assert_allclose(o, o1 * c, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l, l1, rtol=1e-12, atol=1e-12)


def test_rejects_bad_arguments():
    prob = inputs.make_problem(2, [10], [2], inputs.KV_BF16, seed=54, page_size=4)
    bad = inputs.Problem(H=2, seq_lens=np.array([1], np.int32), q_lens=np.array([2], np.int32),
                         page_table=prob.page_table, q=prob.q, kv=prob.kv, kv_dtype="bf16", kv_scale=1.0,
                         page_size=4)
    with pytest.raises(ValueError):
        run_oracle(bad)


@pytest.mark.parametrize("mode", [oracle.MODE_DIRECT, oracle.MODE_FOLDED, oracle.MODE_SPLIT])
def test_closed_form_golden_fixture(mode):
    """The hand-worked call of tests/golden/closed_form_h1_q2_ctx3.json: pages of two keys
    stored out of order, NaN in every cache row that holds no key of the request."""
    from tests import golden_fixture
    g = golden_fixture.load("closed_form_h1_q2_ctx3.json", page_size=2, page_order=[2, 0])
    bounds = [[0, 1, 3]] if mode == oracle.MODE_SPLIT else None
    out, lse = oracle.decode(g["q"].view(torch.int16).numpy().view(np.uint16),
                             g["kv"].view(torch.int16).numpy().view(np.uint16), oracle.KV_BF16, 1.0,
                             g["page_table"], 2, g["seq_lens"], g["q_lens"], g["H"], g["sm_scale"],
                             mode=mode, split_bounds=bounds)
    np.testing.assert_allclose(out, g["out"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, g["lse"], rtol=0, atol=1e-12)
