"""Shared helpers of the GPU parity tests: run the library through its C entry points
on a seeded problem and compare element by element with the float64 oracle."""
import numpy as np
import torch

import oracle
from mla_speculative_verify_gb300 import inputs
from mla_speculative_verify_gb300.binding import PlanOptions
from mla_speculative_verify_gb300.decoder import VerifyDecoder

# tolerance of the benchmark spec: |dout| <= 2e-2 + 2e-2 |ref|, |dLSE| <= 1e-3
OUT_ATOL, OUT_RTOL, LSE_ATOL = 2e-2, 2e-2, 1e-3


def to_device(prob, device="cuda"):
    q = prob.q.to(device)
    kv = prob.kv.to(device)
    pt = torch.from_numpy(prob.page_table).to(device)
    return q, kv, pt


def run_gpu(prob, options: PlanOptions | None = None, device="cuda", decoder=None, tensors=None, check_status=True):
    dec = decoder or VerifyDecoder(prob.seq_lens, prob.q_lens, prob.H, prob.kv_dtype, device, options=options)
    q, kv, pt = tensors or to_device(prob, device)
    out = torch.full((prob.total_q, prob.H, 512), float("nan"), dtype=torch.bfloat16, device=device)
    lse = torch.full((prob.total_q, prob.H), float("nan"), dtype=torch.float32, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    dec.run(q, kv, pt, out, lse, prob.sm_scale, prob.kv_scale, status)
    torch.cuda.synchronize()
    st = int(status.item())
    if check_status:
        assert st == 0, f"device status {st:#x}"
    return out.float().cpu().numpy(), lse.cpu().numpy(), st


def run_oracle(prob, mode=oracle.MODE_SPLIT, chunks=None):
    kvd = oracle.KV_BF16 if prob.kv_dtype == inputs.KV_BF16 else oracle.KV_FP8_E4M3
    bounds = None
    if mode == oracle.MODE_SPLIT:
        bounds = []
        for ctx in prob.seq_lens:
            n = chunks or max(1, min(64, int(ctx) // 2048))
            bounds.append(sorted(set([int(ctx) * i // n for i in range(n + 1)])))
    return oracle.decode(prob.q_bits(), prob.kv_bits(), kvd, prob.kv_scale, prob.page_table, prob.page_size,
                         prob.seq_lens, prob.q_lens, prob.H, prob.sm_scale, mode=mode, split_bounds=bounds)


def assert_close(out, lse, o_ref, l_ref, rows=None):
    if rows is not None:
        out, lse = out[rows], lse[rows]
    assert np.isfinite(out).all(), "non-finite output"
    assert np.isfinite(lse).all(), "non-finite lse"
    err = np.abs(out - o_ref)
    bound = OUT_ATOL + OUT_RTOL * np.abs(o_ref)
    bad = err > bound
    assert not bad.any(), (f"{bad.sum()} of {bad.size} outputs outside tolerance; max err {err.max():.3g}; "
                           f"first at {np.argwhere(bad)[0].tolist()}")
    lerr = np.abs(lse - l_ref)
    assert lerr.max() <= LSE_ATOL, f"max |dLSE| {lerr.max():.3g}"
    return float(err.max()), float(lerr.max())


def oracle_rows(prob, tokens):
    """Oracle for selected verify tokens of a single-request problem, each one as a
    q=1 call over its causal key prefix (the causal-rule pin of the oracle tests)."""
    outs, lses = [], []
    ctx, q = int(prob.seq_lens[0]), int(prob.q_lens[0])
    for i in tokens:
        sub = inputs.Problem(H=prob.H, seq_lens=np.array([ctx - q + i + 1], np.int32), q_lens=np.array([1], np.int32),
                             page_table=prob.page_table, q=prob.q[i:i + 1].clone(), kv=prob.kv,
                             kv_dtype=prob.kv_dtype, kv_scale=prob.kv_scale, sm_scale=prob.sm_scale)
        o, l = run_oracle(sub, chunks=64)
        outs.append(o[0])
        lses.append(l[0])
    return np.stack(outs), np.stack(lses)


def sub_problem(prob, b: int, tokens=None):
    """Request b of a batch as a problem of its own (its Q rows, seq_len, page-table row;
    the cache is shared), optionally cut to its first `tokens` verify tokens with each
    token's causal key range kept (token i of a request with ctx keys and q tokens sees
    ctx - q + i + 1 keys)."""
    ctx, q = int(prob.seq_lens[b]), int(prob.q_lens[b])
    t = q if tokens is None else max(1, min(q, int(tokens)))
    tok0 = int(prob.q_lens[:b].sum())
    return inputs.Problem(H=prob.H, seq_lens=np.array([ctx - q + t], np.int32), q_lens=np.array([t], np.int32),
                          page_table=prob.page_table[b:b + 1], q=prob.q[tok0:tok0 + t].clone(), kv=prob.kv,
                          kv_dtype=prob.kv_dtype, kv_scale=prob.kv_scale, sm_scale=prob.sm_scale)


def token_rows(prob, b: int) -> slice:
    """Global token indices of request b (rows of out / lse)."""
    tok0 = int(prob.q_lens[:b].sum())
    return slice(tok0, tok0 + int(prob.q_lens[b]))
