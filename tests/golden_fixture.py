"""Builds the inputs and the expected result of a closed-form fixture under tests/golden/."""
import json
import os

import numpy as np
import torch

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str, page_size: int, page_order):
    """Inputs laid out with `page_size` keys per page; logical page p lives at physical page
    page_order[p] of a cache with len(page_order) + 1 pages. Cache rows that hold no key of
    the request are NaN. Returns a dict with q (bf16 [total_q, H, 576]), kv (bf16 rows x
    576), page_table (int32 [1, pages]), seq_lens, q_lens, H, sm_scale, and the expected
    out (float64 [total_q, H, 512]) and lse (float64 [total_q, H])."""
    d = json.load(open(os.path.join(HERE, name)))
    H, ctx, q = d["H"], d["seq_lens"][0], d["q_lens"][0]
    q_t = torch.zeros((q, H, 576), dtype=torch.float32)
    for tok, h, col, v in d["q_nonzero"]:
        q_t[tok, h, col] = v
    n_pages = len(page_order)
    assert n_pages * page_size >= ctx
    kv = torch.full(((n_pages + 1) * page_size, 576), float("nan"), dtype=torch.float32)
    for k in d["keys"]:
        j = k["key"]
        row = page_order[j // page_size] * page_size + j % page_size
        kv[row] = 0.0
        for col, v in k["cols"]:
            kv[row, col] = v
    out = np.zeros((q, H, 512))
    for tok, h, col, v in d["expected_out_nonzero"]:
        out[tok, h, col] = v
    lse = np.zeros((q, H))
    for tok, h, v in d["expected_lse"]:
        lse[tok, h] = v
    return dict(q=q_t.to(torch.bfloat16), kv=kv.to(torch.bfloat16),
                page_table=np.array([page_order], dtype=np.int32),
                seq_lens=np.array(d["seq_lens"], dtype=np.int32), q_lens=np.array(d["q_lens"], dtype=np.int32),
                H=H, sm_scale=d["sm_scale"], out=out, lse=lse)
