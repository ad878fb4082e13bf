"""Seeded synthetic inputs for MLA speculative-verify decode.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic. Both the CUDA path (through the tests and the benchmark)
and the float64 oracle consume the exact bytes it produces, so the two sides see
identical inputs.

Recipe (the workloads of the sglang PR #33650 isolated-kernel sweep and the
flashinfer PR #5588 / #5602 Kimi-K3 rows, with synthetic values standing in for
the model traces that are not available):
  * Q ~ N(0, 1) rounded to bf16, shape [sum(q_lens), H, 576].
  * Latent KV rows ~ N(0, 1): bf16, or fp8 e4m3 with one per-tensor scale
    kv_scale = amax / 448 and stored code = e4m3(x / kv_scale) (round to
    nearest even, saturating), shape [num_pages * 64, 576].
  * Page size 64. Pages are drawn from one shuffled global pool
    (torch.randperm); a "contiguous" layout uses the identity page table.
  * sm_scale = 1 / sqrt(192).
  * Cache rows past a request's seq_len inside its last page are filled with
    NaN when ``poison_tail`` is set, so a kernel that reads them shows it.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

D_QK = 576
D_V = 512
PAGE_SIZE = 64
FP8_MAX = 448.0
SM_SCALE = 1.0 / math.sqrt(192.0)

KV_BF16 = "bf16"
KV_FP8 = "fp8"


@dataclass
class Problem:
    """One batch of verify requests with its paged latent cache (host tensors)."""

    H: int
    seq_lens: np.ndarray          # int32 [B]
    q_lens: np.ndarray            # int32 [B]
    page_table: np.ndarray        # int32 [B, max_pages]
    q: torch.Tensor               # bf16 [sum q, H, 576]
    kv: torch.Tensor              # bf16 [rows, 576] or uint8 (e4m3 codes) [rows, 576]
    kv_dtype: str
    kv_scale: float
    sm_scale: float = SM_SCALE
    name: str = ""
    page_size: int = PAGE_SIZE
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.q_lens.sum())

    @property
    def num_pages(self) -> int:
        return int(self.kv.shape[0] // self.page_size)

    def q_bits(self) -> np.ndarray:
        """Q as uint16 bf16 bit patterns (what the oracle reads)."""
        return self.q.view(torch.int16).numpy().view(np.uint16)

    def kv_bits(self) -> np.ndarray:
        """KV as uint16 bf16 bits or uint8 e4m3 codes (what the oracle reads)."""
        if self.kv_dtype == KV_BF16:
            return self.kv.view(torch.int16).numpy().view(np.uint16)
        return self.kv.numpy()


def _randn(gen: torch.Generator, shape, chunk_rows: int = 1 << 18) -> torch.Tensor:
    """N(0,1) float32 drawn in row chunks (bounded temporary memory)."""
    out = torch.empty(shape, dtype=torch.float32)
    flat = out.view(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        flat[r0:r1] = torch.randn((r1 - r0, flat.shape[1]), generator=gen)
    return out


def quantize_e4m3(x: torch.Tensor) -> tuple[torch.Tensor, float]:
    """Per-tensor e4m3 quantisation: scale = amax / 448, codes = e4m3(x / scale)."""
    amax = float(x.abs().max())
    scale = amax / FP8_MAX if amax > 0 else 1.0
    codes = torch.empty(x.shape, dtype=torch.uint8)
    flat_x, flat_c = x.view(x.shape[0], -1), codes.view(x.shape[0], -1)
    step = 1 << 18
    for r0 in range(0, x.shape[0], step):
        r1 = min(x.shape[0], r0 + step)
        y = (flat_x[r0:r1] / scale).clamp_(-FP8_MAX, FP8_MAX)
        flat_c[r0:r1] = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale


def make_problem(H: int, seq_lens, q_lens, kv_dtype: str = KV_BF16, seed: int = 0,
                 contiguous: bool = False, poison_tail: bool = False, extra_pages: int = 0,
                 name: str = "", page_size: int = PAGE_SIZE) -> Problem:
    """Build a seeded problem. Pages of all requests come from one shuffled pool."""
    seq_lens = np.asarray(seq_lens, dtype=np.int32).reshape(-1)
    q_lens = np.asarray(q_lens, dtype=np.int32).reshape(-1)
    assert seq_lens.shape == q_lens.shape
    assert (q_lens >= 1).all() and (seq_lens >= q_lens).all()
    B = seq_lens.shape[0]
    gen = torch.Generator().manual_seed(int(seed))
    P = int(page_size)
    pages_per = (seq_lens + P - 1) // P
    pool = int(pages_per.sum()) + int(extra_pages)
    max_pages = max(1, int(pages_per.max()))
    total_q = int(q_lens.sum())
    q = _randn(gen, (total_q, H, D_QK)).to(torch.bfloat16)
    if contiguous:
        perm = torch.arange(pool, dtype=torch.int64)
    else:
        perm = torch.randperm(pool, generator=gen)
    page_table = np.zeros((B, max_pages), dtype=np.int32)
    o = 0
    for b in range(B):
        n = int(pages_per[b])
        page_table[b, :n] = perm[o:o + n].numpy().astype(np.int32)
        o += n
    x = _randn(gen, (pool * P, D_QK))
    if kv_dtype == KV_BF16:
        kv = x.to(torch.bfloat16)
        kv_scale = 1.0
    elif kv_dtype == KV_FP8:
        kv, kv_scale = quantize_e4m3(x)
    else:
        raise ValueError(kv_dtype)
    del x
    if poison_tail:
        for b in range(B):
            ctx = int(seq_lens[b])
            if ctx % P:
                page = int(page_table[b, ctx // P])
                r0, r1 = page * P + ctx % P, (page + 1) * P
                if kv_dtype == KV_BF16:
                    kv[r0:r1] = float("nan")
                else:
                    kv[r0:r1] = 0x7F  # e4m3 NaN code
    return Problem(H=H, seq_lens=seq_lens, q_lens=q_lens, page_table=page_table, q=q, kv=kv,
                   kv_dtype=kv_dtype, kv_scale=float(kv_scale), name=name, page_size=P)


# ----------------------------------------------------------------------------------------
# The five workload families (sizes as the sweep and the Kimi-K3 rows use them).
# ----------------------------------------------------------------------------------------

def workload_contiguous_small(seed: int = 1001) -> Problem:
    """B=1, H=12, q=2, ctx=4096, bf16, contiguous cache (identity page table)."""
    return make_problem(12, [4096], [2], KV_BF16, seed, contiguous=True, name="h12_q2_ctx4096_bf16_contig")


def workload_sweep_131k(q: int, ctx: int = 131072, seed: int = 1002, kv_dtype: str = KV_BF16) -> Problem:
    """B=1, H=12, q in {1,2,4,8}, ctx=131072, bf16 (or fp8 e4m3), random page table."""
    return make_problem(12, [ctx], [q], kv_dtype, seed, name=f"h12_q{q}_ctx{ctx}_{kv_dtype}")


def workload_long(kv_dtype: str, ctx: int = 1 << 20, q: int = 8, seed: int = 1003) -> Problem:
    """B=1, H=12, q=8, ctx=1,048,576, bf16 or fp8 e4m3, random page table."""
    return make_problem(12, [ctx], [q], kv_dtype, seed, name=f"h12_q{q}_ctx{ctx}_{kv_dtype}")


def workload_h96(q: int, ctx: int, kv_dtype: str, seed: int = 1004) -> Problem:
    """B=1, H=96 (fold F=1), q in {1,8}, ctx in {32768,131072}, bf16 or fp8."""
    return make_problem(96, [ctx], [q], kv_dtype, seed, name=f"h96_q{q}_ctx{ctx}_{kv_dtype}")


def ragged_lengths(pattern: str = "ragged", B: int = 32, ctx_lo: int = 16384, ctx_hi: int = 32768,
                   seed: int = 1005):
    """(seq_lens, q_lens) of the B=32 batch: ctx ~ U[ctx_lo, ctx_hi]; q from {1,2,3,4}
    (seeded MTP-3 pattern) or uniform 4. Both patterns share the context lengths (the same
    geometry, only q differs)."""
    seq_lens = np.random.default_rng(seed).integers(ctx_lo, ctx_hi + 1, size=B)
    if pattern == "ragged":
        q_lens = np.random.default_rng(seed + 1).integers(1, 5, size=B)
    elif pattern == "uniform":
        q_lens = np.full(B, 4)
    else:
        raise ValueError(pattern)
    return seq_lens, q_lens


def workload_ragged(H: int, pattern: str = "ragged", B: int = 32, ctx_lo: int = 16384,
                    ctx_hi: int = 32768, seed: int = 1005) -> Problem:
    """B=32 batch, H in {48,128}, the lengths of ragged_lengths, fp8 e4m3, shuffled global
    page pool."""
    seq_lens, q_lens = ragged_lengths(pattern, B, ctx_lo, ctx_hi, seed)
    return make_problem(H, seq_lens, q_lens, KV_FP8, seed, name=f"h{H}_b{B}_{pattern}_fp8")
