"""Torch-facing convenience wrapper around the C entry points.

``VerifyDecoder`` plans once for a batch shape (seq_lens, q_lens, H, cache dtype),
keeps the plan bytes on the device together with the split-KV workspace, and
enqueues ``mla_decode_run`` on torch device tensors. It only checks shapes,
dtypes and devices and passes raw pointers through; the decode itself runs in the
library's kernels.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import binding

KV_DTYPES = {"bf16": binding.MLA_KV_BF16, "fp8": binding.MLA_KV_FP8_E4M3}
SM_SCALE = 1.0 / math.sqrt(192.0)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


class VerifyDecoder:
    def __init__(self, seq_lens, q_lens, num_heads: int, kv_dtype: str, device="cuda", num_sms: int | None = None,
                 options: binding.PlanOptions | None = None):
        self.device = torch.device(device)
        if self.device.type == "cuda" and self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        if kv_dtype not in KV_DTYPES:
            raise ValueError(f"kv_dtype must be one of {list(KV_DTYPES)}")
        self.kv_dtype = kv_dtype
        self.num_heads = int(num_heads)
        self.seq_lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
        self.q_lens = np.ascontiguousarray(np.asarray(q_lens, dtype=np.int32))
        if num_sms is None:
            num_sms = torch.cuda.get_device_properties(self.device).multi_processor_count
        self.num_sms = int(num_sms)
        if self.device.type == "cuda":
            # clusters of two CTAs the device runs at once, for plans that use them
            opts = binding.PlanOptions() if options is None else options
            if opts.pair_slots == 0 and kv_dtype == "bf16":
                opts = binding.PlanOptions.from_buffer_copy(opts)
                opts.pair_slots = binding.device_pair_slots(self.device.index)
            options = opts
        self.plan_host, self.workspace_bytes = binding.plan(self.seq_lens, self.q_lens, self.num_heads,
                                                            KV_DTYPES[kv_dtype], self.num_sms, options)
        self.info = binding.plan_info(self.plan_host)
        # the plan runs on clusters of two CTAs (PlanHeader.cta_pair, the int32 at byte 64)
        self.cta_pair = bool(int(self.plan_host[64:68].view(np.int32)[0]))
        self.plan_dev = torch.from_numpy(self.plan_host).to(self.device)
        self.workspace = (torch.empty(self.workspace_bytes, dtype=torch.uint8, device=self.device)
                          if self.workspace_bytes else None)
        self.seq_lens_dev = torch.from_numpy(self.seq_lens).to(self.device)
        self.q_lens_dev = torch.from_numpy(self.q_lens).to(self.device)
        self.total_q = int(self.q_lens.sum())

    def run(self, q: torch.Tensor, kv_cache: torch.Tensor, page_table: torch.Tensor, out: torch.Tensor,
            lse: torch.Tensor | None = None, sm_scale: float = SM_SCALE, kv_scale: float = 1.0,
            status: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None,
            seq_lens_dev: torch.Tensor | None = None, q_lens_dev: torch.Tensor | None = None) -> None:
        H = self.num_heads
        want_kv = torch.bfloat16 if self.kv_dtype == "bf16" else torch.uint8
        if q.dtype != torch.bfloat16 or tuple(q.shape) != (self.total_q, H, 576) or not q.is_contiguous():
            raise ValueError(f"q must be a contiguous bf16 tensor of shape {(self.total_q, H, 576)}")
        if kv_cache.dtype not in (want_kv, torch.float8_e4m3fn) or kv_cache.shape[-1] != 576 or not kv_cache.is_contiguous():
            raise ValueError(f"kv_cache must be contiguous {want_kv} [..., 576]")
        if self.kv_dtype == "bf16" and kv_cache.dtype != torch.bfloat16:
            raise ValueError("a bf16 plan needs a bf16 cache")
        rows = kv_cache.numel() // 576
        if rows % 64:
            raise ValueError("kv_cache must hold whole 64-row pages")
        if out.dtype != torch.bfloat16 or tuple(out.shape) != (self.total_q, H, 512) or not out.is_contiguous():
            raise ValueError(f"out must be a contiguous bf16 tensor of shape {(self.total_q, H, 512)}")
        if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (self.total_q, H)):
            raise ValueError("lse must be float32 [total_q, H]")
        if page_table.dtype != torch.int32 or page_table.dim() != 2 or not page_table.is_contiguous():
            raise ValueError("page_table must be a contiguous int32 [batch, stride] tensor")
        for t in (q, kv_cache, out, page_table, lse, status):
            if t is not None and t.device != self.device:
                raise ValueError("all tensors must be on the decoder's device")
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        binding.run(self.plan_dev.data_ptr(), self.plan_host, q.data_ptr(), kv_cache.data_ptr(), page_table.data_ptr(),
                    page_table.shape[1], rows // 64,
                    (seq_lens_dev if seq_lens_dev is not None else self.seq_lens_dev).data_ptr(),
                    (q_lens_dev if q_lens_dev is not None else self.q_lens_dev).data_ptr(),
                    sm_scale, kv_scale, out.data_ptr(), _ptr(lse), _ptr(self.workspace), self.workspace_bytes,
                    _ptr(status), st.cuda_stream)
