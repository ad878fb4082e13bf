"""mla_decode_run_static_ws: the decode for callers that cannot allocate device memory
(plug-in hosts that hand over only the input and output buffers, code that must not let
an allocation synchronise the device, fixed memory plans). It takes its split-KV scratch
from a device array the library owns. This file is collected last on purpose: a failure
here leaves every other GPU test already run.

Checked through the C entry point against mla_decode_run with a caller workspace and
against the float64 oracle, on two calls in a row (the array keeps the previous call's
contents), within the tolerance of the parity tests; the device's free memory is the same
before and after the second call (the entry point allocates nothing); and a plan whose
scratch exceeds the array is rejected."""
import pytest
import torch

from mla_speculative_verify_gb300 import binding, inputs
from mla_speculative_verify_gb300.binding import PlanOptions
from mla_speculative_verify_gb300.decoder import VerifyDecoder
from tests.gpu_util import LSE_ATOL, OUT_ATOL, OUT_RTOL, assert_close, run_oracle

pytestmark = pytest.mark.gpu


def _call_static(dec, prob, q, kv, pt, out, lse, status):
    stream = torch.cuda.current_stream()
    binding.run_static_ws(dec.plan_dev.data_ptr(), dec.plan_host, q.data_ptr(), kv.data_ptr(), pt.data_ptr(),
                          pt.shape[1], kv.numel() // 576 // 64, dec.seq_lens_dev.data_ptr(), dec.q_lens_dev.data_ptr(),
                          prob.sm_scale, prob.kv_scale, out.data_ptr(), lse.data_ptr(), status.data_ptr(),
                          stream.cuda_stream)


@pytest.mark.parametrize("kv_dtype,seq,qlen,H", [(inputs.KV_BF16, 20000, 8, 12), (inputs.KV_FP8, 9000, 4, 48)])
def test_static_workspace_matches_caller_workspace(kv_dtype, seq, qlen, H):
    prob = inputs.make_problem(H, [seq], [qlen], kv_dtype, seed=4100 + qlen)
    dec = VerifyDecoder(prob.seq_lens, prob.q_lens, prob.H, prob.kv_dtype)
    assert 0 < dec.workspace_bytes <= binding.MLA_STATIC_WORKSPACE_BYTES
    q, kv, pt = prob.q.cuda(), prob.kv.cuda(), torch.from_numpy(prob.page_table).cuda()
    shape = (prob.total_q, prob.H)
    ref_out = torch.empty(shape + (512,), dtype=torch.bfloat16, device="cuda")
    ref_lse = torch.empty(shape, dtype=torch.float32, device="cuda")
    dec.run(q, kv, pt, ref_out, ref_lse, prob.sm_scale, prob.kv_scale)
    torch.cuda.synchronize()
    o_ref, l_ref = run_oracle(prob)
    for call in range(2):
        out = torch.full(shape + (512,), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        _call_static(dec, prob, q, kv, pt, out, lse, status)
        torch.cuda.synchronize()
        if call == 1:  # the first call may still load the library's module on this device
            assert torch.cuda.mem_get_info()[0] == free_before, "the static-workspace call allocated device memory"
        assert int(status.item()) == 0
        o, r = out.float(), ref_out.float()
        assert torch.isfinite(o).all()
        assert ((o - r).abs() <= OUT_ATOL + OUT_RTOL * r.abs()).all()
        assert (lse - ref_lse).abs().max().item() <= LSE_ATOL
        assert_close(o.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref)


def test_static_workspace_rejects_a_plan_larger_than_the_array():
    prob = inputs.make_problem(96, [2048], [8], inputs.KV_BF16, seed=4200)
    opts = PlanOptions(force_splits=32)  # 8 tokens x 96 rows x 32 splits partial rows
    dec = VerifyDecoder(prob.seq_lens, prob.q_lens, prob.H, prob.kv_dtype, options=opts)
    assert dec.workspace_bytes > binding.MLA_STATIC_WORKSPACE_BYTES
    q, kv, pt = prob.q.cuda(), prob.kv.cuda(), torch.from_numpy(prob.page_table).cuda()
    out = torch.empty((prob.total_q, prob.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((prob.total_q, prob.H), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.MlaError) as e:
        _call_static(dec, prob, q, kv, pt, out, lse, status)
    assert e.value.code == binding.MLA_ERR_BUFFER
