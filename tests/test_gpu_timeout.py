"""The tensor-core GEMM's bounded waits, made to run out on purpose and
safely: with moe_debug_stall_gemms the next GEMM launch issues no operand
copies (nothing is ever loaded, so no copy is in flight), its MMA issuer's
wait on the first stage gives up after about a second, the launch records
MOE_ERR_TIMEOUT in the status word, drains and frees its tensor memory and
returns; the second GEMM of the call sees the status and writes nothing.  The
context stays usable: the next call computes the same bits as before."""

import time

import torch
import pytest

import combine_moe_gate_gb300 as M

from gpu_util import bits

pytestmark = pytest.mark.gpu


def _bf16(shape, scale, g):
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16).cuda()


def test_gemm_bounded_wait_runs_out_and_the_context_stays_usable():
    e, c_max, m, h, act = 2, 256, 256, 512, "gelu"
    g = torch.Generator().manual_seed(7)
    buf = _bf16((e, c_max, m), 1.0, g)
    w1, b1 = _bf16((e, h, m), m ** -0.5, g), _bf16((e, h), 0.1, g)
    w2, b2 = _bf16((e, m, h), h ** -0.5, g), _bf16((e, m), 0.1, g)
    counts = torch.tensor([200, 131], dtype=torch.int32, device="cuda")
    c_dev = torch.tensor([c_max], dtype=torch.int32, device="cuda")
    ws = torch.empty(M.moe_expert_ffn_workspace_size(M.MOE_BF16, act, e, c_max, m, h),
                     dtype=torch.uint8, device="cuda")

    def run(out):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        M.moe_expert_ffn(buf, counts, c_dev, w1, b1, None, w2, b2, act, ws, out, st)
        torch.cuda.synchronize()
        return int(st.item())

    ref = torch.zeros((e, c_max, m), dtype=torch.bfloat16, device="cuda")
    assert run(ref) == M.MOE_OK
    M.moe_debug_stall_gemms(1)
    try:
        stalled = torch.full((e, c_max, m), -5.0, dtype=torch.bfloat16, device="cuda")
        t0 = time.monotonic()
        code = run(stalled)
        dt = time.monotonic() - t0
    finally:
        M.moe_debug_stall_gemms(0)
    assert code == M.MOE_ERR_TIMEOUT, M.status_str(code)
    assert 0.5 < dt < 30.0, dt
    assert bool((stalled == -5.0).all())       # neither GEMM wrote an output row
    again = torch.zeros_like(ref)
    assert run(again) == M.MOE_OK
    assert (bits(again) == bits(ref)).all()
