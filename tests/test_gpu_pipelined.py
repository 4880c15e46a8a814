"""The capacity-pipelined forward (moe_layer_forward_pipelined) against the
single pass (moe_layer_forward): encode of slot chunk i+1 on a side stream
overlaps the expert FFN of chunk i, and every output -- the encoded rows, the
expert FFN rows, the layer output -- must be bit-identical to the single pass,
because each row is computed by the same kernels in the same order.
"""

import numpy as np
import pytest
import torch

import combine_moe_gate_gb300 as M
import oracle
import synth
from synth import workloads as W
from synth.workloads import Workload

from gpu_util import status_ok

pytestmark = pytest.mark.gpu

CASES = [
    # the e=16 layer (PR #8195 shape) with c_max = c, so the chunks split the kept rows
    (W.BF16_E16_BWD, "c"),
    # small, ragged: 600 tokens, c_max above c
    (Workload(name="pipe_small", s=600, m=256, e=4, k=2, h=512, act="gelu", capacity_factor=0.0), "bound"),
    # SwiGLU, capped capacity with skew
    (Workload(name="pipe_swiglu", s=1024, m=512, e=8, k=2, h=256, act="swiglu", capacity_factor=-1.5,
              skew_alpha=1.0), "bound"),
]


def _c(w, inp):
    x = inp["x"]
    xh = x.view(torch.int16).cpu().numpy().view(np.uint16)
    lg = oracle.gate_logits(xh, inp["wg"].cpu().numpy(),
                            None if inp["bias"] is None else inp["bias"].cpu().numpy())
    idx = oracle.topk(lg, w.k)
    _, need = oracle.locations(idx, w.e)
    return oracle.capacity(w.capacity_factor, w.s, w.e, w.k, need)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
@pytest.mark.parametrize("chunks", [1, 2, 3, 4, 8])
def test_pipelined_forward_is_bit_identical(case, chunks):
    w, cmax_mode = case
    inp = synth.make_inputs_device(w, "cuda")
    c_max = _c(w, inp) if cmax_mode == "c" else None
    norm = w.normalize_gates and w.k >= 2
    flags = M.MOE_FLAG_NORMALIZE_GATES if norm else 0
    args = (inp["x"], inp["wg"], inp["bias"], inp["w1"], inp["b1"], inp["w3"], inp["w2"], inp["b2"],
            w.act, w.k, w.capacity_factor, flags)
    ref = M.alloc_layer(w.s, w.m, w.e, w.k, w.h, w.act, w.capacity_factor, c_max=c_max)
    got = M.alloc_layer(w.s, w.m, w.e, w.k, w.h, w.act, w.capacity_factor, c_max=c_max)
    # stale contents must not matter: only kept rows are compared, and they are written
    got.buf.fill_(7.0)
    got.out.fill_(-3.0)
    M.moe_layer_forward(*args, ref.idx, ref.gates, ref.loc, ref.counts, ref.c_dev, ref.buf, ref.out,
                        ref.y, ref.workspace, ref.status)
    aux = torch.cuda.Stream()
    events = [torch.cuda.Event() for _ in range(chunks + 1)]
    M.moe_layer_forward_pipelined(*args, got.idx, got.gates, got.loc, got.counts, got.c_dev, got.buf,
                                  got.out, got.y, got.workspace, got.status, chunks, aux, events)
    torch.cuda.synchronize()
    status_ok(ref.status)
    status_ok(got.status)
    assert torch.equal(ref.idx, got.idx) and torch.equal(ref.loc, got.loc)
    assert torch.equal(ref.counts, got.counts) and torch.equal(ref.c_dev, got.c_dev)
    c = int(ref.c_dev.item())
    kept = torch.clamp(ref.counts, max=c).cpu().numpy()
    for j in range(w.e):
        r = int(kept[j])
        assert torch.equal(ref.buf[j, :r].view(torch.int16), got.buf[j, :r].view(torch.int16)), j
        assert torch.equal(ref.out[j, :r].view(torch.int16), got.out[j, :r].view(torch.int16)), j
    assert torch.equal(ref.y.view(torch.int16), got.y.view(torch.int16))
