"""GPU gate backward against the oracle (through the C ABI).

The device backward gets the oracle's own idx and gates, so only the backward
is compared.  Tolerances follow from the arithmetic: d_logits may differ by a
relative 2e-5 of the token's scale S_t = sum_r |dg g| + |A| (fp32 evaluation
from fp32 gates), 1e-4 for the raw softmax, whose logits the device recomputes
in another summation order (m * 2^-24 * sum |x w| stays below 1e-4 here); the
products add that error times their other factor plus n * 2^-24 * sum |terms|
for their own fp32 sums of n terms.
"""

import numpy as np
import pytest
import torch

import combine_moe_gate_gb300 as M
import oracle
import synth
from synth.workloads import Workload

from gpu_util import to_dev

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def _w(**kw):
    kw.setdefault("name", "gbwd")
    kw.setdefault("h", 64)
    kw.setdefault("act", "gelu")
    kw.setdefault("capacity_factor", 1.0)
    return Workload(**kw)


CASES = [
    (_w(s=300, m=136, e=8, k=2), True, "all"),
    (_w(s=257, m=264, e=32, k=4, skew_alpha=1.0), True, "all"),
    (_w(s=130, m=512, e=64, k=3, skew_alpha=1.2), True, "all"),
    (_w(s=256, m=64, e=4, k=1, dtype="f32", normalize_gates=False, skew_alpha=0.5), False, "all"),
    (_w(s=200, m=96, e=6, k=2, dtype="f32", normalize_gates=False), False, "all"),
    # several rounds of token groups, expert blocks with a 4-wide tail, a
    # partly filled last feature block
    (_w(s=2500, m=48, e=12, k=2), True, "all"),
    (_w(s=1100, m=36, e=20, k=3, dtype="f32", normalize_gates=False), False, "all"),
    # many ring stages per warp; wide expert counts (d_x in 4-token warp tiles)
    (_w(s=5000, m=200, e=64, k=4, skew_alpha=0.8), True, "all"),
    (_w(s=700, m=264, e=256, k=8), True, "all"),
    (_w(s=530, m=132, e=130, k=6, dtype="f32", normalize_gates=False), False, "all"),
    (_w(s=100, m=40, e=5, k=3), True, "logits_only"),
    (_w(s=100, m=40, e=5, k=3), True, "bias_only"),
]


@pytest.mark.parametrize("w,normalize,outs", CASES,
                         ids=lambda v: getattr(v, "name", str(v)) if not isinstance(v, Workload)
                         else f"s{v.s}_m{v.m}_e{v.e}_k{v.k}_{v.dtype}")
def test_gate_bwd_matches_oracle(w, normalize, outs):
    inp = synth.make_inputs_host(w, parts=("x", "wg", "bias"))
    x, wg, bias = inp["x"], inp["wg"], inp["bias"]
    lg = oracle.gate_logits(x, wg, bias)
    idx = oracle.topk(lg, w.k)
    g = oracle.gates(lg, idx, normalize)
    dg = synth.normal_host(7, "dg", (w.k, w.s), 1.0, "f32")
    ref = oracle.gate_bwd(x, wg, bias, idx, dg, normalize)

    s, m, e = w.s, w.m, w.e
    dev = lambda a: to_dev(a)
    z = lambda *shape: torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
    d_logits = z(s, e)
    d_wg = z(m, e) if outs == "all" else None
    d_bias = z(e) if outs in ("all", "bias_only") else None
    d_x = z(s, m) if outs == "all" else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    flags = M.MOE_FLAG_NORMALIZE_GATES if normalize else 0
    M.moe_gate_bwd(dev(x), dev(wg), None if bias is None else dev(bias), dev(idx), dev(g), dev(dg),
                   d_logits, st, d_wg=d_wg, d_bias=d_bias, d_x=d_x, flags=flags)
    torch.cuda.synchronize()
    assert int(st.item()) == 0

    xf = oracle.to_f32(x).astype(np.float64)
    w64 = wg.astype(np.float64)
    dl = ref["d_logits"]
    a = (dg.astype(np.float64) * g.astype(np.float64)).sum(0)                  # [s]
    scale = np.abs(dg.astype(np.float64) * g.astype(np.float64)).sum(0) + np.abs(a)
    rel = 2e-5 if normalize else 1e-4
    tol_dl = rel * scale + 1e-7                                                 # [s]

    got = d_logits.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - dl) <= tol_dl[:, None]), np.abs(got - dl).max()
    if d_wg is not None:
        tol = np.abs(xf).T @ tol_dl[:, None] + s * U * (np.abs(xf).T @ np.abs(dl))
        assert np.all(np.abs(d_wg.cpu().numpy() - ref["d_wg"]) <= tol)
    if d_bias is not None:
        tol = tol_dl.sum() + s * U * np.abs(dl).sum(0)
        assert np.all(np.abs(d_bias.cpu().numpy() - ref["d_bias"]) <= tol)
    if d_x is not None:
        tol = tol_dl[:, None] * np.abs(w64).sum(1)[None, :] + e * U * (np.abs(dl) @ np.abs(w64).T)
        assert np.all(np.abs(d_x.cpu().numpy() - ref["d_x"]) <= tol)


def _bwd_inputs(w, normalize):
    inp = synth.make_inputs_host(w, parts=("x", "wg", "bias"))
    lg = oracle.gate_logits(inp["x"], inp["wg"], inp["bias"])
    idx = oracle.topk(lg, w.k)
    g = oracle.gates(lg, idx, normalize)
    dg = synth.normal_host(7, "dg", (w.k, w.s), 1.0, "f32")
    return [to_dev(a) for a in (inp["x"], inp["wg"], inp["bias"], idx, g, dg)]


def _run_bwd(w, args, normalize, st):
    x, wg, bias, idx, g, dg = args
    out = [torch.full(sh, float("nan"), dtype=torch.float32, device="cuda")
           for sh in ((w.s, w.e), (w.m, w.e), (w.e,), (w.s, w.m))]
    M.moe_gate_bwd(x, wg, bias, idx, g, dg, out[0], st, d_wg=out[1], d_bias=out[2], d_x=out[3],
                   flags=M.MOE_FLAG_NORMALIZE_GATES if normalize else 0)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("w", [_w(s=8192, m=2048, e=16, k=3), _w(s=3000, m=520, e=256, k=8)],
                         ids=lambda w: f"s{w.s}_m{w.m}_e{w.e}")
def test_gate_bwd_is_deterministic(w):
    """The split sums (token slices, warps, cluster ranks) add in a fixed
    order: two calls give bit-identical outputs."""
    args = _bwd_inputs(w, True)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = _run_bwd(w, args, True, st)
    b = _run_bwd(w, args, True, st)
    assert int(st.item()) == 0
    for u, v in zip(a, b):
        assert torch.equal(u.view(torch.int32), v.view(torch.int32))


def test_gate_bwd_skips_after_error():
    """With the status word already set every kernel skips its stores."""
    w = _w(s=600, m=136, e=24, k=2)
    args = _bwd_inputs(w, True)
    st = torch.full((1,), 3, dtype=torch.int32, device="cuda")
    out = _run_bwd(w, args, True, st)
    assert int(st.item()) == 3
    for o in out:
        assert torch.isnan(o).all()
