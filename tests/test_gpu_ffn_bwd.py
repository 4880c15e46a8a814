"""GPU expert-FFN backward against the oracle (through the C ABI).

The forward runs on the device first (its workspace is the hidden the
backward reads); the oracle's backward takes the same buf, weights and d_out.

Tolerance, from the arithmetic: the device rounds the recomputed
pre-activation, d_hid and d_pre to bf16 between its fp32-accumulated products
(relative 2^-9 each), evaluates the activation derivative at the rounded
pre-activation (|act''| <= 0.8 for GELU; SiLU's terms bounded likewise), reads
the hidden its own forward rounded, and rounds every output to bf16 once.  So
each d_pre (d_a, d_b) element may be off by E = 2^-7 (|d_pre| + |d_hid| |pre|)
(SwiGLU: 2^-7 |d_hid| |b| (1 + |a|) and 2^-7 |d_hid| |a|), and an output
built from it by at most the same product taken over E and absolute values,
plus half a bf16 step of the value; d_w2 by 2^-8 of |d_out|^T |hid|.  The
intermediates are evaluated in fp64 from the same inputs for this bound only;
the expected values are the oracle's.
"""

import numpy as np
import pytest
import torch

import combine_moe_gate_gb300 as M
import oracle
import synth
from synth.workloads import Workload

from gpu_util import to_dev, to_host

pytestmark = pytest.mark.gpu


def _w(**kw):
    kw.setdefault("name", "ffnbwd")
    return Workload(**kw)


CASES = [
    _w(s=300, m=64, e=3, k=2, h=128, act="gelu", capacity_factor=0.0),
    _w(s=333, m=128, e=4, k=2, h=256, act="relu", capacity_factor=1.25),
    _w(s=300, m=192, e=5, k=2, h=320, act="swiglu", capacity_factor=0.0, skew_alpha=1.0),
    _w(s=600, m=200, e=3, k=2, h=136, act="gelu", capacity_factor=0.0),
    # the e=16 layer's expert shape (m=2048, h=4096, GELU): every product
    # spans many 256 x 512 tiles and 64-deep K blocks, and the skew makes the
    # experts' kept rows (the weight gradients' contraction) ragged: ~160 to
    # ~600 rows, i.e. 3 to 10 K blocks, each ending in a partial block
    _w(s=1024, m=2048, e=8, k=3, h=4096, act="gelu", capacity_factor=0.0, skew_alpha=0.5),
]


try:
    from scipy.special import erf as _erf
except ImportError:  # pragma: no cover
    import math

    _erf = np.vectorize(math.erf)


def _f64(a):
    return oracle.to_f32(a).astype(np.float64)


@pytest.mark.parametrize("saved", [False, True, "f32"], ids=["recompute", "saved_pre", "saved_pre_f32"])
@pytest.mark.parametrize("w", CASES, ids=lambda w: f"e{w.e}_m{w.m}_h{w.h}_{w.act}")
def test_expert_ffn_bwd_matches_oracle(w, saved):
    """saved: the forward is moe_expert_ffn_train (its out and hidden must be
    the plain forward's bit for bit, its kept pre-activation -- SwiGLU: a and
    b -- within one bf16 rounding of the fp64 one) and the backward
    moe_expert_ffn_bwd_saved; "f32": with the weight and bias gradients
    stored in fp32."""
    inp = synth.make_inputs_host(w)
    # routing and the encoded buffer (the forward's expert rows are not needed)
    ref = oracle.layer_forward(w, inp, rows=(np.zeros(1, np.int32), np.zeros(1, np.int64)))
    c, e, m = ref["c"], w.e, w.m
    c_max = c + 3
    kept = ref["kept"].astype(np.int64)
    # rows past each expert's kept rows hold large values: none may reach a gradient
    buf_h = synth.bf16_bits_to_f32(synth.normal_host(6, "stale", (e, c_max, m), 50.0, "bf16"))
    for j in range(e):
        buf_h[j, :kept[j]] = ref["buf"][j, :kept[j]]
    d_out_h = synth.bf16_bits_to_f32(synth.normal_host(5, "d_out", (e, c_max, m), 1.0, "bf16"))
    _check_bwd(w, inp, buf_h, d_out_h, ref["needed"], kept, c, c_max, saved)


@pytest.mark.parametrize("act,saved,h", [("gelu", False, 320), ("swiglu", False, 320), ("relu", True, 320),
                                         ("swiglu", True, 320), ("swiglu", True, 200), ("gelu", True, 200)])
def test_expert_ffn_bwd_block_edges(act, saved, h):
    """Kept rows chosen at the weight gradients' 64-row block edges: exactly
    one block, none, a block plus a few rows, a single row, and a count above
    c (kept = c = 200, past three full blocks), with large values in every row
    past the kept ones."""
    w = _w(s=64, m=192, e=5, k=1, h=h, act=act, capacity_factor=0.0)   # h = 200: a partial 32-column box
    inp = synth.make_inputs_host(w)
    e, m = w.e, w.m
    needed = np.array([64, 0, 135, 1, 230], np.int32)
    c, c_max = 200, 208
    kept = np.minimum(needed, c).astype(np.int64)
    buf_h = synth.bf16_bits_to_f32(synth.normal_host(7, "buf_e", (e, c_max, m), 1.0, "bf16"))
    stale = synth.bf16_bits_to_f32(synth.normal_host(8, "stale_e", (e, c_max, m), 50.0, "bf16"))
    d_out_h = synth.bf16_bits_to_f32(synth.normal_host(9, "d_out_e", (e, c_max, m), 1.0, "bf16"))
    for j in range(e):
        buf_h[j, kept[j]:] = stale[j, kept[j]:]
    _check_bwd(w, inp, buf_h, d_out_h, needed, kept, c, c_max, saved)


def _check_bwd(w, inp, buf_h, d_out_h, needed, kept, c, c_max, saved=False):
    e, m, h = w.e, w.m, w.h
    swiglu = w.act == "swiglu"
    bf = torch.bfloat16
    buf = to_dev(buf_h).to(bf)
    counts = to_dev(np.asarray(needed).astype(np.int32))
    c_dev = to_dev(np.array([c], np.int32))
    w1, w3, w2 = to_dev(inp["w1"]), to_dev(inp["w3"]), to_dev(inp["w2"])
    b1, b2 = to_dev(inp["b1"]), to_dev(inp["b2"])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    # forward: its workspace holds the hidden the backward reads
    ws_f = torch.empty(M.moe_expert_ffn_workspace_size(M.MOE_BF16, w.act, e, c_max, m, h),
                       dtype=torch.uint8, device="cuda")
    out = torch.empty((e, c_max, m), dtype=bf, device="cuda")
    M.moe_expert_ffn(buf, counts, c_dev, w1, b1, w3, w2, b2, w.act, ws_f, out, st)
    hid = ws_f[: e * c_max * h * 2].view(bf).view(e, c_max, h)
    if saved:
        ws_t = torch.empty_like(ws_f)
        out_t = torch.empty_like(out)
        pre = torch.empty((e, c_max, 2 * h if swiglu else h), dtype=bf, device="cuda")
        M.moe_expert_ffn_train(buf, counts, c_dev, w1, b1, w3, w2, b2, w.act, ws_t, out_t, pre, st)
        torch.cuda.synchronize()
        hid_t = ws_t[: e * c_max * h * 2].view(bf).view(e, c_max, h)
        for j in range(e):
            r = int(kept[j])
            assert torch.equal(out_t[j, :r].view(torch.int16), out[j, :r].view(torch.int16)), j
            assert torch.equal(hid_t[j, :r].view(torch.int16), hid[j, :r].view(torch.int16)), j
            x = buf_h[j, :r].astype(np.float64)
            mats = [inp["w1"], inp["w3"]] if swiglu else [inp["w1"]]
            for q, wm in enumerate(mats):   # SwiGLU: a, then b
                pre64 = x @ _f64(wm)[j].T + (_f64(inp["b1"])[j] if inp["b1"] is not None else 0.0)
                got = to_host(pre[j, :r, q * h:(q + 1) * h]).astype(np.float64)
                # one bf16 rounding of the fp32-accumulated sum
                tol = (2.0 ** -8 * np.abs(pre64) + 2 * m * 2.0 ** -24 * (np.abs(x) @ np.abs(_f64(wm)[j].T))
                       + 1e-6)
                assert np.all(np.abs(got - pre64) <= tol), (j, q)
        hid = hid_t
    ws = torch.empty(M.moe_expert_ffn_bwd_workspace_size(M.MOE_BF16, w.act, e, c_max, m, h),
                     dtype=torch.uint8, device="cuda")
    d_buf = torch.full((e, c_max, m), 3.0, dtype=bf, device="cuda")
    gdt = torch.float32 if saved == "f32" else bf   # weight and bias gradients
    d_w1 = torch.empty((e, h, m), dtype=gdt, device="cuda")
    d_w3 = torch.empty((e, h, m), dtype=gdt, device="cuda") if swiglu else None
    d_w2 = torch.empty((e, m, h), dtype=gdt, device="cuda")
    d_b1 = None if swiglu else torch.empty((e, h), dtype=gdt, device="cuda")
    d_b2 = None if swiglu else torch.empty((e, m), dtype=gdt, device="cuda")
    if saved:
        M.moe_expert_ffn_bwd_saved(buf, hid, pre, counts, c_dev, w1, w3, w2, w.act,
                                   to_dev(d_out_h).to(bf), ws, d_buf, d_w1, d_w3, d_w2, d_b1, d_b2, st)
    else:
        M.moe_expert_ffn_bwd(buf, hid, counts, c_dev, w1, b1, w3, w2, w.act, to_dev(d_out_h).to(bf),
                             ws, d_buf, d_w1, d_w3, d_w2, d_b1, d_b2, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0

    want = oracle.ffn_bwd(buf_h, inp["w1"], inp["b1"], inp["w3"], inp["w2"], w.act, kept, d_out_h,
                          True)

    # error bounds (fp64 intermediates from the same inputs)
    W1, W2 = _f64(inp["w1"]), _f64(inp["w2"])
    W3 = _f64(inp["w3"]) if swiglu else None
    b1f = None if inp["b1"] is None else _f64(inp["b1"])
    u = 2.0 ** -7
    for j in range(e):
        r = int(kept[j])
        x = buf_h[j, :r].astype(np.float64)
        g = d_out_h[j, :r].astype(np.float64)
        dh = g @ W2[j]                                                   # [r, h]
        a = x @ W1[j].T
        if swiglu:
            b = x @ W3[j].T
            sg = 1.0 / (1.0 + np.exp(-a))
            hid_abs = np.abs(a * sg * b)
            ea = u * np.abs(dh) * np.abs(b) * (1.0 + np.abs(a))
            eb = u * np.abs(dh) * np.abs(a)
            e_buf = ea @ np.abs(W1[j]) + eb @ np.abs(W3[j])
        else:
            pre = a + (b1f[j] if b1f is not None else 0.0)
            if w.act == "relu":
                dact, hid_abs = (pre > 0).astype(np.float64), np.maximum(pre, 0.0)
            else:
                cdf = 0.5 * (1.0 + _erf(pre / np.sqrt(2.0)))
                dact = cdf + pre * np.exp(-0.5 * pre * pre) / np.sqrt(2.0 * np.pi)
                hid_abs = np.abs(pre * cdf)
            ea = u * (np.abs(dh * dact) + np.abs(dh) * np.abs(pre))
            e_buf = ea @ np.abs(W1[j])

        def check(got, ref_v, err, name):
            tol = 1.5 * err + 2.0 ** -8 * np.abs(ref_v) + 1e-6
            assert np.all(np.abs(got - ref_v) <= tol), (name, j, np.abs(got - ref_v).max())

        check(to_host(d_buf)[j, :r], want["d_buf"][j, :r], e_buf, "d_buf")
        check(to_host(d_w1)[j], want["d_w1"][j], ea.T @ np.abs(x), "d_w1")
        check(to_host(d_w2)[j], want["d_w2"][j], 2.0 ** -8 * (np.abs(g).T @ hid_abs), "d_w2")
        if swiglu:
            check(to_host(d_w3)[j], want["d_w3"][j], eb.T @ np.abs(x), "d_w3")
        else:
            check(to_host(d_b1)[j], want["d_b1"][j], ea.sum(0), "d_b1")
            check(to_host(d_b2)[j], want["d_b2"][j], 2.0 ** -9 * np.abs(g).sum(0), "d_b2")
        assert np.all(to_host(d_buf)[j, r:] == 3.0)        # rows past the kept count untouched
