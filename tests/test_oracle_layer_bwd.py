"""Pins for the oracle's whole-layer backward (decode backward, expert MLP
backward, encode backward and gate backward composed).

Runs on the CPU only.  In fp32, central finite differences of the oracle's
own forward layer, L = <dy, y>, are compared with the composed backward for x,
the gate weight, the gate bias and the expert weights.  Only probes whose
perturbation leaves the routing (top-k indices and slots) unchanged are used:
routing is piecewise constant, so its derivative is zero there.
"""

import numpy as np
import pytest

import oracle
import synth
from synth.workloads import Workload

H = np.float32(2.0 ** -6)


def _loss(w, inp, dy):
    f = oracle.layer_forward(w, inp)
    return float((f["y"].astype(np.float64) * dy.astype(np.float64)).sum()), f


def _probes(rng, inp, w, n=4):
    names = ["x", "wg", "w1", "w2"] + (["w3"] if w.act == "swiglu" else ["b1", "b2"])
    if inp.get("bias") is not None:
        names.append("bias")
    out = []
    for name in names:
        shape = inp[name].shape
        for _ in range(n):
            out.append((name, tuple(int(rng.integers(0, d)) for d in shape)))
    return out


GRAD = {"x": "d_x", "wg": "d_wg", "bias": "d_gate_bias", "w1": "d_w1", "w2": "d_w2", "w3": "d_w3",
        "b1": "d_b1", "b2": "d_b2"}


@pytest.mark.parametrize("act,f,skew", [("gelu", 0.0, 0.0), ("gelu", 1.0, 1.0), ("swiglu", 1.25, 0.5)])
def test_layer_backward_matches_finite_differences(act, f, skew):
    w = Workload(name="lbwd", s=14, m=8, e=4, k=2, h=12, act=act, capacity_factor=f, dtype="f32",
                 skew_alpha=skew, seed=3)
    inp = synth.make_inputs_host(w, parts=("x", "wg", "bias", "w1", "w3", "w2", "b1", "b2"))
    dy = synth.normal_host(9, "dy", (w.s, w.m), 1.0, "f32")
    _, fwd = _loss(w, inp, dy)
    grads = oracle.layer_backward(w, inp, fwd, dy)
    rng = np.random.default_rng(17)
    checked = 0
    for name, ix in _probes(rng, inp, w):
        vals = {}
        for sgn in (1, -1):
            q = dict(inp)
            q[name] = inp[name].copy()
            q[name][ix] += sgn * H
            vals[sgn], fq = _loss(w, q, dy)
            if not (np.array_equal(fq["idx"], fwd["idx"]) and np.array_equal(fq["loc"], fwd["loc"])):
                break
        else:
            fd = (vals[1] - vals[-1]) / (2 * float(H))
            an = float(grads[GRAD[name]][ix])
            assert abs(an - fd) <= 2e-3 + 2e-3 * abs(fd), (name, ix, an, fd)
            checked += 1
    assert checked >= 12, checked


def test_identity_chain_through_the_copy_path():
    """With identity experts (out = buf) and the gates held fixed, the copy
    path's d_x is kappa_t dy_t, kappa_t = sum of the token's kept gates: the
    composed decode and encode backward without the gate path."""
    w = Workload(name="lbwd", s=20, m=8, e=4, k=2, h=8, act="relu", capacity_factor=0.75,
                 dtype="f32", seed=5)
    inp = synth.make_inputs_host(w, parts=("x", "wg", "bias"))
    lg = oracle.gate_logits(inp["x"], inp["wg"], inp["bias"])
    idx = oracle.topk(lg, w.k)
    g = oracle.gates(lg, idx, True)
    loc, need = oracle.locations(idx, w.e)
    c = oracle.capacity(w.capacity_factor, w.s, w.e, w.k, need)
    buf = oracle.encode(inp["x"], idx, loc, c, w.e, c)
    dy = synth.normal_host(2, "dy", (w.s, w.m), 1.0, "f32")
    d_out, _ = oracle.decode_bwd(dy, buf, idx, loc, g, c, False)
    dx = oracle.encode_bwd(d_out, idx, loc, c, False)
    kappa = np.where(loc < c, g, 0.0).sum(0)
    assert np.allclose(dx, kappa[:, None] * dy, rtol=1e-6, atol=1e-7)
    assert (loc >= c).any()                    # some routes were dropped
