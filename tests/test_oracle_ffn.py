"""Pins for the oracle's expert FFN: special cases that reduce to a dense MLP
(a library matmul), activation closed forms, and the whole-layer chain."""

import math

import numpy as np
import pytest
import torch

import oracle
import synth


def _torch_mlp(x, w1, b1, w3, w2, b2, act, bf16):
    """Dense MLP with torch fp64 matmuls; the hidden activation is rounded to the
    layer dtype the same way (fp64 -> bf16 through oracle.round_bf16)."""
    X, W1, W2 = (torch.from_numpy(oracle.to_f32(a)).double() for a in (x, w1, w2))
    a = X @ W1.T
    if act == "swiglu":
        b = X @ torch.from_numpy(oracle.to_f32(w3)).double().T
        hid = a / (1 + torch.exp(-a)) * b
    else:
        if b1 is not None:
            a = a + torch.from_numpy(oracle.to_f32(b1)).double()
        hid = torch.relu(a) if act == "relu" else 0.5 * a * (1 + torch.erf(a / math.sqrt(2)))
    hid = hid.numpy()
    hid = np.vectorize(oracle.round_bf16)(hid) if bf16 else hid.astype(np.float32)
    o = torch.from_numpy(hid.astype(np.float64)) @ W2.T
    if b2 is not None and act != "swiglu":
        o = o + torch.from_numpy(oracle.to_f32(b2)).double()
    o = o.numpy()
    return np.vectorize(oracle.round_bf16)(o) if bf16 else o.astype(np.float32)


@pytest.mark.parametrize("act,dt", [("relu", "f32"), ("gelu", "bf16"), ("swiglu", "bf16"),
                                    ("gelu", "f32")])
def test_single_expert_is_dense_mlp(act, dt):
    """e=1, k=1, f=0 routes every token to the one expert in order: the FFN over
    the buffer is a plain dense MLP over x."""
    w = synth.Workload(name="t", s=24, m=16, e=1, k=1, h=40, act=act, capacity_factor=0.0,
                       dtype=dt, normalize_gates=False)
    inp = synth.make_inputs_host(w)
    res = oracle.layer_forward(w, inp)
    assert res["c"] == w.s and np.array_equal(res["loc"][0], np.arange(w.s))
    first = lambda a: None if a is None else a[0]
    want = _torch_mlp(inp["x"], inp["w1"][0], first(inp["b1"]), first(inp["w3"]), inp["w2"][0],
                      first(inp["b2"]), act, dt == "bf16")
    got = res["out"][0]
    if dt == "bf16":
        # fp64 sums in a different association can move a bf16 rounding by one step
        assert np.mean(got == want) > 0.98
        np.testing.assert_allclose(got, want, rtol=2 ** -7, atol=1e-3)
    else:
        np.testing.assert_allclose(got, want, rtol=1e-6, atol=1e-6)
    # k=1 without renormalisation: y = p_top * MLP(x) (the only expert has p = 1)
    np.testing.assert_array_equal(res["gates"], np.ones((1, w.s), np.float32))
    np.testing.assert_array_equal(res["y"], got)


@pytest.mark.parametrize("act,xv,want", [
    ("gelu", 1.0, 0.8413447460685429),     # Phi(1)
    ("gelu", -1.0, -0.15865525393145707),  # -(1 - Phi(1))
    ("relu", -2.5, 0.0),
    ("relu", 2.5, 2.5),
    ("swiglu", 1.0, 0.7310585786300049),   # silu(1) * 1 = 1 / (1 + e^-1)
])
def test_activation_closed_forms(act, xv, want):
    buf = np.full((1, 1, 1), xv, np.float32)
    one = np.ones((1, 1, 1), np.float32)
    out = oracle.ffn_rows(buf, one, None, one if act == "swiglu" else None, one, None, act,
                          [0], [0], False)
    assert abs(out[0, 0] - np.float32(want)) <= 1e-7


def test_bias_and_layout():
    """Hand-built 2-expert case: hidden unit u of expert j reads row u of w1[j]
    (w1 is [e, h, m]); output i reads row i of w2[j] (w2 is [e, m, h])."""
    buf = np.array([[[1.0, 2.0]], [[3.0, -1.0]]], np.float32)         # e=2, cmax=1, m=2
    w1 = np.array([[[1, 0], [0, 1], [1, 1]], [[2, 0], [0, 0], [1, -1]]], np.float32)  # h=3
    b1 = np.array([[0, 0, -2.5], [0, 1, 0]], np.float32)
    w2 = np.array([[[1, 1, 1], [0, 0, 2]], [[1, 0, 0], [1, 1, 1]]], np.float32)
    b2 = np.array([[0.5, 0], [0, -1]], np.float32)
    out = oracle.ffn_rows(buf, w1, b1, None, w2, b2, "relu", [0, 1], [0, 0], False)
    # expert 0: a = [1, 2, 3-2.5=0.5] -> relu same; out = [1+2+0.5+0.5, 2*0.5] = [4, 1]
    # expert 1: a = [6, 0+1, 3+1=4] -> [6, 1, 4]; out = [6, 6+1+4-1] = [6, 10]
    np.testing.assert_array_equal(out, np.array([[4, 1], [6, 10]], np.float32))


def test_layer_forward_tiny_workload_runs():
    w = synth.workloads.TINY_FP32
    inp = synth.make_inputs_host(w)
    res = oracle.layer_forward(w, inp)
    assert res["c"] == 64
    assert res["y"].shape == (w.s, w.m)
    kept = res["loc"] < res["c"]
    # dropped tokens produce exactly zero output rows
    dropped = ~kept.any(0)
    assert np.all(res["y"][dropped] == 0)
    assert np.all(np.isfinite(res["y"]))
