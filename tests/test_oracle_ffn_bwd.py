"""Pins for the oracle's expert-MLP backward.

Runs on the CPU only.  The backward is tied to torch autograd of the same MLP
in fp64 (a library routine, independent of the oracle's C loops), to central
finite differences of the oracle's own forward, and to properties any correct
backward has: rows past an expert's kept count do not matter, gradients are
linear in d_out, and experts are independent of one another.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _case(act, e=3, cmax=5, m=6, h=7, kept=(5, 2, 0), seed=0):
    rng = np.random.default_rng(seed)
    f = lambda *shape, sc=1.0: (rng.standard_normal(shape) * sc).astype(np.float32)
    buf = f(e, cmax, m)
    w1, w3 = f(e, h, m, sc=0.5), f(e, h, m, sc=0.5)
    w2 = f(e, m, h, sc=0.5)
    b1, b2 = f(e, h, sc=0.3), f(e, m, sc=0.3)
    d_out = f(e, cmax, m)
    if act == "swiglu":
        b1 = b2 = None
    else:
        w3 = None
    return dict(buf=buf, w1=w1, b1=b1, w3=w3, w2=w2, b2=b2, d_out=d_out,
                kept=np.array(kept, np.int64))


def _bwd(c, act, bf16=False, d_out=None):
    return oracle.ffn_bwd(c["buf"], c["w1"], c["b1"], c["w3"], c["w2"], act, c["kept"],
                          c["d_out"] if d_out is None else d_out, bf16)


@pytest.mark.parametrize("act", ["relu", "gelu", "swiglu"])
def test_matches_torch_autograd_fp64(act):
    c = _case(act)
    got = _bwd(c, act)
    t = lambda a: None if a is None else torch.tensor(a, dtype=torch.float64, requires_grad=True)
    for ex in range(len(c["kept"])):
        r = int(c["kept"][ex])
        x = t(c["buf"][ex, :r])
        w1, w2 = t(c["w1"][ex]), t(c["w2"][ex])
        if act == "swiglu":
            w3 = t(c["w3"][ex])
            hid = F.silu(x @ w1.T) * (x @ w3.T)
            out = hid @ w2.T
        else:
            b1, b2 = t(c["b1"][ex]), t(c["b2"][ex])
            pre = x @ w1.T + b1
            hid = F.relu(pre) if act == "relu" else F.gelu(pre, approximate="none")
            out = hid @ w2.T + b2
        loss = (out * torch.tensor(c["d_out"][ex, :r], dtype=torch.float64)).sum()
        loss.backward()
        # the oracle feeds fc2 the hidden rounded to fp32: d_w2 differs by that rounding
        tol = dict(rtol=1e-6, atol=1e-6)
        assert np.allclose(got["d_buf"][ex, :r], x.grad.numpy(), **tol)
        assert np.allclose(got["d_w1"][ex], w1.grad.numpy(), **tol)
        assert np.allclose(got["d_w2"][ex], w2.grad.numpy(), **tol)
        if act == "swiglu":
            assert np.allclose(got["d_w3"][ex], w3.grad.numpy(), **tol)
        else:
            assert np.allclose(got["d_b1"][ex], b1.grad.numpy(), **tol)
            assert np.allclose(got["d_b2"][ex], b2.grad.numpy(), **tol)


def _loss(c, act, **over):
    """sum over kept rows of <d_out, out> from the oracle's forward (fp32 mode)."""
    p = dict(c, **over)
    rows_e = np.concatenate([np.full(int(k), j, np.int32) for j, k in enumerate(p["kept"])])
    rows_j = np.concatenate([np.arange(int(k), dtype=np.int64) for k in p["kept"]])
    out = oracle.ffn_rows(p["buf"], p["w1"], p["b1"], p["w3"], p["w2"], p["b2"], act,
                          rows_e, rows_j, False)
    return float((out.astype(np.float64) * p["d_out"][rows_e, rows_j].astype(np.float64)).sum())


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_matches_finite_differences_of_the_forward(act):
    c = _case(act, seed=3)
    got = _bwd(c, act)
    hstep = np.float32(2.0 ** -6)
    probes = [("buf", (0, 1, 2), "d_buf"), ("buf", (1, 0, 5), "d_buf"), ("w1", (0, 3, 1), "d_w1"),
              ("w1", (1, 6, 0), "d_w1"), ("w2", (0, 2, 4), "d_w2"), ("w2", (1, 5, 6), "d_w2")]
    if act == "swiglu":
        probes += [("w3", (0, 0, 0), "d_w3"), ("w3", (1, 4, 3), "d_w3")]
    else:
        probes += [("b1", (0, 2), "d_b1"), ("b2", (1, 3), "d_b2")]
    for name, ix, gname in probes:
        plus, minus = c[name].copy(), c[name].copy()
        plus[ix] += hstep
        minus[ix] -= hstep
        fd = (_loss(c, act, **{name: plus}) - _loss(c, act, **{name: minus})) / (2 * float(hstep))
        an = float(got[gname][ix])
        assert abs(an - fd) <= 2e-3 + 2e-3 * abs(fd), (name, ix, an, fd)


@pytest.mark.parametrize("act", ["relu", "swiglu"])
def test_rows_past_kept_do_not_matter(act):
    c = _case(act, seed=5)
    base = _bwd(c, act)
    junk = dict(c)
    junk["buf"], junk["d_out"] = c["buf"].copy(), c["d_out"].copy()
    for ex, k in enumerate(c["kept"]):
        junk["buf"][ex, k:] = 1e3
        junk["d_out"][ex, k:] = -7.0
    other = _bwd(junk, act)
    for key in base:
        assert np.array_equal(base[key], other[key]), key
    for ex, k in enumerate(c["kept"]):
        assert np.all(other["d_buf"][ex, k:] == 0.0)
    # an expert with no kept rows gets zero weight gradients
    assert np.all(base["d_w1"][2] == 0.0) and np.all(base["d_w2"][2] == 0.0)


@pytest.mark.parametrize("act", ["relu", "gelu", "swiglu"])
def test_linear_in_d_out(act):
    c = _case(act, seed=7)
    a = _bwd(c, act)
    # scaling by a power of two commutes with every rounding: bit-exact
    b = _bwd(c, act, d_out=c["d_out"] * np.float32(4.0))
    for key in a:
        assert np.array_equal(a[key] * np.float32(4.0), b[key]), key
    rng = np.random.default_rng(8)
    d2 = rng.standard_normal(c["d_out"].shape).astype(np.float32)
    s = _bwd(c, act, d_out=c["d_out"] + d2)
    p = _bwd(c, act, d_out=d2)
    for key in a:
        assert np.allclose(s[key], a[key] + p[key], rtol=1e-5, atol=1e-5), key


def test_experts_are_independent():
    c = _case("gelu", e=4, kept=(5, 3, 1, 4), seed=9)
    perm = np.array([2, 0, 3, 1])
    pc = {k: (v[perm] if isinstance(v, np.ndarray) else v) for k, v in c.items()}
    a, b = _bwd(c, "gelu"), _bwd(pc, "gelu")
    for key in a:
        assert np.array_equal(a[key][perm], b[key]), key


def test_bf16_mode_rounds_d_buf_once():
    c = _case("gelu", seed=11)
    f32 = _bwd(c, "gelu")
    bf = _bwd(c, "gelu", bf16=True)
    bits = bf["d_buf"].view(np.uint32)
    assert np.all(bits & np.uint32(0xFFFF) == 0)           # bf16-representable
    rel = np.abs(bf["d_buf"] - f32["d_buf"]) <= 2.0 ** -8 * np.abs(f32["d_buf"]) + 1e-30
    assert rel.all()
    # d_buf does not depend on the hidden's rounding; d_w1 neither
    assert np.array_equal(bf["d_w1"], f32["d_w1"])
