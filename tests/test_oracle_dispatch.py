"""Pins for encode / decode and their backward: sparse loops vs the dense
one-hot einsum, gate-mass conservation, adjoint identities, exact derivatives."""

import numpy as np
import pytest

import oracle
from oracle import dense

import synth


def _routing(seed, s, e, k, f, skew=0.0):
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((s, e)).astype(np.float32)
    if skew:
        lg = lg - np.float32(skew) * np.log(np.arange(1, e + 1, dtype=np.float32))
    idx = oracle.topk(lg, k)
    g = oracle.gates(lg, idx, k >= 2)
    loc, needed = oracle.locations(idx, e)
    c = oracle.capacity(f, s, e, k, needed)
    return idx, g, loc, needed, c


CASES = [
    # seed, s, m, e, k, f, skew, dtype
    (0, 64, 24, 4, 1, 1.0, 0.0, "f32"),
    (1, 96, 16, 6, 2, 0.75, 1.5, "f32"),
    (2, 80, 32, 8, 3, 0.0, 0.0, "bf16"),
    (3, 120, 8, 5, 2, -0.8, 2.0, "bf16"),
]


@pytest.mark.parametrize("case", CASES)
def test_sparse_equals_dense(case):
    seed, s, m, e, k, f, skew, dt = case
    bf16 = dt == "bf16"
    idx, g, loc, needed, c = _routing(seed, s, e, k, f, skew)
    x = oracle.to_f32(synth.normal_host(seed, "x", (s, m), 1.0, dt))
    D = dense.dispatch_mask(idx, loc, c, e)
    C = dense.combine_weights(idx, loc, g, c, e)
    cmax = c + 3  # physical row stride larger than c: the logical [e, c, m] view is a slice
    buf = oracle.encode(x, idx, loc, c, e, cmax)
    assert np.array_equal(buf[:, :c], dense.encode(D, x))   # copies are exact
    assert not buf[:, c:].any()
    out = oracle.to_f32(synth.normal_host(seed, "out", (e, cmax, m), 1.0, dt))
    y = oracle.decode(out, idx, loc, g, c, bf16)
    yd = dense.decode(C, out[:, :c])
    tol = 2 ** -8 if bf16 else 4 * 2 ** -24
    assert np.all(np.abs(y - yd) <= tol * np.abs(yd) + 1e-6 * k)
    dy = oracle.to_f32(synth.normal_host(seed, "dy", (s, m), 1.0, dt))
    d_out, d_g = oracle.decode_bwd(dy, out, idx, loc, g, c, bf16)
    d_out_d, dC = dense.decode_bwd(C, D, dy, out[:, :c])
    assert np.all(np.abs(d_out[:, :c] - d_out_d) <= (2 ** -8 if bf16 else 2 ** -24) * np.abs(d_out_d))
    assert not d_out[:, c:].any()
    # gate gradient of route (r, t) is the slot entry of dC it landed in
    for r in range(k):
        for t in range(s):
            want = dC[t, idx[r, t], loc[r, t]] if loc[r, t] < c else 0.0
            assert abs(d_g[r, t] - want) <= 1e-6 * (1 + abs(want))
    dbuf = oracle.to_f32(synth.normal_host(seed, "dbuf", (e, cmax, m), 1.0, dt))
    dx = oracle.encode_bwd(dbuf, idx, loc, c, bf16)
    dxd = dense.encode_bwd(D, dbuf[:, :c])
    assert np.all(np.abs(dx - dxd) <= tol * np.abs(dxd) + 1e-6 * k)


@pytest.mark.parametrize("f", [0.0, 0.6])
def test_identity_expert_conserves_gate_mass(f):
    """decode(encode(x)) with identity experts equals kappa_t * x_t, kappa_t the
    sum of the token's kept gates; sum_t kappa_t equals the combine mask's mass."""
    s, m, e, k = 200, 12, 6, 2
    idx, g, loc, needed, c = _routing(9, s, e, k, f)
    x = synth.normal_host(9, "x", (s, m), 1.0, "f32")
    buf = oracle.encode(x, idx, loc, c, e, c)
    y = oracle.decode(buf, idx, loc, g, c, False)
    kappa = np.where(loc < c, g, 0).astype(np.float64).sum(0)
    np.testing.assert_allclose(y, kappa[:, None] * x, rtol=3e-7, atol=1e-7)
    C = dense.combine_weights(idx, loc, g, c, e)
    assert abs(kappa.sum() - C.sum()) < 1e-9
    if f == 0.0:  # nothing dropped, gates renormalised: every token keeps mass 1
        assert np.all(np.abs(kappa - 1) <= k * 2 ** -23)
    dx = oracle.encode_bwd(buf, idx, loc, c, False)
    nkept = (loc < c).sum(0)
    np.testing.assert_allclose(dx, nkept[:, None] * x, rtol=3e-7, atol=1e-7)


def test_adjoint_identities():
    """<decode(E), dY> = <E, d_out(dY)> and <encode(x), B> = <x, encode_bwd(B)>,
    in double, with the sparse oracle on fp32 data."""
    s, m, e, k = 150, 20, 5, 3
    idx, g, loc, needed, c = _routing(4, s, e, k, 0.7)
    E = synth.normal_host(4, "E", (e, c, m), 1.0, "f32")
    dY = synth.normal_host(4, "dY", (s, m), 1.0, "f32")
    lhs = np.sum(oracle.decode(E, idx, loc, g, c, False).astype(np.float64) * dY)
    d_out, _ = oracle.decode_bwd(dY, E, idx, loc, g, c, False)
    rhs = np.sum(E.astype(np.float64) * d_out)
    assert abs(lhs - rhs) <= 1e-5 * (abs(lhs) + 1)
    x = synth.normal_host(4, "x", (s, m), 1.0, "f32")
    B = synth.normal_host(4, "B", (e, c, m), 1.0, "f32")
    l2 = np.sum(oracle.encode(x, idx, loc, c, e, c).astype(np.float64) * B)
    r2 = np.sum(x.astype(np.float64) * oracle.encode_bwd(B, idx, loc, c, False))
    assert abs(l2 - r2) <= 1e-5 * (abs(l2) + 1)


def test_gate_gradient_is_exact_derivative():
    """decode is linear in each gate: y(g + d*onehot) - y(g) = d * out[slot]."""
    s, m, e, k = 40, 10, 4, 2
    idx, g, loc, needed, c = _routing(12, s, e, k, 1.0)
    out = synth.normal_host(12, "out", (e, c, m), 1.0, "f32")
    dY = synth.normal_host(12, "dY", (s, m), 1.0, "f32")
    _, d_g = oracle.decode_bwd(dY, out, idx, loc, g, c, False)
    C = dense.combine_weights(idx, loc, g, c, e)
    base = dense.decode(C, out)
    for r in range(k):
        for t in range(0, s, 7):
            g2 = g.astype(np.float64).copy()
            g2[r, t] += 1.0
            C2 = dense.combine_weights(idx, loc, g2, c, e)
            fd = np.sum((dense.decode(C2, out) - base) * dY)
            assert abs(d_g[r, t] - fd) <= 1e-5 * (1 + abs(fd))


def _one_token(vals, gates):
    """One token whose k routes go to experts 0..k-1, slot 0 each, m = 1."""
    k = len(vals)
    out = np.array(vals, np.float32).reshape(k, 1, 1)           # [e = k, c = 1, m = 1]
    idx = np.arange(k, dtype=np.int32).reshape(k, 1)
    loc = np.zeros((k, 1), np.int32)
    g = np.array(gates, np.float32).reshape(k, 1)
    return out, idx, loc, g


def test_decode_accumulates_by_fused_multiply_add_in_route_order():
    """The combine accumulates in fp32 (the DeepSpeed index-dispatch PR, change
    3); the reading adopted is one fused multiply-add per kept route, in
    ascending route order from +0.  Route 0 contributes 1 * (-1), route 1
    (1 + 2^-12)^2 = 1 + 2^-11 + 2^-24: fused, the low bit survives and y =
    2^-11 + 2^-24.  A separate multiply rounds the product to 1 + 2^-11 (tie to
    even) and gives 2^-11; the reverse route order gives 2^-11 as well."""
    u = 1.0 + 2.0 ** -12
    out, idx, loc, g = _one_token([-1.0, u], [1.0, u])
    y = oracle.decode(out, idx, loc, g, 1, False)
    assert y[0, 0] == np.float32(2.0 ** -11 + 2.0 ** -24)


def test_encode_bwd_adds_routes_in_ascending_order():
    """dX sums the kept routes' rows in fp32 in ascending route order from +0:
    2^24 + 1 ties to even at 2^24, and - 2^24 then gives 0.  Descending order
    would give -2^24 + 1 = -16777215 (exact), then + 2^24 = 1."""
    d_buf, idx, loc, _ = _one_token([2.0 ** 24, 1.0, -(2.0 ** 24)], [1.0, 1.0, 1.0])
    dx = oracle.encode_bwd(d_buf, idx, loc, 1, False)
    assert dx[0, 0] == 0.0


def _bf16_of_f32(a):
    return synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(a))


def test_bf16_outputs_are_rounded_once():
    """With bf16 tensors the combine, its K0 twin and dE are rounded to bf16
    exactly once, after the fp32 accumulation (decode, encode backward) or from
    the exact product g * dY (decode backward)."""
    s, m, e, k = 70, 16, 5, 2
    idx, g, loc, needed, c = _routing(21, s, e, k, 0.8)
    cmax = c + 2
    out = _bf16_of_f32(synth.normal_host(21, "out", (e, cmax, m), 1.0, "f32"))
    dy = _bf16_of_f32(synth.normal_host(21, "dy", (s, m), 1.0, "f32"))
    y_b = oracle.decode(out, idx, loc, g, c, True)
    y_f = oracle.decode(out, idx, loc, g, c, False)
    assert np.array_equal(y_b.view(np.uint32), _bf16_of_f32(y_f).view(np.uint32))
    dx_b = oracle.encode_bwd(out, idx, loc, c, True)
    dx_f = oracle.encode_bwd(out, idx, loc, c, False)
    assert np.array_equal(dx_b.view(np.uint32), _bf16_of_f32(dx_f).view(np.uint32))
    d_out, _ = oracle.decode_bwd(dy, out, idx, loc, g, c, True)
    kept = loc < c
    for r, t in zip(*np.nonzero(kept)):
        row = d_out[idx[r, t], loc[r, t]].astype(np.float64)
        exact = np.float64(g[r, t]) * dy[t].astype(np.float64)
        assert np.all(row.astype(np.float32).view(np.uint32) & 0xFFFF == 0)      # bf16 values
        # nearest bf16: within half a bf16 step (2^-8 relative) of the exact product
        assert np.all(np.abs(row - exact) <= np.abs(exact) * 2.0 ** -8)
