"""Pins for the oracle's gate backward (softmax / renormalised gates to logits,
then through logits = x Wg + b).

Runs on the CPU only.  The checks tie it to finite differences of the
oracle's forward gate (itself pinned by closed forms), to closed-form
derivatives, and to the definitions of the three products.
"""

import numpy as np
import pytest

import oracle


def _gates64(logits, idx, normalize):
    return oracle.gates(logits, idx, normalize).astype(np.float64)


def _separated_logits(rng, s, e, gap=0.25):
    """Logits whose sorted neighbours differ by at least `gap`, so a small
    perturbation never changes the top-k selection."""
    base = np.stack([rng.permutation(e) for _ in range(s)]).astype(np.float64)
    return (base * gap + rng.uniform(-0.05, 0.05, size=(s, e))).astype(np.float32)


@pytest.mark.parametrize("normalize,k", [(True, 2), (True, 3), (False, 1), (False, 3)])
def test_d_logits_match_finite_differences(normalize, k):
    rng = np.random.default_rng(10 + k)
    s, e = 6, 5
    lg = _separated_logits(rng, s, e)
    idx = oracle.topk(lg, k)
    dg = rng.standard_normal((k, s)).astype(np.float32)
    # the oracle's backward from these logits: x = I and wg = logits make x Wg
    # = logits exactly (one nonzero product per logit)
    out = oracle.gate_bwd(np.eye(s, dtype=np.float32), lg, None, idx, dg, normalize, chunk=0)
    dl = out["d_logits"]
    h = np.float32(2.0 ** -7)
    for t in range(s):
        for j in range(e):
            lp, lm = lg.copy(), lg.copy()
            lp[t, j] += h
            lm[t, j] -= h
            fd = ((dg * _gates64(lp, idx, normalize)).sum()
                  - (dg * _gates64(lm, idx, normalize)).sum()) / (2 * float(h))
            assert abs(dl[t, j] - fd) <= 2e-3 + 2e-3 * abs(fd), (t, j, dl[t, j], fd)


def test_two_expert_logistic_closed_form():
    """e = 2, k = 1, raw softmax: g = sigma(l0 - l1) for the selected expert 0,
    so dL/dl0 = dg g (1 - g) and dL/dl1 = -dg g (1 - g)."""
    lg = np.array([[1.5, -0.25]], np.float32)
    idx = np.array([[0]], np.int32)
    dg = np.array([[0.75]], np.float32)
    out = oracle.gate_bwd(np.eye(1, dtype=np.float32), lg, None, idx, dg, False, chunk=0)
    g = 1.0 / (1.0 + np.exp(-(1.5 + 0.25)))
    want = 0.75 * g * (1.0 - g)
    assert np.allclose(out["d_logits"][0], [want, -want], rtol=1e-12, atol=1e-15)


def test_degenerate_selections():
    """Renormalised k = 1: every gate is 1, so no gradient reaches the logits.
    Renormalised k = e equals the raw softmax over all experts."""
    rng = np.random.default_rng(4)
    s, e = 7, 4
    lg = rng.standard_normal((s, e)).astype(np.float32)
    eye = np.eye(s, dtype=np.float32)
    idx1 = oracle.topk(lg, 1)
    dg1 = rng.standard_normal((1, s)).astype(np.float32)
    assert np.all(oracle.gate_bwd(eye, lg, None, idx1, dg1, True, chunk=0)["d_logits"] == 0.0)
    idxe = oracle.topk(lg, e)
    dge = rng.standard_normal((e, s)).astype(np.float32)
    a = oracle.gate_bwd(eye, lg, None, idxe, dge, True, chunk=0)["d_logits"]
    b = oracle.gate_bwd(eye, lg, None, idxe, dge, False, chunk=0)["d_logits"]
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


def test_products_through_the_gate_weight():
    """d_wg = x^T dl, d_bias = sum_t dl, d_x = dl wg^T (their definitions, in
    fp64), and a finite difference of the whole scalar through x Wg."""
    rng = np.random.default_rng(5)
    s, m, e, k = 9, 24, 6, 2
    x = rng.standard_normal((s, m)).astype(np.float32)
    wg = (rng.standard_normal((m, e)) * 0.3).astype(np.float32)
    bias = (rng.standard_normal(e) * 0.1).astype(np.float32)
    lg = oracle.gate_logits(x, wg, bias)
    idx = oracle.topk(lg, k)
    dg = rng.standard_normal((k, s)).astype(np.float32)
    out = oracle.gate_bwd(x, wg, bias, idx, dg, True)
    dl = out["d_logits"]
    x64, w64 = x.astype(np.float64), wg.astype(np.float64)
    assert np.allclose(out["d_wg"], x64.T @ dl, rtol=1e-12, atol=1e-13)
    assert np.allclose(out["d_bias"], dl.sum(0), rtol=1e-12, atol=1e-13)
    assert np.allclose(out["d_x"], dl @ w64.T, rtol=1e-12, atol=1e-13)
    # end to end: perturb one weight, keep the selection (checked), compare
    h = np.float32(2.0 ** -8)
    for (i, j) in [(0, 0), (5, 3), (23, 5)]:
        wp, wm = wg.copy(), wg.copy()
        wp[i, j] += h
        wm[i, j] -= h
        lp, lm = oracle.gate_logits(x, wp, bias), oracle.gate_logits(x, wm, bias)
        if not (np.array_equal(oracle.topk(lp, k), idx) and np.array_equal(oracle.topk(lm, k), idx)):
            continue
        fd = ((dg * _gates64(lp, idx, True)).sum() - (dg * _gates64(lm, idx, True)).sum()) / (2 * float(h))
        assert abs(out["d_wg"][i, j] - fd) <= 5e-3 + 5e-3 * abs(fd), (i, j, out["d_wg"][i, j], fd)
