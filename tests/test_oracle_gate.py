"""Pins for the oracle's gate: logit order, top-k selection, softmax gates.

Runs on the CPU only.  Each check ties the oracle to something other than
itself: hand-derived values (tests/golden), brute-force enumeration, exact
integer arithmetic, or closed forms.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _load("gate_order.json")["cases"], ids=lambda c: c["name"])
def test_gate_logit_order_golden(case):
    x = np.array([case["x"]], np.float32)
    wg = np.array(case["wg"], np.float32)
    bias = None if case["bias"] is None else np.array(case["bias"], np.float32)
    got = oracle.gate_logits(x, wg, bias, chunk=case["chunk"])[0]
    want = np.atleast_1d(np.array(case["logit"], np.float32))
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (got, want)


def test_gate_logits_exact_on_small_integers():
    """Integer-valued x and wg with small magnitudes: every fp32 step is exact, so
    the logits equal the exact integer matrix product."""
    rng = np.random.default_rng(1)
    x = rng.integers(-8, 9, size=(37, 70))
    wg = rng.integers(-8, 9, size=(70, 5))
    b = rng.integers(-3, 4, size=5)
    got = oracle.gate_logits(x.astype(np.float32), wg.astype(np.float32), b.astype(np.float32))
    want = x.astype(np.int64) @ wg.astype(np.int64) + b
    assert np.array_equal(got, want.astype(np.float32))


def test_gate_logits_bf16_inputs_widen_exactly():
    import synth

    xb = synth.normal_host(3, "x", (5, 16), 1.0, "bf16")
    wg = synth.normal_host(3, "wg", (16, 3), 0.25, "f32")
    a = oracle.gate_logits(xb, wg)               # uint16 bits: chunks of 8
    b = oracle.gate_logits(synth.bf16_bits_to_f32(xb), wg, chunk=8)
    assert np.array_equal(a, b)


def test_gate_chunk_follows_expert_count_and_dtype():
    """The layer's order: lane-blocked chunks of one 16-byte load (8 bf16 or 4
    fp32 elements) for e <= 32, one sequential accumulator above."""
    assert oracle.gate_chunk(32, True) == 8 and oracle.gate_chunk(1, False) == 4
    assert oracle.gate_chunk(33, True) == 0 and oracle.gate_chunk(256, False) == 0
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 96)).astype(np.float32)
    wg = rng.standard_normal((96, 40)).astype(np.float32)
    seq = oracle.gate_logits(x, wg, chunk=0)
    assert np.array_equal(oracle.gate_logits(x, wg), seq)          # e = 40 > 32
    assert np.array_equal(oracle.gate_logits(x, wg[:, :8]),
                          oracle.gate_logits(x, wg[:, :8], chunk=4))


def test_gate_logits_orders_agree_to_rounding():
    """Every order sums the same exact products: the two orders differ from the
    exact (fp64) dot product by at most a few ulp of the sum of |products|."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((16, 1024)).astype(np.float32)
    wg = (rng.standard_normal((1024, 8)) / 32).astype(np.float32)
    exact = x.astype(np.float64) @ wg.astype(np.float64)
    scale = np.abs(x.astype(np.float64)) @ np.abs(wg.astype(np.float64))
    for chunk in (0, 4, 8):
        got = oracle.gate_logits(x, wg, chunk=chunk).astype(np.float64)
        assert np.all(np.abs(got - exact) <= 1024 * 2.0 ** -24 * scale), chunk


def _brute_topk(v, k):
    """Route r is the expert beaten by exactly r others; a beats b iff
    v[a] > v[b] or (v[a] == v[b] and a < b)."""
    e = len(v)
    rank = [sum(1 for a in range(e) if v[a] > v[b] or (v[a] == v[b] and a < b)) for b in range(e)]
    return [rank.index(r) for r in range(k)]


@pytest.mark.parametrize("e", [1, 2, 3, 4])
def test_topk_exhaustive_small_grids(e):
    """Every logit vector over {0, 1, 2}^e (ties forced), every k."""
    vecs = np.array(list(itertools.product([0.0, 1.0, 2.0], repeat=e)), np.float32)
    for k in range(1, e + 1):
        idx = oracle.topk(vecs, k)
        for t, v in enumerate(vecs):
            want = _brute_topk(list(v), k)
            assert list(idx[:, t]) == want, (v, k, idx[:, t], want)
            # the selected set maximises the sum over all k-subsets
            best = max(sum(v[list(c)]) for c in itertools.combinations(range(e), k))
            assert sum(v[idx[:, t]]) == best


def test_topk_random_and_negative_zero():
    rng = np.random.default_rng(7)
    v = rng.standard_normal((200, 9)).astype(np.float32)
    v[:, 3] = v[:, 5]  # exact ties
    for k in (1, 3, 9):
        idx = oracle.topk(v, k)
        for t in range(v.shape[0]):
            assert list(idx[:, t]) == _brute_topk(list(v[t]), k)
    z = np.array([[0.0, -0.0, -1.0]], np.float32)
    z[0, 0] = -0.0
    z[0, 1] = 0.0
    assert list(oracle.topk(z, 2)[:, 0]) == [0, 1]  # -0 == +0: lower index first


@pytest.mark.parametrize("case", _load("softmax.json")["cases"])
def test_gates_closed_forms(case):
    lg = np.array([case["logits"]], np.float32)
    idx = oracle.topk(lg, case["k"])
    assert list(idx[:, 0]) == case["idx"]
    g = oracle.gates(lg, idx, case["normalize"])[:, 0]
    np.testing.assert_allclose(g, case["gates"], rtol=2e-7, atol=1e-8)


def test_gates_invariants():
    rng = np.random.default_rng(11)
    lg = (3 * rng.standard_normal((300, 16))).astype(np.float32)
    for k in (1, 2, 5):
        idx = oracle.topk(lg, k)
        g = oracle.gates(lg, idx, True)
        assert np.all(np.abs(g.astype(np.float64).sum(0) - 1.0) <= k * 2 ** -23)
        assert np.all(np.diff(g, axis=0) <= 0)          # route order = descending gate
        raw = oracle.gates(lg, idx, False)
        # raw probability of the top expert: closed form 1 / sum exp(l - l_top)
        top = lg[np.arange(300), idx[0]].astype(np.float64)
        want = 1.0 / np.exp(lg.astype(np.float64) - top[:, None]).sum(1)
        np.testing.assert_allclose(raw[0], want, rtol=1e-6)
        # shifting every logit by a constant leaves routing and gates unchanged
        lg2 = lg + np.float32(4.0)
        idx2 = oracle.topk(lg2, k)
        assert np.array_equal(idx, idx2)
        np.testing.assert_allclose(oracle.gates(lg2, idx2, True), g, rtol=2e-6)


def test_two_expert_probability_closed_form():
    a, b = 0.3, -1.7
    lg = np.array([[a, b]], np.float32)
    idx = oracle.topk(lg, 1)
    g = oracle.gates(lg, idx, False)[0, 0]
    want = 1.0 / (1.0 + math.exp(float(np.float32(b)) - float(np.float32(a))))
    assert idx[0, 0] == 0 and abs(g - want) < 1e-7
