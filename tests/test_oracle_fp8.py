"""Pins of the oracle's FP8 (e4m3) functions against the format's definition
(sign, 4 exponent bits with bias 7, 3 mantissa bits, subnormal step 2^-9, no
infinities, largest finite 448) and against the already-pinned bf16 expert
oracle.  The low-precision experts restate the Tutel profile's FP8 inference
formats with one scale per operand row."""

import math

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _value(code):
    """Hand decode from the bit fields (independent of the oracle)."""
    s = -1.0 if code & 0x80 else 1.0
    ef, mf = (code >> 3) & 15, code & 7
    if ef == 15 and mf == 7:
        return math.nan
    if ef == 0:
        return s * mf * 2.0 ** -9
    return s * (1 + mf / 8) * 2.0 ** (ef - 7)


FINITE = [c for c in range(256) if not math.isnan(_value(c))]


@pytest.mark.parametrize("v,code", [
    (0.0, 0x00), (-0.0, 0x80), (1.0, 0x38), (-1.0, 0xB8), (448.0, 0x7E), (-448.0, 0xFE),
    (500.0, 0x7E), (1e9, 0x7E), (-1e30, 0xFE),          # saturation
    (2.0 ** -9, 0x01), (2.0 ** -6, 0x08), (7 * 2.0 ** -9, 0x07),
    (2.0 ** -10, 0x00),                                 # tie between 0 and 2^-9 -> even (0)
    (3 * 2.0 ** -10, 0x02),                             # tie between 1 and 2 quanta -> 2
    (1.0625, 0x38), (1.1875, 0x3A),                     # ties between mantissas -> even
    (0.1, 0x1D), (3.0, 0x44), (240.0, 0x77), (464.0, 0x7E),
])
def test_fp8_encode_known_values(v, code):
    assert oracle.fp8_encode(v) == code
    if abs(v) <= 448 and v == _value(code):
        assert oracle.fp8_decode(code) == v


def test_fp8_decode_every_code():
    for c in range(256):
        want = _value(c)
        got = oracle.fp8_decode(c)
        assert (math.isnan(want) and math.isnan(got)) or got == want, hex(c)
    assert oracle.fp8_encode(float("nan")) & 0x7F == 0x7F


def test_fp8_encode_is_nearest_ties_to_even_brute_force():
    rng = np.random.default_rng(3)
    vals = np.concatenate([
        rng.normal(0, 1, 3000), rng.normal(0, 100, 2000), rng.uniform(-600, 600, 1000),
        rng.normal(0, 0.01, 1000),
        # exact midpoints between neighbouring codes, and values a hair off them
        np.array([(_value(a) + _value(b)) / 2 for a, b in zip(FINITE[:-1], FINITE[1:])
                  if a & 0x80 == b & 0x80 and (a & 0x7F) + 1 == (b & 0x7F)]),
    ]).astype(np.float32)
    table = np.array([_value(c) for c in FINITE])
    for v in vals:
        v = float(v)
        code = oracle.fp8_encode(v)
        if abs(v) >= 448:
            assert code == (0xFE if v < 0 else 0x7E)
            continue
        d = np.abs(table - v)
        best = np.flatnonzero(d == d.min())
        cands = [FINITE[i] for i in best]
        if len(cands) > 1:   # a tie: the even mantissa (ties of +-0 keep the sign)
            cands = [c for c in cands if c & 1 == 0] or cands
            cands = [c for c in cands if (c & 0x80) == (0x80 if math.copysign(1, v) < 0 else 0)] or cands
        assert code in cands, (v, hex(code), [hex(c) for c in cands])


def test_quantize_rows_fp8():
    rng = np.random.default_rng(5)
    x = rng.normal(0, 3, (7, 300)).astype(np.float32)
    x[3] = 0.0
    x[5, 17] = -50.0   # the row's amax is negative
    q, sc = oracle.quantize_rows_fp8(x)
    assert q.dtype == np.uint8 and sc.dtype == np.float32
    for r in range(7):
        amax = np.abs(x[r]).max()
        if amax == 0:
            assert sc[r] == 1.0 and np.all(q[r] == 0)
            continue
        assert sc[r] == np.float32(amax) / np.float32(448.0)
        i = int(np.argmax(np.abs(x[r])))
        assert q[r, i] == (0xFE if x[r, i] < 0 else 0x7E)
        deq = np.array([_value(int(c)) for c in q[r]]) * float(sc[r])
        # within half a step of the value's own binade (3 mantissa bits: 2^-4 relative)
        assert np.all(np.abs(deq - x[r]) <= np.abs(x[r]) * 2.0 ** -4 + float(sc[r]) * 2.0 ** -10)


def test_fc_fp8_identity_weight_and_scaling():
    rng = np.random.default_rng(9)
    qa = rng.integers(0, 256, (5, 16), dtype=np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0x10   # no NaN codes
    sa = rng.uniform(0.5, 2, 5).astype(np.float32)
    one = oracle.fp8_encode(1.0)
    qw = np.zeros((16, 16), np.uint8)
    np.fill_diagonal(qw, one)
    sw = np.ones(16, np.float32)
    out = oracle.fc_fp8(qa, sa, qw, sw, None, None)
    want = np.array([[oracle.round_bf16(float(sa[r]) * _value(int(qa[r, k]))) for k in range(16)]
                     for r in range(5)], np.float32)
    assert np.array_equal(out, want)
    # a power-of-two factor on a row scale moves the (unrounded) result exactly
    qw2 = rng.integers(0, 0x70, (9, 16), dtype=np.uint8)
    sw2 = rng.uniform(0.5, 2, 9).astype(np.float32)
    base = oracle.fc_fp8(qa, np.ones(5, np.float32), qw2, sw2, None, None)
    twice = oracle.fc_fp8(qa, np.full(5, 2.0, np.float32), qw2, sw2, None, None)
    assert np.array_equal(twice, 2 * base)


@pytest.mark.parametrize("act", ["relu", "gelu"])
def test_fc_fp8_equals_the_bf16_expert_oracle_on_e4m3_values(act):
    """With unit scales and operands that are e4m3 values, fc1 of the FP8
    layer is the bf16 expert oracle's fc1 (its fc2 an identity here)."""
    rng = np.random.default_rng(11)
    m = h = 24
    qx = rng.integers(0, 0x60, (6, m), dtype=np.uint8) | (rng.integers(0, 2, (6, m)) * 0x80).astype(np.uint8)
    qw = rng.integers(0, 0x50, (h, m), dtype=np.uint8) | (rng.integers(0, 2, (h, m)) * 0x80).astype(np.uint8)
    b1 = rng.normal(0, 1, h).astype(np.float32)
    b1 = np.array([oracle.round_bf16(float(v)) for v in b1], np.float32)
    xv = np.array([[_value(int(c)) for c in row] for row in qx], np.float32)
    wv = np.array([[_value(int(c)) for c in row] for row in qw], np.float32)
    got = oracle.fc_fp8(qx, np.ones(6, np.float32), qw, np.ones(h, np.float32), b1, act)
    ident = np.eye(m, dtype=np.float32)
    want = oracle.ffn_rows(xv[None], wv[None], b1[None], None, ident[None], None, act,
                           np.zeros(6, np.int32), np.arange(6), True)
    assert np.array_equal(got, want)
