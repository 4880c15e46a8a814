"""The oracle's bf16 rounding of double values, pinned by hand-derived cases.

Every bf16 value the oracle produces (the expert MLP's hidden and output rows,
decode-backward's gate-weighted rows, encode/decode outputs) comes from one
rounding of a double (or exact fp32) value to bfloat16, round to nearest with
ties to even.  The fixture's cases are derived from the format's definition:
exact ties, values just off a tie by less than fp32's resolution (where a
double -> fp32 -> bf16 double rounding gives the other neighbour), overflow at
the largest finite value, subnormals and signed zeros.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden", "bf16_round.json")


def _parse(s):
    return {"inf": math.inf, "-inf": -math.inf}.get(s) if s in ("inf", "-inf") else float.fromhex(s)


with open(GOLD) as f:
    CASES = json.load(f)["cases"]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c["value"])
def test_round_bf16_direct_from_double(case):
    v, want = _parse(case["value"]), _parse(case["want"])
    got = oracle.round_bf16(v)
    assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), case["why"]
    # the result is a bf16 value: its fp32 pattern has 16 zero low bits
    assert np.float32(got).view(np.uint32) & 0xFFFF == 0


def test_fixture_catches_double_rounding():
    """At least one case differs when the value is rounded to fp32 first, in
    every region the fixture covers (near 1, near overflow, subnormal)."""
    def via_f32(v):
        f = float(np.float32(v)) if abs(v) < 3.4028235e38 else v
        return oracle.round_bf16(f)

    differ = [c for c in CASES if via_f32(_parse(c["value"])) != _parse(c["want"])]
    mags = {("one" if 0.5 < abs(_parse(c["value"])) < 4 else
             "max" if abs(_parse(c["value"])) > 1e38 else "sub") for c in differ}
    assert mags == {"one", "max", "sub"}


def test_expert_mlp_rounds_its_double_accumulator_once():
    """ReLU expert, m = 3, h = 1: pre = 1 + 2^-8 + 2^-40 accumulated in double;
    the hidden must be its direct bf16 rounding 1 + 2^-7 (an fp32 step first
    would give the tie 1 + 2^-8 and then 1), and with W2 = 1 and no bias the
    output row is that value in every column."""
    buf = np.array([[[1.0, 2.0 ** -8, 2.0 ** -40]]], np.float32)     # [e=1, c=1, m=3]
    w1 = np.ones((1, 1, 3), np.float32)                                 # [e, h=1, m]
    w2 = np.ones((1, 3, 1), np.float32)                                 # [e, m, h]
    out = oracle.ffn_rows(buf, w1, None, None, w2, None, "relu", np.zeros(1, np.int32),
                          np.zeros(1, np.int64), True)
    assert np.array_equal(out[0], np.full(3, 1.0 + 2.0 ** -7, np.float32))
