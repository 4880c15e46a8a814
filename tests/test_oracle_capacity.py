"""Pins for capacity and slot locations (closed forms, brute force, invariants)."""

import json
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")
with open(os.path.join(GOLD, "capacity.json")) as _f:
    CAP = json.load(_f)


@pytest.mark.parametrize("c", CAP["fixed"], ids=lambda c: f"f{c['f']}_s{c['s']}_e{c['e']}_k{c['k']}")
def test_fixed_capacity_closed_form(c):
    needed = np.zeros(c["e"], np.int64)  # ignored for f > 0
    assert oracle.capacity(c["f"], c["s"], c["e"], c["k"], needed) == c["c"]


@pytest.mark.parametrize("c", CAP["capped_bound"], ids=lambda c: f"f{c['f']}_s{c['s']}")
def test_capped_capacity(c):
    e = c["e"]
    big = np.full(e, 10 ** 7, np.int64)
    assert oracle.capacity(c["f"], c["s"], e, c["k"], big) == c["bound"]
    small = np.zeros(e, np.int64)
    small[e // 2] = c["bound"] - 3
    assert oracle.capacity(c["f"], c["s"], e, c["k"], small) == c["bound"] - 3


def test_adaptive_capacity_is_max_needed():
    needed = np.array([5, 0, 17, 3], np.int64)
    assert oracle.capacity(0.0, 25, 4, 1, needed) == 17


def _brute_loc(idx):
    """loc[r,t] = number of routes before (r,t) in route-major order (r, then t)
    that chose the same expert."""
    k, s = idx.shape
    flat = idx.reshape(-1)
    loc = np.empty_like(flat)
    for n in range(flat.size):
        loc[n] = int(np.count_nonzero(flat[:n] == flat[n]))
    return loc.reshape(k, s)


@pytest.mark.parametrize("seed", range(4))
def test_locations_brute_force(seed):
    rng = np.random.default_rng(seed)
    e, k, s = 5, 3, 41
    idx = np.stack([rng.permutation(e)[:k] for _ in range(s)], axis=1).astype(np.int32)
    loc, needed = oracle.locations(idx, e)
    assert np.array_equal(loc, _brute_loc(idx))
    assert np.array_equal(needed, np.bincount(idx.reshape(-1), minlength=e))


@pytest.mark.parametrize("f", [1.0, 0.5, 0.0, -0.75, -3.0])
def test_locations_invariants(f):
    rng = np.random.default_rng(3)
    e, k, s = 7, 2, 300
    p = np.array([8, 4, 2, 1, 1, 1, 1], np.float64)
    idx = np.stack([rng.choice(e, k, replace=False, p=p / p.sum()) for _ in range(s)], 1).astype(np.int32)
    loc, needed = oracle.locations(idx, e)
    c = oracle.capacity(f, s, e, k, needed)
    kept = loc < c
    for j in range(e):
        lj = np.sort(loc[idx == j])
        assert np.array_equal(lj, np.arange(needed[j]))                # no collision, no hole
        assert np.count_nonzero(kept & (idx == j)) == min(needed[j], c)  # at most c per expert
    if f == 0.0:
        assert kept.all()
    # route priority: a kept route never has a dropped route ahead of it at the same expert
    order = np.argsort(np.arange(k * s))  # route-major order is the flat order
    fl_idx, fl_kept = idx.reshape(-1)[order], kept.reshape(-1)[order]
    for j in range(e):
        kj = fl_kept[fl_idx == j]
        assert not np.any(kj[1:] & ~kj[:-1])


def test_capacity_at_least_s_drops_nothing():
    rng = np.random.default_rng(5)
    e, k, s = 4, 2, 50
    idx = np.stack([rng.permutation(e)[:k] for _ in range(s)], 1).astype(np.int32)
    loc, needed = oracle.locations(idx, e)
    c = oracle.capacity(float(e), s, e, k, needed)   # f*k*s/e = k*s >= s
    assert c >= s and np.all(loc < c)
