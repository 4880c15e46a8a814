"""The seeded input generator: determinism, slicing, numpy == torch forms,
rounding, and the moments of the drawn values."""

import numpy as np
import torch

import synth
from synth import rng


def test_splitmix64_reference_values():
    # SplitMix64 with state 0: the first outputs of the published generator
    # (state += 0x9E3779B97F4A7C15; then the mix) are these well-known values.
    outs = [synth.mix64((i + 1) * synth.GOLDEN) for i in range(3)]
    assert outs == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_streams_deterministic_and_sliceable():
    a = synth.normal_host(5, "w1", (1000,), 0.5, "f32")
    b = synth.normal_host(5, "w1", (1000,), 0.5, "f32")
    assert np.array_equal(a, b)
    part = synth.normal_host(5, "w1", (300,), 0.5, "f32", start=400)
    assert np.array_equal(part, a[400:700])
    assert not np.array_equal(a, synth.normal_host(6, "w1", (1000,), 0.5, "f32"))
    assert not np.array_equal(a, synth.normal_host(5, "w2", (1000,), 0.5, "f32"))


def test_numpy_and_torch_forms_agree():
    n = 1 << 16
    a = synth.normal_host(2, "x", (n,), 1.0, "bf16")
    t = synth.normal_torch(2, "x", (n,), 1.0, "bf16", chunk=1 << 12)
    tb = t.view(torch.int16).numpy().view(np.uint16)
    # identical up to a last-bit difference of the double transcendental functions
    assert np.mean(a == tb) > 0.9999
    a32 = synth.normal_host(2, "x", (n,), 1.0, "f32", start=77)
    t32 = synth.normal_torch(2, "x", (n,), 1.0, "f32", start=77).numpy()
    assert np.max(np.abs(a32 - t32)) <= 1e-6


def test_bf16_rounding_matches_torch():
    v = np.random.default_rng(0).standard_normal(100000).astype(np.float32)
    v[:4] = [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]  # exact ties
    ours = rng.f32_to_bf16_bits(v)
    theirs = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)
    assert np.array_equal(rng.bf16_bits_to_f32(ours), torch.from_numpy(v).to(torch.bfloat16).float().numpy())


def test_moments():
    z = synth.normal_host(0, "x", (1 << 18,), 2.0, "f32").astype(np.float64)
    assert abs(z.mean()) < 0.02 and abs(z.std() - 2.0) < 0.02
    assert abs(np.mean(np.abs(z) < 2.0) - 0.6827) < 0.005


def test_workload_table():
    names = list(synth.WORKLOADS)
    assert len(names) == 4 and len(synth.sweep_points()) == 32
    w = synth.workloads.BF16_E8
    assert (w.s, w.m, w.e, w.k, w.h, w.capacity_factor) == (4096, 1024, 8, 2, 4096, 1.25)
    pts = synth.sweep_points()
    assert [p.seed for p in pts] == list(range(32))
    b = synth.workloads.gate_bias_host(synth.workloads.BF16_E256_SWIGLU)
    assert b[0] == 0 and abs(b[1] + 2 * np.log(2)) < 1e-6
