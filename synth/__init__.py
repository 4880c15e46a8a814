"""Seeded synthetic inputs shared by the CPU oracle, the GPU tests and the bench.

This module only draws numbers.  It contains none of the MoE layer's
arithmetic (no gating, capacity, dispatch, expert or combine step), so the
oracle and the CUDA path can both take their inputs from here without sharing
any computation.

Generator (counter-based, so any slice can be regenerated independently):

* stream key  K = mix64(seed * GOLDEN + fnv1a64(name))
* raw bits    b(n) = mix64(K + (n + 1) * GOLDEN)          (SplitMix64 output n)
* uniform     u(n) = ((b(n) >> 11) + 0.5) * 2**-53        in (0, 1)
* normal      z(i) = sqrt(-2 ln u(2i)) * cos(2 pi u(2i+1)) (Box-Muller, double)
* a tensor element i is  round(scale * z(i))  with round = RNE to fp32, and for
  bf16 a second RNE from that fp32 value to bf16 (documented two-step rounding).

`normal_host` is the authoritative numpy implementation.  `normal_torch` is the
same recipe in torch integer/double ops; it exists so that multi-GB weights of
the large workloads can be drawn directly in device memory.  Tests that use it
copy the drawn input slices back to the host before handing them to the oracle.
"""

from .rng import (  # noqa: F401
    GOLDEN,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    mix64,
    normal_host,
    normal_torch,
    stream_key,
    uniform_host,
)
from .workloads import Workload, WORKLOADS, sweep_points, make_inputs_host, make_inputs_device  # noqa: F401
