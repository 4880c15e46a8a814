"""Helpers shared by the GPU parity tests: host<->device moves and tolerances.

Tolerance (the layer's stated bar): |got - want| <= atol + rtol*|want| with
fp32: rtol = atol = 1e-5;  bf16: rtol = 2e-2, atol = 1e-2.  Integer outputs and
pure copies are compared bit for bit.
"""

import numpy as np
import torch

TOL = {"f32": (1e-5, 1e-5), "bf16": (2e-2, 1e-2)}


def to_dev(a, device="cuda"):
    """numpy -> device tensor.  uint16 arrays are bf16 bit patterns."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def to_host(t):
    """device tensor -> numpy (bf16 widened to fp32 values exactly)."""
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()


def bits(t):
    """Raw bit patterns of a tensor (for bit-exact comparisons)."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy()
    if t.dtype == torch.float32:
        return t.view(torch.int32).cpu().numpy()
    return t.cpu().numpy()


def f32_bits(a):
    a = np.ascontiguousarray(a, np.float32)
    return a.view(np.int32)


def bf16_bits_of_f32(a):
    """fp32 arrays that hold bf16 values -> their int16 bf16 patterns."""
    return (np.ascontiguousarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16).view(np.int16)


def assert_close(got, want, dt, what=""):
    rtol, atol = TOL[dt]
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    err = np.abs(got - want)
    bad = err > atol + rtol * np.abs(want)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first at "
                             f"{tuple(i)}: got {got[tuple(i)]!r} want {want[tuple(i)]!r}")


def status_ok(st):
    v = int(st.item())
    assert v == 0, f"device status {v}"
