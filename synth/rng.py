"""Counter-based normal generator (SplitMix64 + Box-Muller), numpy and torch forms.

Both forms compute, for element n of a named stream, exactly the recipe in the
package docstring.  All integer arithmetic is modulo 2**64.
"""

import math

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
_C1 = 0xBF58476D1CE4E5B9
_C2 = 0x94D049BB133111EB
_M64 = (1 << 64) - 1
_CHUNK = 1 << 22  # elements per host chunk (bounds temporary memory)


def _mix64_int(z: int) -> int:
    z &= _M64
    z = ((z ^ (z >> 30)) * _C1) & _M64
    z = ((z ^ (z >> 27)) * _C2) & _M64
    return z ^ (z >> 31)


def mix64(z):
    """SplitMix64 finaliser on a numpy uint64 array (or a Python int)."""
    if isinstance(z, int):
        return _mix64_int(z)
    z = np.asarray(z, dtype=np.uint64).copy()
    z ^= z >> np.uint64(30)
    z *= np.uint64(_C1)
    z ^= z >> np.uint64(27)
    z *= np.uint64(_C2)
    z ^= z >> np.uint64(31)
    return z


def _fnv1a64(name: str) -> int:
    h = 0xCBF29CE484222325
    for byte in name.encode("utf-8"):
        h ^= byte
        h = (h * 0x100000001B3) & _M64
    return h


def stream_key(seed: int, name: str) -> int:
    return _mix64_int((seed * GOLDEN + _fnv1a64(name)) & _M64)


def uniform_host(key: int, start: int, count: int) -> np.ndarray:
    """u(n) for n in [start, start+count), float64 in (0, 1)."""
    n = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        b = mix64(np.uint64(key) + (n + np.uint64(1)) * np.uint64(GOLDEN))
    return ((b >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = (u & 0x7F800000) == 0x7F800000
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    r = np.where(nan & ((u & 0x7FFFFF) != 0), (u >> 16) | 0x40, r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32 values."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_host(seed: int, name: str, shape, scale: float = 1.0, dtype: str = "f32",
                start: int = 0) -> np.ndarray:
    """Seeded N(0, scale^2) tensor.  dtype 'f32' -> float32 array, 'bf16' -> uint16 bits.

    `start` offsets the element counter, so `normal_host(..., start=a)` of length L
    equals elements [a, a+L) of the same stream drawn whole.
    """
    shape = tuple(int(d) for d in shape)
    count = int(np.prod(shape, dtype=np.int64)) if shape else 1
    if dtype not in ("f32", "bf16"):
        raise ValueError(f"unknown dtype {dtype!r}")
    key = stream_key(seed, name)
    # converted chunk by chunk, so that a multi-GB tensor needs no full-size temporaries
    out = np.empty(count, dtype=np.float32 if dtype == "f32" else np.uint16)
    for c0 in range(0, count, _CHUNK):
        c1 = min(count, c0 + _CHUNK)
        u = uniform_host(key, 2 * (start + c0), 2 * (c1 - c0))
        z = np.sqrt(-2.0 * np.log(u[0::2])) * np.cos(2.0 * math.pi * u[1::2])
        v = (scale * z).astype(np.float32)
        out[c0:c1] = v if dtype == "f32" else f32_to_bf16_bits(v)
    return out.reshape(shape)


def _signed(c: int) -> int:
    return c - (1 << 64) if c >= (1 << 63) else c


def _lsr(z, s: int):
    """Logical right shift of an int64 torch tensor viewed as uint64."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix64_torch(z):
    z = z ^ _lsr(z, 30)
    z = z * _signed(_C1)
    z = z ^ _lsr(z, 27)
    z = z * _signed(_C2)
    return z ^ _lsr(z, 31)


def normal_torch(seed: int, name: str, shape, scale: float = 1.0, dtype: str = "f32",
                 device="cpu", start: int = 0, chunk: int = 1 << 26):
    """Same stream as `normal_host`, drawn with torch ops on `device`.

    Returns a torch.float32 or torch.bfloat16 tensor.
    """
    import torch

    shape = tuple(int(d) for d in shape)
    count = 1
    for d in shape:
        count *= d
    key = _signed(stream_key(seed, name))
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]
    out = torch.empty(count, dtype=tdt, device=device)
    g = _signed(GOLDEN)
    for c0 in range(0, count, chunk):
        c1 = min(count, c0 + chunk)
        n = torch.arange(2 * (start + c0), 2 * (start + c1), dtype=torch.int64, device=device)
        b = _mix64_torch(key + (n + 1) * g)
        u = (_lsr(b, 11).to(torch.float64) + 0.5) * (2.0 ** -53)
        del n, b
        z = torch.sqrt(-2.0 * torch.log(u[0::2])) * torch.cos(2.0 * math.pi * u[1::2])
        del u
        out[c0:c1] = (scale * z).to(torch.float32).to(tdt)
        del z
    return out.view(shape)
