"""The allocation-free capacity entry point, checked against the regular one.

moe_capacity_locations_noalloc serves callers that cannot allocate device
memory themselves (a plugin inside an engine that owns the whole device
memory pool, or a path where cudaMalloc's implicit synchronisation is not
acceptable): its scratch lives in a fixed 1 MiB array inside the library.
This file is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

import combine_moe_gate_gb300 as M

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 1 << 20  # MOE_CAPACITY_NOALLOC_SCRATCH_BYTES


def _noalloc_fn():
    lib = M.load()
    fn = lib.moe_capacity_locations_noalloc
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.argtypes = [P, I64, I, I, ctypes.c_float, I64, P, P, P, P, P]
    fn.restype = I
    return fn


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _routing(seed, s, e, k, skew):
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((s, e)) - skew * np.log(np.arange(1, e + 1))
    idx = np.argsort(-lg, axis=1, kind="stable")[:, :k].T.copy()
    return torch.from_numpy(idx.astype(np.int32)).cuda()


def _with_workspace(idx, e, f, c_max):
    k, s = idx.shape
    ws = torch.empty(M.moe_capacity_workspace_size(s, e, k), dtype=torch.uint8, device="cuda")
    out = [torch.full((k, s), -1, dtype=torch.int32, device="cuda"),
           torch.full((e,), -1, dtype=torch.int32, device="cuda"),
           torch.full((1,), -1, dtype=torch.int32, device="cuda"),
           torch.zeros(1, dtype=torch.int32, device="cuda")]
    M.moe_capacity_locations(idx, e, f, c_max, ws, *out)
    return out


def _noalloc(fn, idx, e, f, c_max):
    k, s = idx.shape
    out = [torch.full((k, s), -1, dtype=torch.int32, device="cuda"),
           torch.full((e,), -1, dtype=torch.int32, device="cuda"),
           torch.full((1,), -1, dtype=torch.int32, device="cuda"),
           torch.zeros(1, dtype=torch.int32, device="cuda")]
    st = fn(_ptr(idx), s, e, k, f, c_max, *[_ptr(t) for t in out],
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == M.MOE_OK, M.status_str(st)
    return out


def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    fn = _noalloc_fn()
    cases = [(1, 16384, 256, 8, -1.5, 2.0), (2, 9000, 64, 2, 0.0, 1.2)]
    for seed, s, e, k, f, skew in cases:   # two calls in a row, different shapes and data
        idx = _routing(seed, s, e, k, skew)
        c_max = M.moe_capacity_bound(f, s, e, k)
        want = _with_workspace(idx, e, f, c_max)
        got = _noalloc(fn, idx, e, f, c_max)
        torch.cuda.synchronize()
        for g, w in zip(got, want):       # integer outputs: bit-exact
            assert torch.equal(g, w)
        assert int(got[3].item()) == 0


def test_noalloc_rejects_shapes_beyond_the_scratch_limit():
    fn = _noalloc_fn()
    e, k = 1024, 32
    s = (SCRATCH_BYTES // 4 // e + 1) * 4096 // k   # one chunk more than the array holds
    assert M.moe_capacity_workspace_size(s, e, k) > SCRATCH_BYTES
    idx = torch.zeros((k, s), dtype=torch.int32, device="cuda")
    out = [torch.empty((k, s), dtype=torch.int32, device="cuda"),
           torch.empty((e,), dtype=torch.int32, device="cuda"),
           torch.empty((1,), dtype=torch.int32, device="cuda"),
           torch.zeros(1, dtype=torch.int32, device="cuda")]
    before = M.launch_count()
    st = fn(_ptr(idx), s, e, k, 1.0, 1 << 20, *[_ptr(t) for t in out],
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == M.MOE_ERR_UNSUPPORTED
    assert M.launch_count() == before
