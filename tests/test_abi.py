"""The C ABI on the host: the library loads and exports every symbol the header
declares; host-side logic (capacity bound, workspace sizes, argument checks)
behaves as documented.  No call here reaches a kernel launch."""

import ctypes
import json
import os

import numpy as np
import pytest
import torch

import combine_moe_gate_gb300 as M
import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_library_exports_every_declared_symbol():
    lib = M.load()
    names = M.declared_symbols()
    assert len(names) >= 14
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # exported with C linkage: visible to a plain dlsym by the unmangled name
    raw = ctypes.CDLL(M.LIB_PATH)
    for n in names:
        ctypes.cast(getattr(raw, n), ctypes.c_void_p)


def test_status_strings():
    assert M.status_str(M.MOE_OK) == "ok"
    assert "c_max" in M.status_str(M.MOE_ERR_CAPACITY)
    assert M.status_str(99) == "unknown status"


def test_debug_stall_hook_arguments():
    lib = M.load()
    assert lib.moe_debug_stall_gemms(-1) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_debug_stall_gemms(3) == M.MOE_OK
    assert lib.moe_debug_stall_gemms(0) == M.MOE_OK   # cancels: no GEMM launch stalls after this
    with pytest.raises(M.MoEError):
        M.moe_debug_stall_gemms(-2)
    assert "timed out" in M.status_str(M.MOE_ERR_TIMEOUT)


def test_capacity_bound_matches_closed_forms():
    with open(os.path.join(GOLD, "capacity.json")) as f:
        cap = json.load(f)
    for c in cap["fixed"]:
        assert M.moe_capacity_bound(c["f"], c["s"], c["e"], c["k"]) == c["c"]
    for c in cap["capped_bound"]:
        assert M.moe_capacity_bound(c["f"], c["s"], c["e"], c["k"]) == c["bound"]
    assert M.moe_capacity_bound(0.0, 8192, 16, 3) == 8192       # no-drop: at most s per expert
    assert M.moe_capacity_bound(-100.0, 50, 2, 2) == 50          # capped by s
    assert M.moe_capacity_bound(1.0, 10, 4, 5) == -1             # k > e: invalid


@pytest.mark.parametrize("f", [0.3, 1.0, 1.25, 1.7, 2.0, 3.3])
def test_capacity_bound_agrees_with_oracle(f):
    rng = np.random.default_rng(int(f * 10))
    for _ in range(50):
        e = int(rng.integers(1, 300))
        k = int(rng.integers(1, min(e, 32) + 1))
        s = int(rng.integers(1, 100000))
        want = oracle.capacity(f, s, e, k, np.zeros(e, np.int64))
        assert M.moe_capacity_bound(f, s, e, k) == want


def test_workspace_sizes():
    ws = M.moe_capacity_workspace_size(16384, 256, 8)
    assert ws >= 32 * 256 * 4 and ws % 256 == 0
    h = M.moe_expert_ffn_workspace_size(M.MOE_BF16, "gelu", 8, 1280, 1024, 4096)
    assert h == 8 * 1280 * 4096 * 2
    assert M.moe_layer_workspace_size(M.MOE_BF16, "gelu", 4096, 1024, 8, 2, 1280, 4096) >= h + 256
    assert M.moe_expert_ffn_workspace_size(7, "gelu", 8, 1280, 1024, 4096) == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake device pointers are only safe without a GPU")
def test_invalid_arguments_are_rejected_before_launch():
    lib = M.load()
    before = M.launch_count()
    A = ctypes.c_void_p(0x10000)      # 16-byte aligned fake addresses (never dereferenced)
    B = ctypes.c_void_p(0x20000)
    odd = ctypes.c_void_p(0x30004)
    INV = M.MOE_ERR_INVALID_ARG
    gate = lib.moe_gate_topk
    # k > e, k = 0, s = 0, m not a multiple of 8 for bf16, NULL / misaligned x
    assert gate(A, M.MOE_BF16, B, None, 10, 64, 4, 5, 0, A, B, A, None) == INV
    assert gate(A, M.MOE_BF16, B, None, 10, 64, 4, 0, 0, A, B, A, None) == INV
    assert gate(A, M.MOE_BF16, B, None, 0, 64, 4, 1, 0, A, B, A, None) == INV
    assert gate(A, M.MOE_BF16, B, None, 10, 60, 4, 1, 0, A, B, A, None) == INV
    assert gate(None, M.MOE_BF16, B, None, 10, 64, 4, 1, 0, A, B, A, None) == INV
    assert gate(odd, M.MOE_BF16, B, None, 10, 64, 4, 1, 0, A, B, A, None) == INV
    assert gate(A, 5, B, None, 10, 64, 4, 1, 0, A, B, A, None) == INV
    assert gate(A, M.MOE_BF16, B, None, 10, 64, 4, 1, 8, A, B, A, None) == INV  # unknown flag
    cap = lib.moe_capacity_locations
    assert cap(A, 100, 4, 2, 1.0, 0, A, 1 << 20, A, A, A, A, None) == INV        # c_max = 0
    assert cap(A, 100, 4, 2, 1.0, 50, A, 0, A, A, A, A, None) == INV             # workspace too small
    assert cap(A, 100, 4, 2, float("nan"), 50, A, 1 << 20, A, A, A, A, None) == INV
    # the allocation-free variant: idx, s, e, k, f, c_max, loc, counts, c_dev, status, stream
    na = lib.moe_capacity_locations_noalloc
    nok = (A, 100, 4, 2, 1.0, 50, A, B, A, B, None)
    def nac(**kw):
        a = list(nok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return na(*a)
    assert nac(a5=0) == INV                                      # c_max < 1
    assert nac(a5=1 << 31) == INV                                # c_max beyond int32
    assert nac(a4=float("nan")) == INV                           # NaN capacity factor
    assert nac(a3=5) == INV and nac(a3=0) == INV                 # k > e, k = 0
    assert nac(a2=0) == INV and nac(a2=2000) == INV              # e = 0, e > 1024
    assert nac(a1=0) == INV                                      # s = 0
    for i in (0, 6, 7, 8, 9):                                    # idx, loc, counts, c_dev, status
        assert nac(**{f"a{i}": None}) == INV
        assert nac(**{f"a{i}": ctypes.c_void_p(0x30002)}) == INV # not 4-byte aligned
    # the pipelined layer: ..., dev_status, chunks, stream, aux_stream, events
    pl = lib.moe_layer_forward_pipelined
    ev = (ctypes.c_void_p * 3)(A, B, A)
    pok = [A, M.MOE_BF16, B, None, A, None, None, A, None, 1, 64, 64, 8, 2, 128, 1.0, 16, 0,
           A, B, A, B, A, A, B, A, A, 1 << 30, A, 2, None, None, ev]
    def plc(**kw):
        a = list(pok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return pl(*a)
    assert plc(a29=0) == INV and plc(a29=65) == INV             # chunks outside [1, 64]
    assert plc(a32=None) == INV                                  # events required
    assert plc(a32=(ctypes.c_void_p * 3)(A, None, A)) == INV     # every event required
    assert plc(a27=0) == INV                                     # workspace too small
    assert plc(a0=odd) == INV and plc(a25=odd) == INV            # misaligned x / y
    ffn = lib.moe_expert_ffn
    # SwiGLU takes no biases and needs w3
    assert ffn(A, M.MOE_BF16, A, A, A, B, A, A, None, 2, 4, 64, 64, 64, A, 1 << 30, A, A, None) == INV
    assert ffn(A, M.MOE_BF16, A, A, A, None, None, A, None, 2, 4, 64, 64, 64, A, 1 << 30, A, A, None) == INV
    assert ffn(A, M.MOE_BF16, A, A, A, None, None, A, None, 7, 4, 64, 64, 64, A, 1 << 30, A, A, None) == INV
    dec = lib.moe_decode
    assert dec(A, M.MOE_F32, A, A, A, A, 10, 6, 4, 1, 8, A, A, None) == INV    # m % 4 != 0 (fp32)
    enc = lib.moe_encode
    assert enc(A, M.MOE_BF16, A, A, None, A, 10, 64, 4, 1, 8, M.MOE_FLAG_ZERO_FILL, A, A, None) == INV
    # gate backward: x, wg, bias, s, m, e, k, flags, idx, gates, d_gates, d_logits,
    # d_wg, d_bias, d_x, status, stream
    gbwd = lib.moe_gate_bwd
    ok = (A, M.MOE_BF16, B, None, 10, 64, 8, 2, 1, A, B, A, B, None, None, None, A, None)
    def gb(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return gbwd(*a)
    assert gb(a6=300) == M.MOE_ERR_UNSUPPORTED                   # e > 256
    assert gb(a7=9) == INV                                       # k > e
    assert gb(a5=60) == INV                                      # bf16 rows not a multiple of 8
    assert gb(a8=4) == INV                                       # unknown flag
    assert gb(a0=odd) == INV and gb(a2=odd) == INV               # misaligned x / wg
    assert gb(a12=None) == INV                                   # d_logits is required
    assert gb(a11=None) == INV and gb(a10=None) == INV           # d_gates, gates are required
    assert gb(a13=odd) == INV and gb(a15=odd) == INV             # misaligned d_wg / d_x
    assert gb(a3=odd) == INV                                     # misaligned bias
    dbwd = lib.moe_decode_bwd
    # dy, out, dt, idx, loc, gates, counts, c_dev, s, m, e, k, c_max, flags, d_out, d_gates, status
    assert dbwd(A, A, M.MOE_BF16, A, A, A, None, A, 10, 64, 4, 1, 0, 0, A, A, A, None) == INV
    assert dbwd(A, A, M.MOE_BF16, A, A, A, None, A, 10, 64, 4, 1, 8, M.MOE_FLAG_ZERO_FILL, A, A, A,
                None) == INV                                     # zero fill needs counts
    assert dbwd(odd, A, M.MOE_BF16, A, A, A, None, A, 10, 64, 4, 1, 8, 0, A, A, A, None) == INV
    ebwd = lib.moe_encode_bwd
    # d_buf, dt, idx, loc, c_dev, s, m, e, k, c_max, dx, status
    assert ebwd(A, M.MOE_BF16, A, A, A, 10, 64, 4, 5, 8, A, A, None) == INV      # k > e
    assert ebwd(A, M.MOE_BF16, A, A, A, 10, 64, 4, 1, 8, odd, A, None) == INV    # misaligned dx
    fb = lib.moe_expert_ffn_bwd
    # buf, hid, dt, counts, c_dev, w1, b1, w3, w2, act, e, c_max, m, h, d_out, ws, ws_bytes,
    # d_buf, d_w1, d_w3, d_w2, d_b1, d_b2, status, stream
    fok = [A, B, M.MOE_BF16, A, A, A, None, None, B, 1, 4, 64, 64, 128, A, B, 1 << 40, A, B, None,
           A, None, None, A, None]
    def fbc(**kw):
        a = list(fok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return fb(*a)
    assert fbc(a2=M.MOE_F32) == M.MOE_ERR_UNSUPPORTED           # bf16 only
    assert fbc(a9=2) == INV                                      # SwiGLU needs w3 and d_w3
    assert fbc(a9=2, a7=A, a19=B, a6=A) == INV                   # ... and takes no bias
    assert fbc(a16=0) == INV                                     # workspace too small
    assert fbc(a13=100) == INV                                   # h not a multiple of 8
    assert fbc(a1=odd) == INV and fbc(a17=odd) == INV            # misaligned hid / d_buf
    # the saved-pre backward: buf, hid, pre, dt, counts, c_dev, w1, w3, w2, act, e, c_max, m, h,
    # d_out, ws, ws_bytes, d_buf, wgrad_dt, d_w1, d_w3, d_w2, d_b1, d_b2, status, stream
    fs = lib.moe_expert_ffn_bwd_saved
    sok = [A, B, A, M.MOE_BF16, A, A, A, None, B, 1, 4, 64, 64, 128, A, B, 1 << 40, A, M.MOE_F32,
           B, None, A, None, None, A, None]
    def fsc(**kw):
        a = list(sok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return fs(*a)
    assert fsc(a2=None) == INV and fsc(a2=odd) == INV            # pre required, aligned
    assert fsc(a9=2) == INV                                      # SwiGLU needs w3 and d_w3
    assert fsc(a3=M.MOE_F32) == M.MOE_ERR_UNSUPPORTED
    assert fsc(a16=0) == INV                                     # workspace too small
    assert fsc(a18=7) == INV                                     # weight gradients bf16 or fp32
    assert fsc(a19=odd) == INV                                   # misaligned d_w1
    # the training forward: buf, dt, counts, c_dev, w1, b1, w3, w2, b2, act, e, c_max, m, h, ws,
    # ws_bytes, out, pre, status, stream
    ft = lib.moe_expert_ffn_train
    tok = [A, M.MOE_BF16, A, A, A, None, None, B, None, 1, 4, 64, 64, 128, A, 1 << 40, B, A, A, None]
    def ftc(**kw):
        a = list(tok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return ft(*a)
    assert ftc(a17=None) == INV and ftc(a17=odd) == INV          # pre required, aligned
    assert ftc(a9=2) == INV                                      # SwiGLU needs w3 (none here)
    assert ftc(a1=M.MOE_F32) == M.MOE_ERR_UNSUPPORTED            # bf16 only
    assert ftc(a15=0) == INV                                     # workspace too small
    # e4m3 row quantisation: src, batches, rows_per_batch, cols, counts, c_dev, q, scale, status
    qr = lib.moe_quantize_rows_fp8
    qok = [A, 2, 8, 64, None, None, B, A, B, None]
    def qrc(**kw):
        a = list(qok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return qr(*a)
    assert qrc(a3=40) == INV and qrc(a3=0) == INV                # cols not a multiple of 16
    assert qrc(a1=0) == INV and qrc(a2=0) == INV                 # no rows
    assert qrc(a4=A) == INV                                      # counts without c_dev
    assert qrc(a0=odd) == INV and qrc(a6=odd) == INV             # misaligned src / codes
    assert qrc(a7=None) == INV                                   # scales required
    # e4m3 experts: buf_q, buf_scale, counts, c_dev, w1_q, w1_scale, b1, w2_q, w2_scale, b2,
    # act, e, c_max, m, h, ws, ws_bytes, out, status, stream
    f8 = lib.moe_expert_ffn_fp8
    f8ok = [A, A, A, A, B, A, None, B, A, None, 1, 4, 64, 64, 128, A, 1 << 40, B, A, None]
    def f8c(**kw):
        a = list(f8ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f8(*a)
    assert f8c(a10=2) == M.MOE_ERR_UNSUPPORTED                  # SwiGLU
    assert f8c(a13=72) == INV and f8c(a14=40) == INV             # m, h not multiples of 16
    assert f8c(a16=0) == INV                                     # workspace too small
    assert f8c(a0=odd) == INV and f8c(a17=odd) == INV            # misaligned codes / out
    assert f8c(a5=odd) == INV                                    # misaligned weight scales
    assert M.moe_expert_ffn_fp8_workspace_size(4, 64, 64, 128) >= 4 * 64 * 128 * 3 + 4 * 64 * 4
    assert M.moe_expert_ffn_fp8_workspace_size(4, 64, 72, 128) == 0
    assert M.launch_count() == before
