"""GB300-native top-k MoE layer hot path: Python binding of libmoe_gate.so.

Every step runs in the CUDA library (include/moe_gate.h); this module only
marshals torch tensors into the C ABI: data pointers, sizes taken from the
tensor shapes, the current CUDA stream.  There is no fallback: if the library
is missing, importing the entry points raises.

Functions keep the C names:
    moe_gate_topk, moe_capacity_locations, moe_capacity_locations_noalloc,
    moe_encode, moe_expert_ffn,
    moe_decode, moe_decode_bwd, moe_encode_bwd, moe_layer_forward, moe_gate_bwd
plus the size queries and `MoEError`.
"""

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmoe_gate.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "moe_gate.h")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_CAPACITY, MOE_ERR_TIMEOUT = range(6)
MOE_F32, MOE_BF16 = 0, 1
ACT = {"relu": 0, "gelu": 1, "swiglu": 2}
MOE_FLAG_NORMALIZE_GATES = 1
MOE_FLAG_ZERO_FILL = 2

_lib = None


class MoEError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {status_str(code)} ({code})")


def load():
    """Load libmoe_gate.so (build it first with combine_moe_gate_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                           "(run `python -m combine_moe_gate_gb300.build`)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, I64, U, F, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint,
                           ctypes.c_float, ctypes.c_size_t)
    sigs = {
        "moe_gate_topk": (I, [P, I, P, P, I64, I, I, I, U, P, P, P, P]),
        "moe_gate_bwd": (I, [P, I, P, P, I64, I, I, I, U, P, P, P, P, P, P, P, P, P]),
        "moe_capacity_bound": (I64, [F, I64, I, I]),
        "moe_capacity_workspace_size": (SZ, [I64, I, I]),
        "moe_capacity_locations": (I, [P, I64, I, I, F, I64, P, SZ, P, P, P, P, P]),
        "moe_capacity_locations_noalloc": (I, [P, I64, I, I, F, I64, P, P, P, P, P]),
        "moe_encode": (I, [P, I, P, P, P, P, I64, I, I, I, I64, U, P, P, P]),
        "moe_expert_ffn_workspace_size": (SZ, [I, I, I, I64, I, I]),
        "moe_expert_ffn": (I, [P, I, P, P, P, P, P, P, P, I, I, I64, I, I, P, SZ, P, P, P]),
        "moe_expert_ffn_train": (I, [P, I, P, P, P, P, P, P, P, I, I, I64, I, I, P, SZ, P, P, P, P]),
        "moe_expert_ffn_bwd_workspace_size": (SZ, [I, I, I, I64, I, I]),
        "moe_expert_ffn_bwd": (I, [P, P, I, P, P, P, P, P, P, I, I, I64, I, I, P, P, SZ, P, P, P,
                                   P, P, P, P, P]),
        "moe_expert_ffn_bwd_saved": (I, [P, P, P, I, P, P, P, P, P, I, I, I64, I, I, P, P, SZ, P, I,
                                         P, P, P, P, P, P, P]),
        "moe_decode": (I, [P, I, P, P, P, P, I64, I, I, I, I64, P, P, P]),
        "moe_decode_bwd": (I, [P, P, I, P, P, P, P, P, I64, I, I, I, I64, U, P, P, P, P]),
        "moe_encode_bwd": (I, [P, I, P, P, P, I64, I, I, I, I64, P, P, P]),
        "moe_layer_workspace_size": (SZ, [I, I, I64, I, I, I, I64, I]),
        "moe_layer_forward": (I, [P, I, P, P, P, P, P, P, P, I, I64, I, I, I, I, F, I64, U,
                                  P, P, P, P, P, P, P, P, P, SZ, P, P]),
        "moe_layer_forward_host": (I, [P, P, P, I, P, P, P, P, P, P, P, I, I64, I, I, I, I, F, I64,
                                       U, P, P, P, P, P, P, P, P, P, SZ, P, P]),
        "moe_layer_forward_pipelined": (I, [P, I, P, P, P, P, P, P, P, I, I64, I, I, I, I, F, I64,
                                            U, P, P, P, P, P, P, P, P, P, SZ, P, I, P, P, P]),
        "moe_probe_fp32_fma": (I, [I, I, I, P, P]),
        "moe_quantize_rows_fp8": (I, [P, I64, I64, I, P, P, P, P, P, P]),
        "moe_expert_ffn_fp8_workspace_size": (SZ, [I, I64, I, I]),
        "moe_expert_ffn_fp8": (I, [P, P, P, P, P, P, P, P, P, P, I, I, I64, I, I, P, SZ, P, P, P]),
        "moe_status_str": (ctypes.c_char_p, [I]),
        "moe_launch_count": (ctypes.c_uint64, []),
        "moe_debug_stall_gemms": (I, [I]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def declared_symbols():
    """Names of the functions include/moe_gate.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(moe_\w+)\s*\(", text, re.M)))


def status_str(code) -> str:
    return load().moe_status_str(int(code)).decode()


def launch_count() -> int:
    return int(load().moe_launch_count())


def moe_debug_stall_gemms(n):
    """Error-path test hook: the next n tensor-core GEMM launches issue no
    operand copies, so each times out after about a second with
    MOE_ERR_TIMEOUT in its status word (n = 0 cancels)."""
    _check(load().moe_debug_stall_gemms(int(n)), "moe_debug_stall_gemms")


def _ptr(t, name="tensor", dtype=None, shape=None):
    """Device address of a contiguous CUDA tensor; checks the dtype and shape
    when given (a mismatch here would let a kernel read or write out of
    bounds).  None passes through as NULL."""
    if t is None:
        return None
    if shape is not None and tuple(t.shape) != tuple(int(d) for d in shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if not _on_device(t):
        raise ValueError(f"{name}: must be a CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _on_device(t) -> bool:
    return t.is_cuda


def _i32():
    import torch

    return torch.int32


def _f32():
    import torch

    return torch.float32


def _dt(t):
    import torch

    if t.dtype == torch.bfloat16:
        return MOE_BF16
    if t.dtype == torch.float32:
        return MOE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code, where):
    if code != MOE_OK:
        raise MoEError(code, where)


def _act(act):
    return ACT[act] if isinstance(act, str) else int(act)


# ------------------------------------------------------------------ sizes
def moe_capacity_bound(capacity_factor, s, e, k) -> int:
    return int(load().moe_capacity_bound(float(capacity_factor), int(s), int(e), int(k)))


def moe_capacity_workspace_size(s, e, k) -> int:
    return int(load().moe_capacity_workspace_size(int(s), int(e), int(k)))


def moe_expert_ffn_workspace_size(dtype, act, e, c_max, m, h) -> int:
    return int(load().moe_expert_ffn_workspace_size(int(dtype), _act(act), int(e), int(c_max),
                                                    int(m), int(h)))


def moe_expert_ffn_bwd_workspace_size(dtype, act, e, c_max, m, h) -> int:
    return int(load().moe_expert_ffn_bwd_workspace_size(int(dtype), _act(act), int(e), int(c_max),
                                                        int(m), int(h)))


def moe_layer_workspace_size(dtype, act, s, m, e, k, c_max, h) -> int:
    return int(load().moe_layer_workspace_size(int(dtype), _act(act), int(s), int(m), int(e),
                                               int(k), int(c_max), int(h)))


# ------------------------------------------------------------ entry points
def moe_gate_topk(x, wg, bias, k, idx, gates, dev_status, flags=0, stream=None):
    """x [s, m]; wg [m, e] fp32; bias [e] fp32 or None -> idx [k, s] int32, gates [k, s] fp32."""
    s, m = x.shape
    e = wg.shape[1]
    k = int(k)
    I, F = _i32(), _f32()
    _check(load().moe_gate_topk(
        _ptr(x, "x"), _dt(x), _ptr(wg, "wg", F, (m, e)), _ptr(bias, "bias", F, (e,)), s, m, e, k,
        int(flags), _ptr(idx, "idx", I, (k, s)), _ptr(gates, "gates", F, (k, s)),
        _ptr(dev_status, "dev_status", I), _stream(stream)), "moe_gate_topk")


def moe_capacity_locations(idx, e, capacity_factor, c_max, workspace, loc, counts, c_dev,
                           dev_status, stream=None):
    k, s = idx.shape
    I = _i32()
    _check(load().moe_capacity_locations(
        _ptr(idx, "idx", I), s, int(e), k, float(capacity_factor), int(c_max),
        _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _ptr(loc, "loc", I, (k, s)), _ptr(counts, "counts", I, (int(e),)),
        _ptr(c_dev, "c_dev", I), _ptr(dev_status, "dev_status", I), _stream(stream)),
        "moe_capacity_locations")


def moe_capacity_locations_noalloc(idx, e, capacity_factor, c_max, loc, counts, c_dev,
                                   dev_status, stream=None):
    """moe_capacity_locations with its scratch in the library's fixed device
    array (for callers that cannot allocate device memory); see the header."""
    k, s = idx.shape
    I = _i32()
    _check(load().moe_capacity_locations_noalloc(
        _ptr(idx, "idx", I), s, int(e), k, float(capacity_factor), int(c_max),
        _ptr(loc, "loc", I, (k, s)), _ptr(counts, "counts", I, (int(e),)),
        _ptr(c_dev, "c_dev", I), _ptr(dev_status, "dev_status", I), _stream(stream)),
        "moe_capacity_locations_noalloc")


def moe_encode(x, idx, loc, counts, c_dev, buf, dev_status, flags=0, stream=None):
    """buf is [e, c_max, m]."""
    s, m = x.shape
    k = idx.shape[0]
    e, c_max, _ = buf.shape
    I = _i32()
    _check(load().moe_encode(
        _ptr(x, "x"), _dt(x), _ptr(idx, "idx", I, (k, s)), _ptr(loc, "loc", I, (k, s)),
        _ptr(counts, "counts", I, (e,)), _ptr(c_dev, "c_dev", I), s, m, e, k, c_max, int(flags),
        _ptr(buf, "buf", x.dtype, (e, c_max, m)), _ptr(dev_status, "dev_status", I),
        _stream(stream)), "moe_encode")


def moe_expert_ffn(buf, counts, c_dev, w1, b1, w3, w2, b2, act, workspace, out, dev_status,
                   stream=None):
    e, c_max, m = buf.shape
    h = w1.shape[1]
    I, dt = _i32(), buf.dtype
    _check(load().moe_expert_ffn(
        _ptr(buf, "buf"), _dt(buf), _ptr(counts, "counts", I, (e,)), _ptr(c_dev, "c_dev", I),
        _ptr(w1, "w1", dt, (e, h, m)), _ptr(b1, "b1", dt, (e, h)), _ptr(w3, "w3", dt, (e, h, m)),
        _ptr(w2, "w2", dt, (e, m, h)), _ptr(b2, "b2", dt, (e, m)), _act(act), e, c_max, m, h,
        _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _ptr(out, "out", dt, (e, c_max, m)), _ptr(dev_status, "dev_status", I),
        _stream(stream)), "moe_expert_ffn")


def moe_expert_ffn_train(buf, counts, c_dev, w1, b1, w3, w2, b2, act, workspace, out, pre,
                         dev_status, stream=None):
    """moe_expert_ffn (bf16) that also keeps what moe_expert_ffn_bwd_saved
    needs: the pre-activation [e, c_max, h] (ReLU / GELU) or [a | b]
    [e, c_max, 2h] (SwiGLU)."""
    e, c_max, m = buf.shape
    h = w1.shape[1]
    I, dt = _i32(), buf.dtype
    hp = 2 * h if _act(act) == ACT["swiglu"] else h
    _check(load().moe_expert_ffn_train(
        _ptr(buf, "buf"), _dt(buf), _ptr(counts, "counts", I, (e,)), _ptr(c_dev, "c_dev", I),
        _ptr(w1, "w1", dt, (e, h, m)), _ptr(b1, "b1", dt, (e, h)), _ptr(w3, "w3", dt, (e, h, m)),
        _ptr(w2, "w2", dt, (e, m, h)), _ptr(b2, "b2", dt, (e, m)), _act(act), e, c_max, m, h,
        _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _ptr(out, "out", dt, (e, c_max, m)), _ptr(pre, "pre", dt, (e, c_max, hp)),
        _ptr(dev_status, "dev_status", I), _stream(stream)), "moe_expert_ffn_train")


def moe_expert_ffn_fp8_workspace_size(e, c_max, m, h) -> int:
    return int(load().moe_expert_ffn_fp8_workspace_size(int(e), int(c_max), int(m), int(h)))


def moe_quantize_rows_fp8(src, q, scale, dev_status, counts=None, c_dev=None, stream=None):
    """e4m3 codes (uint8, src's shape) and per-row fp32 scales of a bf16 tensor
    [rows, cols] or [batches, rows, cols]; with counts / c_dev only the kept
    rows of each batch."""
    import torch

    shape = tuple(src.shape) if src.dim() == 3 else (1,) + tuple(src.shape)
    b, r, c = shape
    I = _i32()
    _check(load().moe_quantize_rows_fp8(
        _ptr(src, "src", torch.bfloat16), b, r, c,
        _ptr(counts, "counts", I, (b,)) if counts is not None else None,
        _ptr(c_dev, "c_dev", I) if c_dev is not None else None,
        _ptr(q, "q", torch.uint8, tuple(src.shape)),
        _ptr(scale, "scale", _f32(), tuple(src.shape[:-1])), _ptr(dev_status, "dev_status", I),
        _stream(stream)), "moe_quantize_rows_fp8")


def moe_expert_ffn_fp8(buf_q, buf_scale, counts, c_dev, w1_q, w1_scale, b1, w2_q, w2_scale, b2,
                       act, workspace, out, dev_status, stream=None):
    import torch

    e, c_max, m = buf_q.shape
    h = w1_q.shape[1]
    I, F, U8, bf = _i32(), _f32(), torch.uint8, torch.bfloat16
    _check(load().moe_expert_ffn_fp8(
        _ptr(buf_q, "buf_q", U8), _ptr(buf_scale, "buf_scale", F, (e, c_max)),
        _ptr(counts, "counts", I, (e,)), _ptr(c_dev, "c_dev", I),
        _ptr(w1_q, "w1_q", U8, (e, h, m)), _ptr(w1_scale, "w1_scale", F, (e, h)),
        _ptr(b1, "b1", bf, (e, h)), _ptr(w2_q, "w2_q", U8, (e, m, h)),
        _ptr(w2_scale, "w2_scale", F, (e, m)), _ptr(b2, "b2", bf, (e, m)), _act(act), e, c_max,
        m, h, _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _ptr(out, "out", bf, (e, c_max, m)), _ptr(dev_status, "dev_status", I), _stream(stream)),
        "moe_expert_ffn_fp8")


def moe_expert_ffn_bwd(buf, hid, counts, c_dev, w1, b1, w3, w2, act, d_out, workspace, d_buf,
                       d_w1, d_w3, d_w2, d_b1, d_b2, dev_status, stream=None):
    """Gradient of moe_expert_ffn over the kept rows (bf16); hid is the
    forward's hidden (its workspace after the call)."""
    e, c_max, m = buf.shape
    h = w1.shape[1]
    I, dt = _i32(), buf.dtype
    _check(load().moe_expert_ffn_bwd(
        _ptr(buf, "buf"), _ptr(hid, "hid", dt, (e, c_max, h)), _dt(buf),
        _ptr(counts, "counts", I, (e,)), _ptr(c_dev, "c_dev", I), _ptr(w1, "w1", dt, (e, h, m)),
        _ptr(b1, "b1", dt, (e, h)), _ptr(w3, "w3", dt, (e, h, m)), _ptr(w2, "w2", dt, (e, m, h)),
        _act(act), e, c_max, m, h, _ptr(d_out, "d_out", dt, (e, c_max, m)),
        _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _ptr(d_buf, "d_buf", dt, (e, c_max, m)), _ptr(d_w1, "d_w1", dt, (e, h, m)),
        _ptr(d_w3, "d_w3", dt, (e, h, m)), _ptr(d_w2, "d_w2", dt, (e, m, h)),
        _ptr(d_b1, "d_b1", dt, (e, h)), _ptr(d_b2, "d_b2", dt, (e, m)),
        _ptr(dev_status, "dev_status", I), _stream(stream)), "moe_expert_ffn_bwd")


def moe_expert_ffn_bwd_saved(buf, hid, pre, counts, c_dev, w1, w3, w2, act, d_out, workspace,
                             d_buf, d_w1, d_w3, d_w2, d_b1, d_b2, dev_status, stream=None):
    """moe_expert_ffn_bwd with what moe_expert_ffn_train kept: nothing is
    recomputed.  The weight and bias gradients are all bf16 or all fp32
    (kept in fp32); w3 / d_w3 for SwiGLU only."""
    import torch

    e, c_max, m = buf.shape
    h = w1.shape[1]
    I, dt = _i32(), buf.dtype
    hp = 2 * h if _act(act) == ACT["swiglu"] else h
    gdt = d_w1.dtype
    if gdt not in (torch.bfloat16, torch.float32):
        raise ValueError(f"d_w1: dtype {gdt}, expected bfloat16 or float32")
    _check(load().moe_expert_ffn_bwd_saved(
        _ptr(buf, "buf"), _ptr(hid, "hid", dt, (e, c_max, h)),
        _ptr(pre, "pre", dt, (e, c_max, hp)), _dt(buf), _ptr(counts, "counts", I, (e,)),
        _ptr(c_dev, "c_dev", I), _ptr(w1, "w1", dt, (e, h, m)), _ptr(w3, "w3", dt, (e, h, m)),
        _ptr(w2, "w2", dt, (e, m, h)), _act(act), e, c_max, m, h,
        _ptr(d_out, "d_out", dt, (e, c_max, m)),
        _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _ptr(d_buf, "d_buf", dt, (e, c_max, m)), _dt(d_w1), _ptr(d_w1, "d_w1", gdt, (e, h, m)),
        _ptr(d_w3, "d_w3", gdt, (e, h, m)),
        _ptr(d_w2, "d_w2", gdt, (e, m, h)), _ptr(d_b1, "d_b1", gdt, (e, h)),
        _ptr(d_b2, "d_b2", gdt, (e, m)), _ptr(dev_status, "dev_status", I), _stream(stream)),
        "moe_expert_ffn_bwd_saved")


def moe_decode(out, idx, loc, gates, c_dev, y, dev_status, stream=None):
    e, c_max, m = out.shape
    k, s = idx.shape
    I, F = _i32(), _f32()
    _check(load().moe_decode(
        _ptr(out, "out"), _dt(out), _ptr(idx, "idx", I), _ptr(loc, "loc", I, (k, s)),
        _ptr(gates, "gates", F, (k, s)), _ptr(c_dev, "c_dev", I), s, m, e, k, c_max,
        _ptr(y, "y", out.dtype, (s, m)), _ptr(dev_status, "dev_status", I), _stream(stream)),
        "moe_decode")


def moe_decode_bwd(dy, out, idx, loc, gates, counts, c_dev, d_out, d_gates, dev_status, flags=0,
                   stream=None):
    e, c_max, m = out.shape
    k, s = idx.shape
    I, F, dt = _i32(), _f32(), out.dtype
    _check(load().moe_decode_bwd(
        _ptr(dy, "dy", dt, (s, m)), _ptr(out, "out"), _dt(out), _ptr(idx, "idx", I),
        _ptr(loc, "loc", I, (k, s)), _ptr(gates, "gates", F, (k, s)),
        _ptr(counts, "counts", I, (e,)), _ptr(c_dev, "c_dev", I), s, m, e, k, c_max, int(flags),
        _ptr(d_out, "d_out", dt, (e, c_max, m)), _ptr(d_gates, "d_gates", F, (k, s)),
        _ptr(dev_status, "dev_status", I), _stream(stream)), "moe_decode_bwd")


def moe_gate_bwd(x, wg, bias, idx, gates, d_gates, d_logits, dev_status, d_wg=None, d_bias=None,
                 d_x=None, flags=0, stream=None):
    """Gate backward: d_gates [k, s] fp32 -> d_logits [s, e] and, when given,
    d_wg [m, e], d_bias [e], d_x [s, m] (all fp32)."""
    s, m = x.shape
    e = wg.shape[1]
    k = idx.shape[0]
    I, F = _i32(), _f32()
    _check(load().moe_gate_bwd(
        _ptr(x, "x"), _dt(x), _ptr(wg, "wg", F, (m, e)), _ptr(bias, "bias", F, (e,)), s, m, e, k,
        int(flags), _ptr(idx, "idx", I, (k, s)), _ptr(gates, "gates", F, (k, s)),
        _ptr(d_gates, "d_gates", F, (k, s)), _ptr(d_logits, "d_logits", F, (s, e)),
        _ptr(d_wg, "d_wg", F, (m, e)), _ptr(d_bias, "d_bias", F, (e,)),
        _ptr(d_x, "d_x", F, (s, m)), _ptr(dev_status, "dev_status", I), _stream(stream)),
        "moe_gate_bwd")


def moe_encode_bwd(d_buf, idx, loc, c_dev, dx, dev_status, stream=None):
    e, c_max, m = d_buf.shape
    k, s = idx.shape
    I = _i32()
    _check(load().moe_encode_bwd(
        _ptr(d_buf, "d_buf"), _dt(d_buf), _ptr(idx, "idx", I), _ptr(loc, "loc", I, (k, s)),
        _ptr(c_dev, "c_dev", I), s, m, e, k, c_max, _ptr(dx, "dx", d_buf.dtype, (s, m)),
        _ptr(dev_status, "dev_status", I), _stream(stream)), "moe_encode_bwd")


def moe_layer_forward(x, wg, gate_bias, w1, b1, w3, w2, b2, act, k, capacity_factor, flags,
                      idx, gates, loc, counts, c_dev, buf, out, y, workspace, dev_status,
                      stream=None):
    s, m = x.shape
    e, c_max, _ = buf.shape
    h = w1.shape[1]
    k = int(k)
    I, F, dt = _i32(), _f32(), x.dtype
    _check(load().moe_layer_forward(
        _ptr(x, "x"), _dt(x), _ptr(wg, "wg", F, (m, e)), _ptr(gate_bias, "gate_bias", F, (e,)),
        _ptr(w1, "w1", dt, (e, h, m)), _ptr(b1, "b1", dt, (e, h)), _ptr(w3, "w3", dt, (e, h, m)),
        _ptr(w2, "w2", dt, (e, m, h)), _ptr(b2, "b2", dt, (e, m)), _act(act), s, m, e, k, h,
        float(capacity_factor), c_max, int(flags), _ptr(idx, "idx", I, (k, s)),
        _ptr(gates, "gates", F, (k, s)), _ptr(loc, "loc", I, (k, s)),
        _ptr(counts, "counts", I, (e,)), _ptr(c_dev, "c_dev", I), _ptr(buf, "buf", dt, (e, c_max, m)),
        _ptr(out, "out", dt, (e, c_max, m)), _ptr(y, "y", dt, (s, m)), _ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _ptr(dev_status, "dev_status", I),
        _stream(stream)), "moe_layer_forward")


def moe_layer_forward_host(x_host, y_host, x, wg, gate_bias, w1, b1, w3, w2, b2, act, k,
                           capacity_factor, flags, idx, gates, loc, counts, c_dev, buf, out, y,
                           workspace, dev_status, stream=None):
    """moe_layer_forward with x read from, and y written to, host tensors
    (pinned for asynchronous copies); x and y are the device buffers."""
    s, m = x.shape
    e, c_max, _ = buf.shape
    h = w1.shape[1]
    k = int(k)
    I, F, dt = _i32(), _f32(), x.dtype
    for name, t in (("x_host", x_host), ("y_host", y_host)):
        if t.is_cuda or tuple(t.shape) != (s, m) or t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name}: must be a contiguous host tensor [{s}, {m}] of {dt}")
    _check(load().moe_layer_forward_host(
        ctypes.c_void_p(x_host.data_ptr()), ctypes.c_void_p(y_host.data_ptr()), _ptr(x, "x"), _dt(x),
        _ptr(wg, "wg", F, (m, e)), _ptr(gate_bias, "gate_bias", F, (e,)),
        _ptr(w1, "w1", dt, (e, h, m)), _ptr(b1, "b1", dt, (e, h)), _ptr(w3, "w3", dt, (e, h, m)),
        _ptr(w2, "w2", dt, (e, m, h)), _ptr(b2, "b2", dt, (e, m)), _act(act), s, m, e, k, h,
        float(capacity_factor), c_max, int(flags), _ptr(idx, "idx", I, (k, s)),
        _ptr(gates, "gates", F, (k, s)), _ptr(loc, "loc", I, (k, s)),
        _ptr(counts, "counts", I, (e,)), _ptr(c_dev, "c_dev", I), _ptr(buf, "buf", dt, (e, c_max, m)),
        _ptr(out, "out", dt, (e, c_max, m)), _ptr(y, "y", dt, (s, m)), _ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _ptr(dev_status, "dev_status", I),
        _stream(stream)), "moe_layer_forward_host")


def moe_layer_forward_pipelined(x, wg, gate_bias, w1, b1, w3, w2, b2, act, k, capacity_factor,
                                flags, idx, gates, loc, counts, c_dev, buf, out, y, workspace,
                                dev_status, chunks, aux_stream, events, stream=None):
    """moe_layer_forward with encode of capacity chunk i+1 (on aux_stream)
    overlapping the FFN of chunk i (on stream); events: 1 + chunks
    torch.cuda.Event objects."""
    s, m = x.shape
    e, c_max, _ = buf.shape
    h = w1.shape[1]
    k, chunks = int(k), int(chunks)
    if len(events) < chunks + 1:
        raise ValueError(f"events: need {chunks + 1}, got {len(events)}")
    for ev in events[:chunks + 1]:   # the handles exist once the events are recorded or created
        if getattr(ev, "cuda_event", 0) == 0:
            ev.record(torch_current_stream())
    handles = (ctypes.c_void_p * (chunks + 1))(*[ctypes.c_void_p(ev.cuda_event) for ev in
                                                 events[:chunks + 1]])
    I, F, dt = _i32(), _f32(), x.dtype
    _check(load().moe_layer_forward_pipelined(
        _ptr(x, "x"), _dt(x), _ptr(wg, "wg", F, (m, e)), _ptr(gate_bias, "gate_bias", F, (e,)),
        _ptr(w1, "w1", dt, (e, h, m)), _ptr(b1, "b1", dt, (e, h)), _ptr(w3, "w3", dt, (e, h, m)),
        _ptr(w2, "w2", dt, (e, m, h)), _ptr(b2, "b2", dt, (e, m)), _act(act), s, m, e, k, h,
        float(capacity_factor), c_max, int(flags), _ptr(idx, "idx", I, (k, s)),
        _ptr(gates, "gates", F, (k, s)), _ptr(loc, "loc", I, (k, s)),
        _ptr(counts, "counts", I, (e,)), _ptr(c_dev, "c_dev", I), _ptr(buf, "buf", dt, (e, c_max, m)),
        _ptr(out, "out", dt, (e, c_max, m)), _ptr(y, "y", dt, (s, m)), _ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _ptr(dev_status, "dev_status", I), chunks,
        _stream(stream), _stream(aux_stream), handles), "moe_layer_forward_pipelined")


def torch_current_stream():
    import torch

    return torch.cuda.current_stream()


def moe_probe_fp32_fma(packed, blocks, iters, out, stream=None):
    """Launch the fp32 FMA throughput probe (blocks * 256 * iters * 32 flop)."""
    _check(load().moe_probe_fp32_fma(int(bool(packed)), int(blocks), int(iters),
                                     _ptr(out, "out", _f32()), _stream(stream)), "moe_probe_fp32_fma")


from .layer import MoELayerBuffers, alloc_layer, run_layer, run_layer_host  # noqa: E402,F401
