"""ctypes wrappers around the C oracle, plus the whole-layer forward chain.

Arrays are numpy.  Values that are bf16 in the layer may be passed either as
uint16 bit patterns (widened exactly) or as float32 values.  Outputs rounded to
bf16 come back as float32 arrays holding bf16 values.
"""

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

ACT = {"relu": 0, "gelu": 1, "swiglu": 2}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available).  Returns the .so path."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _SO + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _SO)
    return _SO


def _L():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
            sig = {
                "orc_gate_logits": [P, P, P, I64, I32, I32, I32, P],
                "orc_gate_bwd": [P, P, P, P, P, I64, I32, I32, I32, I32, P, P, P, P],
                "orc_topk": [P, I64, I32, I32, P],
                "orc_gates": [P, P, I64, I32, I32, I32, P],
                "orc_locations": [P, I64, I32, I32, P, P],
                "orc_capacity": [D, I64, I32, I32, P],
                "orc_encode": [P, P, P, I64, I64, I32, I32, I32, I64, P],
                "orc_decode": [P, P, P, P, I64, I64, I32, I32, I32, I64, I32, P],
                "orc_decode_bwd": [P, P, P, P, P, I64, I64, I32, I32, I32, I64, I32, P, P],
                "orc_encode_bwd": [P, P, P, I64, I64, I32, I32, I32, I64, I32, P],
                "orc_ffn_rows": [P, P, P, P, P, P, I32, I32, I64, I32, I32, I32, P, P, I64, P],
                "orc_ffn_bwd": [P, P, P, P, P, I32, I32, I64, I32, I32, I32, P, P, P, P, P, P, P,
                                P],
                "orc_round_bf16": [D],
                "orc_quantize_rows_fp8": [P, I64, I32, P, P],
                "orc_fc_fp8": [P, P, P, P, P, I32, I64, I32, I32, P],
                "orc_fp8_decode": [ctypes.c_uint8],
                "orc_fp8_encode": [ctypes.c_float],
                "orc_set_threads": [I32],
                "orc_get_threads": [],
            }
            for name, args in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = None
            lib.orc_capacity.restype = I64
            lib.orc_round_bf16.restype = ctypes.c_float
            lib.orc_fp8_decode.restype = ctypes.c_float
            lib.orc_fp8_encode.restype = ctypes.c_uint8
            lib.orc_get_threads.restype = I32
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def to_f32(a):
    """float32 contiguous view of a tensor given as fp32 values or bf16 bits."""
    if a is None:
        return None
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return np.ascontiguousarray(a, dtype=np.float32)


def set_threads(n: int):
    _L().orc_set_threads(int(n))


def get_threads() -> int:
    return int(_L().orc_get_threads())


def round_bf16(v: float) -> float:
    return float(_L().orc_round_bf16(float(v)))


def gate_chunk(e, x_is_bf16):
    """The logit summation order the layer uses for e experts: chunk width V of
    the lane-blocked order (8 for bf16 x, 4 for fp32 x) for e <= 32, else 0 (one
    sequential accumulator)."""
    if e > 32:
        return 0
    return 8 if x_is_bf16 else 4


def gate_logits(x, wg, bias=None, chunk=None):
    """fp32 logits [s, e] in the layer's summation order (see orc_gate_logits),
    then + bias.  chunk=None picks the order from e and from x's dtype (bf16 bits
    given as uint16 -> 8, fp32 -> 4)."""
    x_is_bf16 = np.asarray(x).dtype == np.uint16
    x, wg, bias = to_f32(x), to_f32(wg), to_f32(bias)
    s, m = x.shape
    e = wg.shape[1]
    if chunk is None:
        chunk = gate_chunk(e, x_is_bf16)
    out = np.empty((s, e), np.float32)
    _L().orc_gate_logits(_p(x), _p(wg), _p(bias), s, m, e, int(chunk), _p(out))
    return out


def topk(logits, k):
    logits = to_f32(logits)
    s, e = logits.shape
    idx = np.empty((k, s), np.int32)
    _L().orc_topk(_p(logits), s, e, k, _p(idx))
    return idx


def gates(logits, idx, normalize):
    logits = to_f32(logits)
    idx = np.ascontiguousarray(idx, np.int32)
    s, e = logits.shape
    k = idx.shape[0]
    g = np.empty((k, s), np.float32)
    _L().orc_gates(_p(logits), _p(idx), s, e, k, int(bool(normalize)), _p(g))
    return g


def gate_bwd(x, wg, bias, idx, d_gates, normalize, chunk=None):
    """Backward of the gate values to the logits, the gate weight, its bias and
    x (float64 arrays d_logits [s, e], d_wg [m, e], d_bias [e], d_x [s, m]);
    the forward logits are recomputed in the layer's order."""
    lg = gate_logits(x, wg, bias, chunk)
    x, wg = to_f32(x), to_f32(wg)
    idx = np.ascontiguousarray(idx, np.int32)
    dg = np.ascontiguousarray(d_gates, np.float32)
    s, m = x.shape
    e = wg.shape[1]
    k = idx.shape[0]
    out = dict(d_logits=np.empty((s, e)), d_wg=np.empty((m, e)), d_bias=np.empty(e),
               d_x=np.empty((s, m)))
    _L().orc_gate_bwd(_p(x), _p(wg), _p(lg), _p(idx), _p(dg), s, m, e, k, int(bool(normalize)),
                      _p(out["d_logits"]), _p(out["d_wg"]), _p(out["d_bias"]), _p(out["d_x"]))
    return out


def locations(idx, e):
    idx = np.ascontiguousarray(idx, np.int32)
    k, s = idx.shape
    loc = np.empty((k, s), np.int32)
    needed = np.zeros(e, np.int64)
    _L().orc_locations(_p(idx), s, e, k, _p(loc), _p(needed))
    return loc, needed


def capacity(f, s, e, k, needed):
    needed = np.ascontiguousarray(needed, np.int64)
    return int(_L().orc_capacity(float(np.float32(f)), s, e, k, _p(needed)))


def kept_rows(needed, c):
    return np.minimum(np.asarray(needed, np.int64), c)


def encode(x, idx, loc, c, e, cmax, buf=None):
    x = to_f32(x)
    idx = np.ascontiguousarray(idx, np.int32)
    loc = np.ascontiguousarray(loc, np.int32)
    s, m = x.shape
    k = idx.shape[0]
    if buf is None:
        buf = np.zeros((e, cmax, m), np.float32)
    _L().orc_encode(_p(x), _p(idx), _p(loc), c, s, m, e, k, cmax, _p(buf))
    return buf


def decode(out, idx, loc, g, c, bf16):
    out = to_f32(out)
    e, cmax, m = out.shape
    idx = np.ascontiguousarray(idx, np.int32)
    loc = np.ascontiguousarray(loc, np.int32)
    g = np.ascontiguousarray(g, np.float32)
    k, s = idx.shape
    y = np.empty((s, m), np.float32)
    _L().orc_decode(_p(out), _p(idx), _p(loc), _p(g), c, s, m, e, k, cmax, int(bf16), _p(y))
    return y


def decode_bwd(dy, out, idx, loc, g, c, bf16):
    dy, out = to_f32(dy), to_f32(out)
    e, cmax, m = out.shape
    idx = np.ascontiguousarray(idx, np.int32)
    loc = np.ascontiguousarray(loc, np.int32)
    g = np.ascontiguousarray(g, np.float32)
    k, s = idx.shape
    d_out = np.zeros((e, cmax, m), np.float32)
    d_g = np.empty((k, s), np.float32)
    _L().orc_decode_bwd(_p(dy), _p(out), _p(idx), _p(loc), _p(g), c, s, m, e, k, cmax,
                        int(bf16), _p(d_out), _p(d_g))
    return d_out, d_g


def encode_bwd(d_buf, idx, loc, c, bf16):
    d_buf = to_f32(d_buf)
    e, cmax, m = d_buf.shape
    idx = np.ascontiguousarray(idx, np.int32)
    loc = np.ascontiguousarray(loc, np.int32)
    k, s = idx.shape
    dx = np.empty((s, m), np.float32)
    _L().orc_encode_bwd(_p(d_buf), _p(idx), _p(loc), c, s, m, e, k, cmax, int(bf16), _p(dx))
    return dx


def ffn_rows(buf, w1, b1, w3, w2, b2, act, rows_e, rows_j, bf16):
    """Expert MLP outputs for the listed (expert, row) pairs -> [len(rows), m]."""
    buf, w1, b1, w3, w2, b2 = (to_f32(a) for a in (buf, w1, b1, w3, w2, b2))
    e, cmax, m = buf.shape
    h = w1.shape[1]
    re = np.ascontiguousarray(rows_e, np.int32)
    rj = np.ascontiguousarray(rows_j, np.int64)
    out = np.empty((len(re), m), np.float32)
    _L().orc_ffn_rows(_p(buf), _p(w1), _p(b1), _p(w3), _p(w2), _p(b2), ACT[act], e, cmax, m, h,
                      int(bf16), _p(re), _p(rj), len(re), _p(out))
    return out


def ffn_bwd(buf, w1, b1, w3, w2, act, kept, d_out, bf16):
    """Backward of the expert MLP over the kept rows (row j < kept[e] of expert
    e) for L = sum <d_out, out>: d_buf [e, cmax, m] (layer dtype, 0 past the
    kept rows), d_w1 / d_w3 [e, h, m], d_w2 [e, m, h], d_b1 [e, h], d_b2 [e, m]
    (fp32; d_w3 for SwiGLU only, the biases for ReLU/GELU only)."""
    buf, w1, b1, w3, w2, d_out = (to_f32(a) for a in (buf, w1, b1, w3, w2, d_out))
    e, cmax, m = buf.shape
    h = w1.shape[1]
    kept = np.ascontiguousarray(kept, np.int64)
    assert kept.shape == (e,) and np.all((kept >= 0) & (kept <= cmax))
    swiglu = act == "swiglu"
    out = dict(d_buf=np.empty((e, cmax, m), np.float32), d_w1=np.empty((e, h, m), np.float32),
               d_w2=np.empty((e, m, h), np.float32))
    if swiglu:
        out["d_w3"] = np.empty((e, h, m), np.float32)
    else:
        out["d_b1"] = np.empty((e, h), np.float32)
        out["d_b2"] = np.empty((e, m), np.float32)
    _L().orc_ffn_bwd(_p(buf), _p(w1), _p(b1), _p(w3), _p(w2), ACT[act], e, cmax, m, h, int(bf16),
                     _p(kept), _p(d_out), _p(out["d_buf"]), _p(out["d_w1"]), _p(out.get("d_b1")),
                     _p(out.get("d_w3")), _p(out["d_w2"]), _p(out.get("d_b2")))
    return out


def layer_forward(w, inp, cmax=None, rows=None):
    """The full forward chain on the CPU for workload `w` with inputs `inp`.

    Returns a dict with logits, idx, gates, loc, needed, c, buf, out (expert
    outputs at kept rows; other rows 0) and y.  `rows`, if given, restricts the
    FFN to those (expert, row) pairs (the rest of `out` stays 0) and y is then
    not computed.
    """
    bf16 = w.dtype == "bf16"
    lg = gate_logits(inp["x"], inp["wg"], inp.get("bias"))
    idx = topk(lg, w.k)
    g = gates(lg, idx, w.normalize_gates and w.k >= 2)
    loc, needed = locations(idx, w.e)
    c = capacity(w.capacity_factor, w.s, w.e, w.k, needed)
    cmax = c if cmax is None else cmax
    buf = encode(inp["x"], idx, loc, c, w.e, cmax)
    kept = kept_rows(needed, c)
    res = dict(logits=lg, idx=idx, gates=g, loc=loc, needed=needed, c=c, buf=buf, kept=kept)
    full = rows is None
    if full:
        re = np.concatenate([np.full(int(kept[j]), j, np.int32) for j in range(w.e)])
        rj = np.concatenate([np.arange(int(kept[j]), dtype=np.int64) for j in range(w.e)])
    else:
        re, rj = rows
    o = ffn_rows(buf, inp["w1"], inp.get("b1"), inp.get("w3"), inp["w2"], inp.get("b2"),
                 w.act, re, rj, bf16)
    out = np.zeros_like(buf)
    out[np.asarray(re, np.int64), np.asarray(rj, np.int64)] = o
    res["out"] = out
    if full:
        res["y"] = decode(out, idx, loc, g, c, bf16)
    return res


def layer_backward(w, inp, fwd, dy):
    """Backward of the layer forward for L = <dy, y>, from `fwd` =
    layer_forward(w, inp) (full): decode backward gives d_out (the experts'
    output gradient) and d_gates; the expert MLP backward over the kept rows
    gives d_buf and the weight gradients; encode backward turns d_buf into the
    copy path's d_x, and the gate backward of d_gates gives the gate path's
    d_x, d_wg and the gate bias gradient.  d_x is the sum of the two paths (in
    double); routing (top-k, slots, drops) is piecewise constant."""
    bf16 = w.dtype == "bf16"
    c = fwd["c"]
    d_out, d_g = decode_bwd(dy, fwd["out"], fwd["idx"], fwd["loc"], fwd["gates"], c, bf16)
    ffn = ffn_bwd(fwd["buf"], inp["w1"], inp.get("b1"), inp.get("w3"), inp["w2"], w.act,
                  fwd["kept"], d_out, bf16)
    dx_copy = encode_bwd(ffn["d_buf"], fwd["idx"], fwd["loc"], c, bf16)
    gate = gate_bwd(inp["x"], inp["wg"], inp.get("bias"), fwd["idx"], d_g,
                    w.normalize_gates and w.k >= 2)
    res = dict(ffn)
    res.update(d_out=d_out, d_gates=d_g, d_logits=gate["d_logits"], d_wg=gate["d_wg"],
               d_gate_bias=gate["d_bias"],
               d_x=dx_copy.astype(np.float64) + gate["d_x"])
    return res



# ----------------------------------------------------------- FP8 experts
FP8_ACT = {None: -1, "none": -1, "relu": 0, "gelu": 1}


def fp8_decode(code: int) -> float:
    """The value of one e4m3 code (NaN for 0x7F / 0xFF)."""
    return float(_L().orc_fp8_decode(int(code) & 0xFF))


def fp8_encode(v: float) -> int:
    """e4m3 code of v: nearest, ties to even, saturating to +-448."""
    return int(_L().orc_fp8_encode(float(v)))


def quantize_rows_fp8(x):
    """Row-wise e4m3 quantisation of a 2-D array (fp32 values or bf16 bits):
    (codes uint8 [rows, cols], scales fp32 [rows]), scale = amax / 448."""
    x = np.ascontiguousarray(to_f32(x))
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    sc = np.empty(rows, np.float32)
    _L().orc_quantize_rows_fp8(_p(x), rows, cols, _p(q), _p(sc))
    return q, sc


def fc_fp8(qa, sa, qw, sw, bias, act):
    """act(sa[r] sw[n] sum_k a[r, k] w[n, k] + bias[n]) rounded to bf16, a and w
    e4m3 codes [rows, K] and [N, K]: [rows, N] float32 holding bf16 values."""
    qa = np.ascontiguousarray(qa, np.uint8)
    qw = np.ascontiguousarray(qw, np.uint8)
    sa = np.ascontiguousarray(sa, np.float32)
    sw = np.ascontiguousarray(sw, np.float32)
    bias = None if bias is None else np.ascontiguousarray(to_f32(bias))
    rows, K = qa.shape
    N = qw.shape[0]
    out = np.empty((rows, N), np.float32)
    _L().orc_fc_fp8(_p(qa), _p(sa), _p(qw), _p(sw), _p(bias), FP8_ACT[act], rows, K, N, _p(out))
    return out
