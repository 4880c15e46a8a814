"""GPU parity, kernel by kernel, against the CPU oracle at sizes the oracle
finishes in seconds (several tiles plus ragged tails).  Every call goes through
the C ABI (libmoe_gate.so via the ctypes binding)."""

import numpy as np
import pytest
import torch

import oracle
import synth
import combine_moe_gate_gb300 as M
from gpu_util import assert_close, bits, bf16_bits_of_f32, f32_bits, status_ok, to_dev, to_host

pytestmark = pytest.mark.gpu


def _w(**kw):
    base = dict(name="t", act="gelu", capacity_factor=1.0, dtype="bf16")
    base.update(kw)
    return synth.Workload(**base)


GATE_CASES = [
    _w(s=256, m=64, e=4, k=1, h=128, dtype="f32", normalize_gates=False),
    _w(s=333, m=200, e=8, k=2, h=64),
    _w(s=517, m=96, e=16, k=3, h=64),
    _w(s=300, m=136, e=32, k=4, h=64, skew_alpha=1.0),
    _w(s=700, m=512, e=64, k=2, h=64, skew_alpha=1.2),
    _w(s=130, m=64, e=100, k=6, h=64),
    _w(s=129, m=256, e=256, k=8, h=64, skew_alpha=2.0),
    _w(s=77, m=40, e=5, k=5, h=64),
    _w(s=64, m=32, e=3, k=1, h=64, dtype="f32", normalize_gates=False),
    # several 512-byte feature slices with a ragged last one (lane-blocked order)
    _w(s=150, m=520, e=7, k=2, h=64, dtype="f32"),
    _w(s=100, m=1032, e=32, k=4, h=64, skew_alpha=0.5),
    # e <= 32 batches large enough for the resident kernel's 64 / e tokens per
    # warp group (smaller ones take 32 / e: twice the groups)
    _w(s=16400, m=64, e=16, k=2, h=64),
    _w(s=12000, m=72, e=32, k=4, h=64, skew_alpha=0.5),
    _w(s=20000, m=48, e=8, k=2, h=64),
]


def _gate_gpu(inp, w):
    x, wg, b = to_dev(inp["x"]), to_dev(inp["wg"]), to_dev(inp["bias"])
    idx = torch.full((w.k, w.s), -7, dtype=torch.int32, device="cuda")
    g = torch.full((w.k, w.s), -7.0, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    flags = M.MOE_FLAG_NORMALIZE_GATES if (w.normalize_gates and w.k >= 2) else 0
    M.moe_gate_topk(x, wg, b, w.k, idx, g, st, flags=flags)
    torch.cuda.synchronize()
    status_ok(st)
    return idx.cpu().numpy(), g.cpu().numpy()


@pytest.mark.parametrize("w", GATE_CASES, ids=lambda w: f"s{w.s}_m{w.m}_e{w.e}_k{w.k}_{w.dtype}")
def test_gate_topk(w):
    inp = synth.make_inputs_host(w, parts=("x", "wg", "bias"))
    lg = oracle.gate_logits(inp["x"], inp["wg"], inp["bias"])
    idx_o = oracle.topk(lg, w.k)
    g_o = oracle.gates(lg, idx_o, w.normalize_gates and w.k >= 2)
    idx, g = _gate_gpu(inp, w)
    assert np.array_equal(idx, idx_o)
    assert_close(g, g_o, "f32", "gates")


def test_gate_ties_break_to_lower_index():
    """Duplicated gate columns give bit-identical logits: the lower expert wins."""
    s, m, e, k = 200, 64, 8, 3
    x = synth.normal_host(5, "x", (s, m), 1.0, "bf16")
    wg = synth.normal_host(5, "wg", (m, e), 0.125, "f32")
    wg[:, 5] = wg[:, 1]
    wg[:, 6] = wg[:, 2]
    w = _w(s=s, m=m, e=e, k=k, h=64)
    idx, g = _gate_gpu(dict(x=x, wg=wg, bias=None), w)
    lg = oracle.gate_logits(x, wg)
    io = oracle.topk(lg, k)
    assert np.array_equal(idx, io)
    both = (idx == 1).any(0) & (idx == 5).any(0)
    assert both.any()
    for t in np.nonzero(both)[0]:
        assert list(idx[:, t]).index(1) < list(idx[:, t]).index(5)
    zero = dict(x=np.zeros((s, m), np.uint16), wg=wg, bias=np.zeros(e, np.float32))
    idx0, g0 = _gate_gpu(zero, w)       # all logits 0: experts 0..k-1, equal gates
    assert np.all(idx0 == np.arange(k)[:, None])
    assert np.allclose(g0, 1.0 / k, rtol=1e-6)


def _routing(seed, s, e, k, skew=0.0):
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((s, e)).astype(np.float32)
    if skew:
        lg -= np.float32(skew) * np.log(np.arange(1, e + 1, dtype=np.float32))
    idx = oracle.topk(lg, k)
    g = oracle.gates(lg, idx, k >= 2)
    return idx, g


CAP_CASES = [
    (0, 256, 4, 1, 1.0, 0.0),
    (1, 4096, 8, 2, 1.25, 0.0),
    (2, 3000, 16, 3, 0.0, 0.0),
    (3, 5000, 64, 2, -1.25, 1.2),
    (4, 2049, 256, 8, -1.5, 2.0),
    (5, 1, 1, 1, 1.0, 0.0),
    (6, 9999, 7, 7, 0.5, 0.0),
    (7, 700, 1000, 3, 2.0, 0.3),
    (8, 12345, 32, 4, 0.0, 3.0),
]


@pytest.mark.parametrize("case", CAP_CASES, ids=lambda c: f"s{c[1]}_e{c[2]}_k{c[3]}_f{c[4]}")
def test_capacity_locations(case):
    seed, s, e, k, f, skew = case
    idx, _ = _routing(seed, s, e, k, skew)
    loc_o, need_o = oracle.locations(idx, e)
    c_o = oracle.capacity(f, s, e, k, need_o)
    c_max = M.moe_capacity_bound(f, s, e, k)
    assert c_max >= c_o
    ws = torch.empty(M.moe_capacity_workspace_size(s, e, k), dtype=torch.uint8, device="cuda")
    loc = torch.full((k, s), -1, dtype=torch.int32, device="cuda")
    counts = torch.full((e,), -1, dtype=torch.int32, device="cuda")
    c_dev = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_capacity_locations(to_dev(idx), e, f, c_max, ws, loc, counts, c_dev, st)
    torch.cuda.synchronize()
    status_ok(st)
    assert int(c_dev.item()) == c_o
    assert np.array_equal(counts.cpu().numpy(), need_o.astype(np.int32))
    assert np.array_equal(loc.cpu().numpy(), loc_o)


def test_capacity_overflow_sets_status():
    s, e, k = 1000, 4, 2
    idx, _ = _routing(11, s, e, k, 2.0)
    ws = torch.empty(M.moe_capacity_workspace_size(s, e, k), dtype=torch.uint8, device="cuda")
    loc = torch.empty((k, s), dtype=torch.int32, device="cuda")
    counts = torch.empty((e,), dtype=torch.int32, device="cuda")
    c_dev = torch.empty((1,), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_capacity_locations(to_dev(idx), e, 0.0, 16, ws, loc, counts, c_dev, st)
    torch.cuda.synchronize()
    assert int(st.item()) == M.MOE_ERR_CAPACITY
    # downstream kernels see the status and write nothing
    x = to_dev(synth.normal_host(1, "x", (s, 64), 1.0, "bf16"))
    buf = torch.full((e, 16, 64), 3.0, dtype=torch.bfloat16, device="cuda")
    M.moe_encode(x, to_dev(idx), loc, counts, c_dev, buf, st)
    torch.cuda.synchronize()
    assert bool((buf == 3.0).all())


DISPATCH_CASES = [
    # seed, s, m, e, k, f, skew, dtype
    (0, 256, 64, 4, 1, 1.0, 0.0, "f32"),
    (1, 333, 200, 8, 2, 1.25, 0.0, "bf16"),
    (2, 500, 1032, 16, 3, 0.0, 0.0, "bf16"),
    (3, 400, 136, 64, 2, -1.25, 1.2, "bf16"),
    (4, 300, 7168, 32, 8, -1.5, 2.0, "bf16"),
    (5, 257, 12, 5, 2, 0.6, 0.0, "f32"),
]


def _dispatch_setup(case):
    seed, s, m, e, k, f, skew, dt = case
    idx, g = _routing(seed, s, e, k, skew)
    loc, need = oracle.locations(idx, e)
    c = oracle.capacity(f, s, e, k, need)
    c_max = c + 5
    x = synth.normal_host(seed, "x", (s, m), 1.0, dt)
    d = dict(idx=to_dev(idx), loc=to_dev(loc), gates=to_dev(g), counts=to_dev(need.astype(np.int32)),
             c_dev=to_dev(np.array([c], np.int32)), x=to_dev(x),
             st=torch.zeros(1, dtype=torch.int32, device="cuda"))
    return dict(seed=seed, s=s, m=m, e=e, k=k, c=c, c_max=c_max, dt=dt, idx=idx, g=g, loc=loc,
                need=need, x=x, d=d)


def _bits_of(a, dt):
    return bf16_bits_of_f32(a) if dt == "bf16" else f32_bits(a)


@pytest.mark.parametrize("case", DISPATCH_CASES, ids=lambda c: f"s{c[1]}_m{c[2]}_e{c[3]}_k{c[4]}_{c[7]}")
def test_encode_and_zero_fill(case):
    S = _dispatch_setup(case)
    e, c, c_max, m, dt = S["e"], S["c"], S["c_max"], S["m"], S["dt"]
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    want = oracle.encode(S["x"], S["idx"], S["loc"], c, e, c_max)
    kept = oracle.kept_rows(S["need"], c)
    d = S["d"]
    buf = torch.full((e, c_max, m), 7.0, dtype=tdt, device="cuda")
    M.moe_encode(d["x"], d["idx"], d["loc"], d["counts"], d["c_dev"], buf, d["st"])
    torch.cuda.synchronize()
    status_ok(d["st"])
    got = to_host(buf)
    for j in range(e):
        assert np.array_equal(_bits_of(got[j, :kept[j]], dt), _bits_of(want[j, :kept[j]], dt))
        assert np.all(got[j, kept[j]:] == 7.0)  # untouched without ZERO_FILL
    buf.fill_(7.0)
    M.moe_encode(d["x"], d["idx"], d["loc"], d["counts"], d["c_dev"], buf, d["st"],
                 flags=M.MOE_FLAG_ZERO_FILL)
    torch.cuda.synchronize()
    got = to_host(buf)
    assert np.array_equal(got[:, :c], want[:, :c])   # the full logical [e, c, m] view
    assert np.all(got[:, c:] == 7.0)


@pytest.mark.parametrize("case", DISPATCH_CASES, ids=lambda c: f"s{c[1]}_m{c[2]}_e{c[3]}_k{c[4]}_{c[7]}")
def test_decode_and_backward(case):
    S = _dispatch_setup(case)
    e, c, c_max, m, s, k, dt = S["e"], S["c"], S["c_max"], S["m"], S["s"], S["k"], S["dt"]
    bf16 = dt == "bf16"
    tdt = torch.bfloat16 if bf16 else torch.float32
    d = S["d"]
    out = synth.normal_host(S["seed"], "out", (e, c_max, m), 1.0, dt)
    dy = synth.normal_host(S["seed"], "dy", (s, m), 1.0, dt)
    out_d, dy_d = to_dev(out), to_dev(dy)
    # decode: same fp32 fused multiply-add order as the oracle -> bit-identical
    y = torch.empty((s, m), dtype=tdt, device="cuda")
    M.moe_decode(out_d, d["idx"], d["loc"], d["gates"], d["c_dev"], y, d["st"])
    y_o = oracle.decode(out, S["idx"], S["loc"], S["g"], c, bf16)
    # backward of decode
    d_out = torch.full((e, c_max, m), 5.0, dtype=tdt, device="cuda")
    d_g = torch.full((k, s), 9.0, dtype=torch.float32, device="cuda")
    M.moe_decode_bwd(dy_d, out_d, d["idx"], d["loc"], d["gates"], d["counts"], d["c_dev"], d_out,
                     d_g, d["st"], flags=M.MOE_FLAG_ZERO_FILL)
    d_out_o, d_g_o = oracle.decode_bwd(dy, out, S["idx"], S["loc"], S["g"], c, bf16)
    # backward of encode, fed with the oracle's d_out
    dx = torch.empty((s, m), dtype=tdt, device="cuda")
    dbuf = synth.normal_host(S["seed"], "dbuf", (e, c_max, m), 1.0, dt)
    M.moe_encode_bwd(to_dev(dbuf), d["idx"], d["loc"], d["c_dev"], dx, d["st"])
    dx_o = oracle.encode_bwd(dbuf, S["idx"], S["loc"], c, bf16)
    torch.cuda.synchronize()
    status_ok(d["st"])
    assert_close(to_host(y), y_o, dt, "decode")
    assert np.array_equal(bits(y), _bits_of(y_o, dt))
    got = to_host(d_out)
    assert np.array_equal(_bits_of(got[:, :c], dt), _bits_of(d_out_o[:, :c], dt))  # exact product
    assert np.all(got[:, c:] == 5.0)
    assert_close(d_g.cpu().numpy(), d_g_o, "f32" if not bf16 else "bf16", "d_gates")
    assert np.all(d_g.cpu().numpy()[S["loc"] >= c] == 0.0)
    assert np.array_equal(bits(dx), _bits_of(dx_o, dt))


FFN_CASES = [
    _w(s=256, m=64, e=4, k=1, h=128, act="relu", dtype="f32", normalize_gates=False),
    _w(s=300, m=64, e=3, k=2, h=96, act="gelu", dtype="f32", capacity_factor=0.0),
    _w(s=333, m=128, e=4, k=2, h=256, act="gelu", capacity_factor=1.25),
    _w(s=300, m=192, e=8, k=2, h=320, act="swiglu", capacity_factor=0.0, skew_alpha=1.0),
    _w(s=200, m=256, e=5, k=1, h=512, act="relu", capacity_factor=-2.0, skew_alpha=1.5),
    _w(s=600, m=200, e=3, k=2, h=136, act="gelu", capacity_factor=0.0),
    _w(s=900, m=64, e=6, k=3, h=1024, act="swiglu", capacity_factor=1.5, skew_alpha=0.7),
]


@pytest.mark.parametrize("w", FFN_CASES, ids=lambda w: f"e{w.e}_m{w.m}_h{w.h}_{w.act}_{w.dtype}")
def test_expert_ffn(w):
    inp = synth.make_inputs_host(w)
    ref = oracle.layer_forward(w, inp)
    c, e, m, h = ref["c"], w.e, w.m, w.h
    c_max = c + 3
    bf16 = w.dtype == "bf16"
    tdt = torch.bfloat16 if bf16 else torch.float32
    buf_h = np.zeros((e, c_max, m), np.float32)
    buf_h[:, :c] = ref["buf"][:, :c]
    buf = to_dev(buf_h).to(tdt)
    dt_code = M.MOE_BF16 if bf16 else M.MOE_F32
    ws = torch.empty(M.moe_expert_ffn_workspace_size(dt_code, w.act, e, c_max, m, h),
                     dtype=torch.uint8, device="cuda")
    out = torch.full((e, c_max, m), 3.0, dtype=tdt, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_expert_ffn(buf, to_dev(ref["needed"].astype(np.int32)), to_dev(np.array([c], np.int32)),
                     to_dev(inp["w1"]), to_dev(inp["b1"]), to_dev(inp["w3"]), to_dev(inp["w2"]),
                     to_dev(inp["b2"]), w.act, ws, out, st)
    torch.cuda.synchronize()
    status_ok(st)
    got = to_host(out)
    for j in range(e):
        kj = int(ref["kept"][j])
        assert_close(got[j, :kj], ref["out"][j, :kj], w.dtype, f"expert {j}")
        assert np.all(got[j, kj:] == 3.0)  # rows past the kept count are not written


LAYER_CASES = [
    synth.workloads.TINY_FP32,
    _w(s=512, m=256, e=8, k=2, h=512, act="gelu", capacity_factor=1.25),
    _w(s=400, m=128, e=16, k=3, h=256, act="gelu", capacity_factor=0.0),
    _w(s=300, m=256, e=32, k=4, h=128, act="swiglu", capacity_factor=-1.5, skew_alpha=2.0),
]


@pytest.mark.parametrize("w", LAYER_CASES, ids=lambda w: f"s{w.s}_e{w.e}_k{w.k}_{w.act}_{w.dtype}")
def test_layer_forward(w):
    inp = synth.make_inputs_host(w)
    ref = oracle.layer_forward(w, inp)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    bufs = M.alloc_layer(w.s, w.m, w.e, w.k, w.h, w.act, w.capacity_factor, dtype=tdt)
    M.run_layer(to_dev(inp["x"]), to_dev(inp["wg"]), to_dev(inp["bias"]), to_dev(inp["w1"]),
                to_dev(inp["b1"]), to_dev(inp["w3"]), to_dev(inp["w2"]), to_dev(inp["b2"]), w.act,
                w.k, w.capacity_factor, bufs, normalize_gates=w.normalize_gates and w.k >= 2)
    torch.cuda.synchronize()
    status_ok(bufs.status)
    assert np.array_equal(bufs.idx.cpu().numpy(), ref["idx"])
    assert np.array_equal(bufs.loc.cpu().numpy(), ref["loc"])
    assert int(bufs.c_dev.item()) == ref["c"]
    assert_close(bufs.gates.cpu().numpy(), ref["gates"], "f32", "gates")
    assert_close(to_host(bufs.y), ref["y"], w.dtype, "y")


def test_determinism_repeat_bitwise():
    w = LAYER_CASES[1]
    inp = synth.make_inputs_host(w)
    args = [to_dev(inp[n]) for n in ("x", "wg", "bias", "w1", "b1", "w3", "w2", "b2")]
    outs = []
    for _ in range(2):
        bufs = M.alloc_layer(w.s, w.m, w.e, w.k, w.h, w.act, w.capacity_factor)
        M.run_layer(*args, w.act, w.k, w.capacity_factor, bufs)
        torch.cuda.synchronize()
        outs.append((bits(bufs.y), bufs.idx.cpu().numpy(), bufs.loc.cpu().numpy()))
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


def test_ffn_gelu_epilogue_matches_exact_erf():
    """Identity fc1/fc2 weights make out = bf16(GELU(x)) exactly, so the tensor-core
    epilogue's GELU is compared with the oracle's exact double-precision erf form
    on a dense sweep of bf16 inputs in [-6, 6]: every value within one bf16 step
    (or 2e-6 absolute in the far negative tail, where the erfc approximation is
    only absolutely accurate and GELU itself is tiny) and, wherever |GELU| >=
    1e-3, nearly all bit-identical."""
    m = h = 64
    xs = np.linspace(-6.0, 6.0, 64 * 256).astype(np.float32)
    xb = synth.f32_to_bf16_bits(xs).reshape(256, 64)        # 256 rows of 64 values
    rows = xb.shape[0]
    eye = synth.f32_to_bf16_bits(np.eye(h, m, dtype=np.float32))[None]  # [1, h, m]
    buf = xb[None]                                             # [1, rows, m]
    counts = np.array([rows], np.int32)
    ws = torch.empty(M.moe_expert_ffn_workspace_size(M.MOE_BF16, "gelu", 1, rows, m, h),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((1, rows, m), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_expert_ffn(to_dev(buf), to_dev(counts), to_dev(counts), to_dev(eye), None, None,
                     to_dev(eye), None, "gelu", ws, out, st)
    torch.cuda.synchronize()
    status_ok(st)
    got = to_host(out)[0]
    want = oracle.ffn_rows(buf, eye, None, None, eye, None, "gelu", np.zeros(rows, np.int32),
                           np.arange(rows), True)
    step = np.abs(want) * 2.0 ** -7                 # one bf16 step at the value
    assert np.all(np.abs(got - want) <= np.maximum(step * 1.01, 2e-6))
    big = np.abs(want) >= 1e-3                      # where relative accuracy is meaningful
    assert np.mean(got[big] == want[big]) > 0.99
