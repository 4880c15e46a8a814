"""The Python binding refuses tensors the C ABI would misread: wrong shape or
dtype, non-contiguous views, host memory.  Runs on the CPU; every case raises
before the library is called, so nothing is launched."""

import pytest
import torch

import combine_moe_gate_gb300 as M

pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="host tensors stand in for device ones only without a GPU")


@pytest.fixture
def host_as_device(monkeypatch):
    """Let host tensors pass the device check so that the shape, dtype and
    layout checks behind it can be exercised; every call below fails one of
    those, so the library is never reached."""
    monkeypatch.setattr(M, "_on_device", lambda t: True)


def _gate_args(s=16, m=64, e=8, k=2):
    return dict(x=torch.zeros((s, m), dtype=torch.bfloat16), wg=torch.zeros((m, e)),
                bias=torch.zeros(e), k=k, idx=torch.zeros((k, s), dtype=torch.int32),
                gates=torch.zeros((k, s)), dev_status=torch.zeros(1, dtype=torch.int32))


def _call(fn, **over):
    a = _gate_args()
    a.update(over)
    before = M.launch_count()
    try:
        fn(**a)
    finally:
        assert M.launch_count() == before


def test_wrong_shape_is_rejected(host_as_device):
    with pytest.raises(ValueError, match="gates: shape"):
        _call(M.moe_gate_topk, gates=torch.zeros((2, 15)))
    with pytest.raises(ValueError, match="wg: shape"):
        _call(M.moe_gate_topk, wg=torch.zeros((32, 8)))
    with pytest.raises(ValueError, match="bias: shape"):
        _call(M.moe_gate_topk, bias=torch.zeros(9))


def test_wrong_dtype_is_rejected(host_as_device):
    with pytest.raises(TypeError, match="idx: dtype"):
        _call(M.moe_gate_topk, idx=torch.zeros((2, 16), dtype=torch.int64))
    with pytest.raises(TypeError, match="wg: dtype"):
        _call(M.moe_gate_topk, wg=torch.zeros((64, 8), dtype=torch.float64))
    with pytest.raises(TypeError, match="unsupported dtype"):
        _call(M.moe_gate_topk, x=torch.zeros((16, 64), dtype=torch.float16))


def test_non_contiguous_view_is_rejected(host_as_device):
    wg_t = torch.zeros((8, 64)).t()            # [64, 8] with transposed strides
    with pytest.raises(ValueError, match="wg: must be contiguous"):
        _call(M.moe_gate_topk, wg=wg_t)


def test_host_tensor_is_rejected():
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        _call(M.moe_gate_topk)


def test_backward_and_layer_entry_points_check_their_outputs(host_as_device):
    s, m, e, k, c_max, h = 16, 64, 8, 2, 6, 32
    i32 = dict(dtype=torch.int32)
    bf = dict(dtype=torch.bfloat16)
    idx, loc = torch.zeros((k, s), **i32), torch.zeros((k, s), **i32)
    st, c_dev, counts = torch.zeros(1, **i32), torch.zeros(1, **i32), torch.zeros(e, **i32)
    out = torch.zeros((e, c_max, m), **bf)
    with pytest.raises(ValueError, match="y: shape"):
        M.moe_decode(out, idx, loc, torch.zeros((k, s)), c_dev, torch.zeros((s, m + 8), **bf), st)
    with pytest.raises(TypeError, match="dx: dtype"):
        M.moe_encode_bwd(out, idx, loc, c_dev, torch.zeros((s, m)), st)
    with pytest.raises(ValueError, match="d_out: shape"):
        M.moe_decode_bwd(torch.zeros((s, m), **bf), out, idx, loc, torch.zeros((k, s)), counts,
                         c_dev, torch.zeros((e, c_max + 1, m), **bf), torch.zeros((k, s)), st)
    with pytest.raises(ValueError, match="d_x: shape"):
        M.moe_gate_bwd(torch.zeros((s, m), **bf), torch.zeros((m, e)), None, idx,
                       torch.zeros((k, s)), torch.zeros((k, s)), torch.zeros((s, e)), st,
                       d_x=torch.zeros((s, m - 8)))
    with pytest.raises(ValueError, match="w2: shape"):
        M.moe_expert_ffn(out, counts, c_dev, torch.zeros((e, h, m), **bf), None, None,
                         torch.zeros((e, h, m), **bf), None, "gelu", torch.zeros(16, dtype=torch.uint8),
                         torch.zeros((e, c_max, m), **bf), st)
    with pytest.raises(ValueError, match="counts: shape"):
        M.moe_capacity_locations_noalloc(idx, e, 1.0, c_max, loc, torch.zeros(e + 1, **i32), c_dev,
                                         st)
    with pytest.raises(TypeError, match="loc: dtype"):
        M.moe_capacity_locations_noalloc(idx, e, 1.0, c_max, torch.zeros((k, s)), counts, c_dev, st)
    with pytest.raises(TypeError, match="b1: dtype"):
        M.moe_layer_forward(torch.zeros((s, m), **bf), torch.zeros((m, e)), None,
                            torch.zeros((e, h, m), **bf), torch.zeros((e, h)), None,
                            torch.zeros((e, m, h), **bf), None, "gelu", k, 1.0, 0, idx,
                            torch.zeros((k, s)), loc, counts, c_dev, out, out,
                            torch.zeros((s, m), **bf), torch.zeros(16, dtype=torch.uint8), st)


class _StubLib:
    """Records each call's arguments instead of calling the library."""

    def __init__(self):
        self.calls = {}

    def __getattr__(self, name):
        def fn(*args):
            self.calls[name] = args
            return 0
        return fn


@pytest.fixture
def stub(monkeypatch, host_as_device):
    lib = _StubLib()
    monkeypatch.setattr(M, "load", lambda: lib)
    monkeypatch.setattr(M, "_stream", lambda s: None)
    return lib


def test_well_formed_calls_pass_and_marshal_their_sizes(stub):
    s, m, e, k, h, c_max = 24, 64, 8, 2, 32, 10
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    z = lambda *shape, dtype=f32: torch.zeros(shape, dtype=dtype)
    x, wg, gb = z(s, m, dtype=bf), z(m, e), z(e)
    idx, loc, gates = z(k, s, dtype=i32), z(k, s, dtype=i32), z(k, s)
    counts, c_dev, st = z(e, dtype=i32), z(1, dtype=i32), z(1, dtype=i32)
    buf, out = z(e, c_max, m, dtype=bf), z(e, c_max, m, dtype=bf)
    w1, w2, b1, b2 = z(e, h, m, dtype=bf), z(e, m, h, dtype=bf), z(e, h, dtype=bf), z(e, m, dtype=bf)
    ws = z(4096, dtype=torch.uint8)
    M.moe_gate_topk(x, wg, gb, k, idx, gates, st, flags=1)
    M.moe_capacity_locations(idx, e, 1.25, c_max, ws, loc, counts, c_dev, st)
    M.moe_capacity_locations_noalloc(idx, e, 1.25, c_max, loc, counts, c_dev, st)
    M.moe_encode(x, idx, loc, counts, c_dev, buf, st)
    M.moe_expert_ffn(buf, counts, c_dev, w1, b1, None, w2, b2, "gelu", ws, out, st)
    M.moe_decode(out, idx, loc, gates, c_dev, z(s, m, dtype=bf), st)
    M.moe_decode_bwd(z(s, m, dtype=bf), out, idx, loc, gates, counts, c_dev, z(e, c_max, m, dtype=bf),
                     z(k, s), st)
    M.moe_encode_bwd(out, idx, loc, c_dev, z(s, m, dtype=bf), st)
    M.moe_gate_bwd(x, wg, gb, idx, gates, z(k, s), z(s, e), st, d_wg=z(m, e), d_bias=z(e),
                   d_x=z(s, m))
    M.moe_layer_forward(x, wg, gb, w1, b1, None, w2, b2, "gelu", k, 1.25, 1, idx, gates, loc,
                        counts, c_dev, buf, out, z(s, m, dtype=bf), ws, st)
    class _Ev:
        cuda_event = 1

    M.moe_layer_forward_pipelined(x, wg, gb, w1, b1, None, w2, b2, "gelu", k, 1.25, 1, idx, gates,
                                  loc, counts, c_dev, buf, out, z(s, m, dtype=bf), ws, st, 3, None,
                                  [_Ev()] * 4)
    M.moe_expert_ffn_bwd(buf, z(e, c_max, h, dtype=bf), counts, c_dev, w1, b1, None, w2, "gelu",
                         z(e, c_max, m, dtype=bf), ws, z(e, c_max, m, dtype=bf), z(e, h, m, dtype=bf),
                         None, z(e, m, h, dtype=bf), z(e, h, dtype=bf), z(e, m, dtype=bf), st)
    M.moe_expert_ffn_train(buf, counts, c_dev, w1, b1, None, w2, b2, "gelu", ws, out,
                           z(e, c_max, h, dtype=bf), st)
    M.moe_expert_ffn_bwd_saved(buf, z(e, c_max, h, dtype=bf), z(e, c_max, 2 * h, dtype=bf), counts,
                               c_dev, w1, w1, w2, "swiglu", z(e, c_max, m, dtype=bf), ws,
                               z(e, c_max, m, dtype=bf), z(e, h, m), z(e, h, m), z(e, m, h), None, None,
                               st)
    c = stub.calls
    assert c["moe_expert_ffn_bwd"][10:14] == (e, c_max, m, h)
    assert c["moe_expert_ffn_train"][10:14] == (e, c_max, m, h)
    assert c["moe_expert_ffn_bwd_saved"][10:14] == (e, c_max, m, h)
    assert c["moe_expert_ffn_bwd_saved"][18] == M.MOE_F32   # fp32 weight gradients
    assert c["moe_gate_topk"][4:8] == (s, m, e, k)
    assert c["moe_capacity_locations"][1:4] == (s, e, k)
    assert c["moe_capacity_locations_noalloc"][1:4] == (s, e, k)
    assert c["moe_capacity_locations_noalloc"][5] == c_max
    assert c["moe_encode"][6:11] == (s, m, e, k, c_max)
    assert c["moe_expert_ffn"][10:14] == (e, c_max, m, h)
    assert c["moe_decode"][6:11] == (s, m, e, k, c_max)
    assert c["moe_decode_bwd"][8:13] == (s, m, e, k, c_max)
    assert c["moe_encode_bwd"][5:10] == (s, m, e, k, c_max)
    assert c["moe_gate_bwd"][4:8] == (s, m, e, k)
    assert c["moe_layer_forward"][10:15] == (s, m, e, k, h)
    assert c["moe_layer_forward"][16] == c_max
    assert c["moe_layer_forward_pipelined"][10:15] == (s, m, e, k, h)
    assert c["moe_layer_forward_pipelined"][16] == c_max and c["moe_layer_forward_pipelined"][29] == 3
    with pytest.raises(ValueError, match="events: need 4"):
        M.moe_layer_forward_pipelined(x, wg, gb, w1, b1, None, w2, b2, "gelu", k, 1.25, 1, idx,
                                      gates, loc, counts, c_dev, buf, out, z(s, m, dtype=bf), ws, st,
                                      3, None, [_Ev()] * 3)
