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
    with pytest.raises(TypeError, match="b1: dtype"):
        M.moe_layer_forward(torch.zeros((s, m), **bf), torch.zeros((m, e)), None,
                            torch.zeros((e, h, m), **bf), torch.zeros((e, h)), None,
                            torch.zeros((e, m, h), **bf), None, "gelu", k, 1.0, 0, idx,
                            torch.zeros((k, s)), loc, counts, c_dev, out, out,
                            torch.zeros((s, m), **bf), torch.zeros(16, dtype=torch.uint8), st)
