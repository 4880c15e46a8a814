"""The oracle's sparse index path against the dense one-hot formulation at the
workloads' own shapes (DeepSpeed PR #8195, "Testing": the sparse dispatch must
match the dense einsum; "MoE training systems: DeepSpeed-MoE vs Tutel", section
3.5: dispatch as einsum('TEC,TM->ECM') over the one-hot mask, combine its
gate-weighted transpose).

* the whole tiny fp32 layer (s=256, m=64, e=4, k=1): gate, capacity and the
  oracle's expert MLP feed both paths, and the layer output y of the sparse
  chain equals the dense dispatch -> MLP on every slot -> dense combine;
* the bf16 e=8 layer's shape (s=4096, m=1024, e=8, k=2, c=1280, a [s, e, c]
  mask of 42 M entries) with its real routing: encode, decode, decode
  backward and encode backward, sparse == dense.

Dense sums are float64 (BLAS); the sparse path accumulates in fp32 in route
order (and rounds bf16 outputs once), so the comparisons allow that rounding:
one fp32 (or bf16) rounding of a sum of k terms.
"""

import numpy as np

import oracle
import synth
from oracle import dense
from synth import workloads as W


def _route(w, x, wg, bias=None):
    lg = oracle.gate_logits(x, wg, bias)
    idx = oracle.topk(lg, w.k)
    g = oracle.gates(lg, idx, w.normalize_gates and w.k >= 2)
    loc, needed = oracle.locations(idx, w.e)
    c = oracle.capacity(w.capacity_factor, w.s, w.e, w.k, needed)
    return idx, g, loc, needed, c


def test_tiny_layer_sparse_chain_equals_dense_chain():
    w = W.TINY_FP32
    inp = synth.make_inputs_host(w)
    ref = oracle.layer_forward(w, inp)
    idx, g, loc, c = ref["idx"], ref["gates"], ref["loc"], ref["c"]
    D = dense.dispatch_mask(idx, loc, c, w.e)
    C = dense.combine_weights(idx, loc, g, c, w.e)
    x = oracle.to_f32(inp["x"])
    buf_d = dense.encode(D, x)                                   # [e, c, m]
    assert np.array_equal(ref["buf"][:, :c], buf_d)
    # the expert MLP on every slot of the dense buffer (empty slots hold zero
    # rows; their combine weight is zero)
    re = np.repeat(np.arange(w.e, dtype=np.int32), c)
    rj = np.tile(np.arange(c, dtype=np.int64), w.e)
    out_d = oracle.ffn_rows(buf_d.astype(np.float32), inp["w1"], inp["b1"], None, inp["w2"],
                            inp["b2"], w.act, re, rj, False).reshape(w.e, c, w.m)
    kept = oracle.kept_rows(ref["needed"], c)
    for j in range(w.e):
        assert np.array_equal(out_d[j, :kept[j]], ref["out"][j, :kept[j]])
    y_d = dense.decode(C, out_d)
    # k = 1: one product per token, rounded once to fp32 on the sparse side
    assert np.all(np.abs(ref["y"] - y_d) <= 2.0 ** -24 * np.abs(y_d) + 1e-30)
    # tokens whose route was dropped get exactly zero on both sides
    dropped = (loc >= c).all(0)
    assert dropped.any() and not ref["y"][dropped].any() and not y_d[dropped].any()


def test_bf16_e8_shape_sparse_equals_dense():
    w = W.BF16_E8
    s, m, e, k = w.s, w.m, w.e, w.k
    inp = synth.make_inputs_host(w, parts=("x", "wg"))
    idx, g, loc, needed, c = _route(w, inp["x"], inp["wg"])
    assert c == 1280
    D = dense.dispatch_mask(idx, loc, c, e)
    C = dense.combine_weights(idx, loc, g, c, e)
    assert D.shape == (s, e, c) and D.sum() == (loc < c).sum()
    x = oracle.to_f32(inp["x"])
    cmax = c + 5
    buf = oracle.encode(x, idx, loc, c, e, cmax)
    assert np.array_equal(buf[:, :c], dense.encode(D, x))
    out = oracle.to_f32(synth.normal_host(11, "out", (e, cmax, m), 1.0, "bf16"))
    y = oracle.decode(out, idx, loc, g, c, True)
    yd = dense.decode(C, out[:, :c])
    # fused multiply-adds of k=2 products in fp32 (each rounding at most 2^-24
    # of the sum of the products' magnitudes), then one bf16 rounding
    mag = dense.decode(np.abs(C), np.abs(out[:, :c]))
    assert np.all(np.abs(y - yd) <= 2.0 ** -8 * np.abs(yd) + 2 * 2.0 ** -23 * mag + 1e-30)
    dy = oracle.to_f32(synth.normal_host(11, "dy", (s, m), 1.0, "bf16"))
    d_out, d_g = oracle.decode_bwd(dy, out, idx, loc, g, c, True)
    d_out_d, dC = dense.decode_bwd(C, D, dy, out[:, :c])
    assert np.all(np.abs(d_out[:, :c] - d_out_d) <= 2.0 ** -8 * np.abs(d_out_d))
    kept = loc < c
    r_k, t_k = np.nonzero(kept)
    want = dC[t_k, idx[r_k, t_k], loc[r_k, t_k]]
    # fp32 dot product of m = 1024 terms against the exact one
    bound = 1024 * 2.0 ** -24 * np.abs(dy[t_k] * out[idx[r_k, t_k], loc[r_k, t_k]]).sum(1)
    assert np.all(np.abs(d_g[r_k, t_k] - want) <= bound + 1e-30)
    assert not d_g[~kept].any()
    dbuf = oracle.to_f32(synth.normal_host(11, "dbuf", (e, cmax, m), 1.0, "bf16"))
    dx = oracle.encode_bwd(dbuf, idx, loc, c, True)
    dxd = dense.encode_bwd(D, dbuf[:, :c])
    mag = dense.encode_bwd(D, np.abs(dbuf[:, :c]))
    assert np.all(np.abs(dx - dxd) <= 2.0 ** -8 * np.abs(dxd) + 2 * 2.0 ** -23 * mag + 1e-30)
