"""GPU parity on the full-size workloads, through the one-call layer entry point
(moe_layer_forward) that the bench times.

Inputs are drawn on the device (synth.make_inputs_device) and the slices the
oracle needs are copied back to the host.  The oracle then checks:
  * routing over the whole batch: top-k indices, slot locations, per-expert
    counts and capacity bit for bit, gates within the fp32 tolerance;
  * encode over every kept route: the slot row equals the token row bit for bit;
  * the expert FFN on sampled rows (first, last and random kept rows of a few
    experts) within the bf16 tolerance;
  * the layer output y on sampled tokens: the oracle's FFN rows for every kept
    route of the token, combined by the oracle's decode (bf16 tolerance);
  * decode alone on sampled tokens with identity experts (the encoded buffer as
    expert output): bit for bit, both sides accumulate in fp32 in route order;
  * for the backward workload, decode_bwd and encode_bwd over the whole batch.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
import combine_moe_gate_gb300 as M
from synth import workloads as W
from gpu_util import assert_close, bf16_bits_of_f32, status_ok

pytestmark = pytest.mark.gpu


def _host_bits(t):
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


class _Weights:
    """Host copies of single experts' weights, fetched on demand."""

    def __init__(self, inp):
        self.inp = inp
        self.cache = {}

    def get(self, j):
        if j not in self.cache:
            sl = lambda n: None if self.inp[n] is None else _host_bits(self.inp[n][j:j + 1])
            self.cache[j] = {n: sl(n) for n in ("w1", "w3", "w2", "b1", "b2")}
        return self.cache[j]


def _ffn_expected(w, wts, x_h, j, rows_tokens):
    """Oracle FFN outputs of expert j for the listed token rows (in order)."""
    ww = wts.get(j)
    buf = x_h[np.asarray(rows_tokens)][None]            # [1, n, m]
    return oracle.ffn_rows(buf, ww["w1"], ww["b1"], ww["w3"], ww["w2"], ww["b2"], w.act,
                           np.zeros(len(rows_tokens), np.int32), np.arange(len(rows_tokens)),
                           w.dtype == "bf16")


def run_and_check(w, weight_seed=None, n_ffn_experts=3, n_tokens=4, rng_seed=0):
    rng = np.random.default_rng(rng_seed)
    torch.cuda.synchronize()
    inp = synth.make_inputs_device(w, "cuda", weight_seed=weight_seed)
    x_h = _host_bits(inp["x"])
    wg_h = inp["wg"].cpu().numpy()
    bias_h = None if inp["bias"] is None else inp["bias"].cpu().numpy()
    bf16 = w.dtype == "bf16"
    tdt = torch.bfloat16 if bf16 else torch.float32

    # ---- oracle routing over the whole batch
    lg = oracle.gate_logits(x_h, wg_h, bias_h)
    idx_o = oracle.topk(lg, w.k)
    norm = w.normalize_gates and w.k >= 2
    g_o = oracle.gates(lg, idx_o, norm)
    loc_o, need_o = oracle.locations(idx_o, w.e)
    c_o = oracle.capacity(w.capacity_factor, w.s, w.e, w.k, need_o)
    kept_o = oracle.kept_rows(need_o, c_o)
    c_max = max(c_o, 1)

    # ---- the layer on the GPU
    bufs = M.alloc_layer(w.s, w.m, w.e, w.k, w.h, w.act, w.capacity_factor, dtype=tdt,
                         c_max=c_max)
    M.run_layer(inp["x"], inp["wg"], inp["bias"], inp["w1"], inp["b1"], inp["w3"], inp["w2"],
                inp["b2"], w.act, w.k, w.capacity_factor, bufs, normalize_gates=norm)
    torch.cuda.synchronize()
    status_ok(bufs.status)

    # routing: bit-exact
    assert np.array_equal(bufs.idx.cpu().numpy(), idx_o), "top-k indices"
    assert np.array_equal(bufs.loc.cpu().numpy(), loc_o), "slot locations"
    assert np.array_equal(bufs.counts.cpu().numpy(), need_o.astype(np.int32)), "counts"
    assert int(bufs.c_dev.item()) == c_o, "capacity"
    assert_close(bufs.gates.cpu().numpy(), g_o, "f32", "gates")

    # encode: every kept slot holds its token's row
    kept = loc_o < c_o
    r_k, t_k = np.nonzero(kept)
    j_k, l_k = idx_o[r_k, t_k], loc_o[r_k, t_k]
    rows = bufs.buf[torch.from_numpy(j_k).cuda().long(), torch.from_numpy(l_k).cuda().long()]
    assert np.array_equal(_host_bits(rows), x_h[t_k]), "encoded rows"
    del rows

    # slot -> token map (oracle's)
    slot_tok = {}
    for r, t, j, l in zip(r_k, t_k, j_k, l_k):
        slot_tok[(int(j), int(l))] = int(t)

    wts = _Weights(inp)
    # expert FFN: sampled rows of a few experts (most loaded, least loaded, random)
    live = np.nonzero(kept_o > 0)[0]
    pick = {int(live[np.argmax(kept_o[live])]), int(live[np.argmin(kept_o[live])])}
    while len(pick) < min(n_ffn_experts, len(live)):
        pick.add(int(rng.choice(live)))
    for j in sorted(pick):
        kj = int(kept_o[j])
        rws = sorted({0, kj - 1, int(rng.integers(kj)), int(rng.integers(kj))})
        want = _ffn_expected(w, wts, x_h, j, [slot_tok[(j, r)] for r in rws])
        got = bufs.out[j, torch.tensor(rws).cuda()].float().cpu().numpy()
        assert_close(got, want, w.dtype, f"ffn expert {j}")

    # layer output on sampled tokens: oracle FFN rows of each kept route + oracle decode
    toks = rng.choice(w.s, size=min(n_tokens, w.s), replace=False)
    outs, q = [], 0
    idx_m = np.zeros((w.k, len(toks)), np.int32)
    loc_m = np.ones((w.k, len(toks)), np.int32)     # loc 1 >= c 1: dropped
    g_m = np.zeros((w.k, len(toks)), np.float32)
    for ti, t in enumerate(toks):
        for r in range(w.k):
            g_m[r, ti] = g_o[r, t]
            if kept[r, t]:
                outs.append(_ffn_expected(w, wts, x_h, int(idx_o[r, t]), [int(t)])[0])
                idx_m[r, ti], loc_m[r, ti] = q, 0
                q += 1
    if outs:
        out_m = np.stack(outs)[:, None, :]
        y_want = oracle.decode(out_m, idx_m, loc_m, g_m, 1, bf16)
    else:
        y_want = np.zeros((len(toks), w.m), np.float32)
    y_got = bufs.y[torch.from_numpy(toks).cuda().long()].float().cpu().numpy()
    assert_close(y_got, y_want, w.dtype, "layer output y")

    # decode alone, identity experts: decode the encoded buffer; the oracle's slot
    # rows are the host token rows they hold.  Bit-exact on sampled tokens (both
    # sides accumulate in fp32 in ascending route order).
    # (the oracle's gates are fed to the GPU: both sides then multiply identical values)
    y2 = torch.empty((w.s, w.m), dtype=tdt, device="cuda")
    g_dev = torch.from_numpy(g_o).cuda()
    M.moe_decode(bufs.buf, bufs.idx, bufs.loc, g_dev, bufs.c_dev, y2, bufs.status)
    torch.cuda.synchronize()
    status_ok(bufs.status)
    toks2 = rng.choice(w.s, size=min(64, w.s), replace=False)
    rows_needed = {}
    idx_m2 = np.zeros((w.k, len(toks2)), np.int32)
    loc_m2 = np.ones((w.k, len(toks2)), np.int32)
    for ti, t in enumerate(toks2):
        for r in range(w.k):
            if kept[r, t]:
                key = (int(idx_o[r, t]), int(loc_o[r, t]))
                idx_m2[r, ti] = rows_needed.setdefault(key, len(rows_needed))
                loc_m2[r, ti] = 0
    keys = sorted(rows_needed, key=rows_needed.get)
    if keys:
        out_rows = x_h[np.array([slot_tok[k_] for k_ in keys])][:, None, :]
        y2_want = oracle.decode(out_rows, idx_m2, loc_m2, g_o[:, toks2], 1, bf16)
        y2_got = y2[torch.from_numpy(toks2).cuda().long()]
        want_bits = bf16_bits_of_f32(y2_want) if bf16 else y2_want.view(np.int32)
        got_bits = (y2_got.view(torch.int16) if bf16 else y2_got.view(torch.int32)).cpu().numpy()
        assert np.array_equal(got_bits, want_bits), "decode of the encoded buffer"
    del y2

    res = dict(idx=idx_o, loc=loc_o, g=g_o, c=c_o, c_max=c_max, need=need_o)
    return inp, bufs, res


def test_tiny_fp32_full_layer():
    w = W.TINY_FP32
    inp = synth.make_inputs_host(w)
    ref = oracle.layer_forward(w, inp)
    run_and_check(w, n_ffn_experts=4, n_tokens=16)
    # tiny: the whole output checked against the whole oracle chain
    bufs = M.alloc_layer(w.s, w.m, w.e, w.k, w.h, w.act, w.capacity_factor, dtype=torch.float32)
    dev = lambda a: None if a is None else torch.from_numpy(a).cuda()
    M.run_layer(dev(inp["x"]), dev(inp["wg"]), None, dev(inp["w1"]), dev(inp["b1"]), None,
                dev(inp["w2"]), dev(inp["b2"]), w.act, w.k, w.capacity_factor, bufs,
                normalize_gates=False)
    torch.cuda.synchronize()
    assert_close(bufs.y.cpu().numpy(), ref["y"], "f32", "y")


def test_bf16_e8_bench_workload():
    run_and_check(W.BF16_E8, n_ffn_experts=4, n_tokens=8)


def test_bf16_e16_forward_and_backward():
    w = W.BF16_E16_BWD
    inp, bufs, res = run_and_check(w, n_ffn_experts=4, n_tokens=6)
    # backward of decode and encode over the whole batch
    c, c_max = res["c"], res["c_max"]
    out_in = synth.normal_torch(w.seed + 1000, "out", (w.e, c_max, w.m), 1.0, w.dtype, "cuda")
    out_h = _host_bits(out_in)         # drawn expert outputs (an input of the backward)
    dy_h = _host_bits(inp["dy"])
    d_out = torch.empty_like(out_in)
    d_g = torch.empty((w.k, w.s), dtype=torch.float32, device="cuda")
    dx = torch.empty((w.s, w.m), dtype=torch.bfloat16, device="cuda")
    g_dev = torch.from_numpy(res["g"]).cuda()    # oracle gates: identical products on both sides
    M.moe_decode_bwd(inp["dy"], out_in, bufs.idx, bufs.loc, g_dev, bufs.counts, bufs.c_dev,
                     d_out, d_g, bufs.status)
    d_out_o, d_g_o = oracle.decode_bwd(dy_h, out_h, res["idx"], res["loc"], res["g"], c, True)
    # encode backward of the oracle's d_out (identity-expert chain: dx_t = kappa_t dy_t)
    d_in = torch.from_numpy(bf16_bits_of_f32(d_out_o)).cuda().view(torch.bfloat16)
    M.moe_encode_bwd(d_in, bufs.idx, bufs.loc, bufs.c_dev, dx, bufs.status)
    dx_o = oracle.encode_bwd(d_out_o, res["idx"], res["loc"], c, True)
    torch.cuda.synchronize()
    status_ok(bufs.status)
    kept_rows = oracle.kept_rows(res["need"], c)
    got = d_out.view(torch.int16).cpu().numpy()
    want = bf16_bits_of_f32(d_out_o)
    for j in range(w.e):
        assert np.array_equal(got[j, :kept_rows[j]], want[j, :kept_rows[j]]), f"d_out expert {j}"
    assert_close(d_g.cpu().numpy(), d_g_o, "bf16", "d_gates")
    assert np.array_equal(dx.view(torch.int16).cpu().numpy(), bf16_bits_of_f32(dx_o)), "dx"


def test_bf16_e256_swiglu_skewed():
    run_and_check(W.BF16_E256_SWIGLU, n_ffn_experts=3, n_tokens=2)


@pytest.mark.parametrize("p", range(32))
def test_dynamic_load_sweep_point(p):
    w = W.sweep_points()[p]
    run_and_check(w, weight_seed=0, n_ffn_experts=2, n_tokens=2, rng_seed=p)
