"""GPU parity on the full-size workloads, through the one-call layer entry point
(moe_layer_forward) that the bench times.

Inputs are drawn on the device (synth.make_inputs_device) and copied back to
the host for the oracle.  The oracle then checks:
  * routing over the whole batch: top-k indices, slot locations, per-expert
    counts and capacity bit for bit, gates within the fp32 tolerance;
  * encode over every kept route: the slot row equals the token row bit for bit;
  * the expert FFN output (bf16 / fp32 tolerance against the oracle's MLP of
    the same slot row): on every kept row for the tiny, e=8 and e=16 layers;
    on the e=256 layer and the sweep points, on every kept route of 1024
    sampled tokens plus one row of every 256-row tile of every expert those
    routes leave uncovered;
  * the layer output y (the oracle's decode of the oracle's FFN rows): on the
    whole batch for the tiny, e=8 and e=16 layers, on the 1024 sampled tokens
    otherwise;
  * decode alone with identity experts (the encoded buffer as expert output):
    bit for bit, both sides accumulate in fp32 in route order (whole batch or
    the sampled tokens);
  * for the e=16 layer, decode_bwd and encode_bwd over the whole batch.
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

TILE_ROWS = 256        # output rows of one expert-FFN tile (a CTA pair's M)
SAMPLE_TOKENS = 1024


def _host_bits(t):
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


class _Weights:
    """Expert weights on the device (drawn once per weight set) and host fp32
    copies of single experts, fetched on demand; the sweep's 32 points share
    one weight set."""

    NAMES = ("w1", "w3", "w2", "b1", "b2")

    def __init__(self):
        self.key = None
        self.dev = {}
        self.host = {}

    def get_device(self, w, weight_seed):
        key = (w.e, w.m, w.h, w.act, w.dtype, w.biases, w.seed if weight_seed is None else weight_seed)
        if key != self.key:
            self.key, self.dev, self.host = None, {}, {}
            torch.cuda.empty_cache()
            self.dev = synth.make_inputs_device(w, "cuda", weight_seed=weight_seed, parts=self.NAMES)
            self.key = key
        return self.dev

    def expert(self, j):
        if j not in self.host:
            self.host[j] = {n: None if t is None else oracle.to_f32(_host_bits(t[j:j + 1]))
                            for n, t in self.dev.items()}
        return self.host[j]


_WEIGHTS = _Weights()


def _ffn_rows_by_slot(w, x_h, slots, slot_tok):
    """Oracle FFN outputs for the listed (expert, slot) pairs: each slot's row
    is its token's x row.  Returns {slot: row}."""
    by_e = {}
    for (j, l) in slots:
        by_e.setdefault(j, []).append(l)
    got = {}
    for j, ls in sorted(by_e.items()):
        ww = _WEIGHTS.expert(j)
        buf = x_h[np.asarray([slot_tok[(j, l)] for l in ls])][None]       # [1, n, m]
        o = oracle.ffn_rows(buf, ww["w1"], ww["b1"], ww["w3"], ww["w2"], ww["b2"], w.act,
                            np.zeros(len(ls), np.int32), np.arange(len(ls), dtype=np.int64),
                            w.dtype == "bf16")
        for l, row in zip(ls, o):
            got[(j, l)] = row
    return got


def _compact_decode(w, toks, idx_o, loc_o, kept, g_o, rows):
    """The oracle's decode of token list `toks` from the slot rows `rows`
    ({(j, l): row}), as a compact [n, 1, m] expert buffer."""
    idx_m = np.zeros((w.k, len(toks)), np.int32)
    loc_m = np.ones((w.k, len(toks)), np.int32)     # loc 1 >= c 1: dropped
    outs, pos = [], {}
    for ti, t in enumerate(toks):
        for r in range(w.k):
            if kept[r, t]:
                key = (int(idx_o[r, t]), int(loc_o[r, t]))
                if key not in pos:
                    pos[key] = len(outs)
                    outs.append(rows[key])
                idx_m[r, ti], loc_m[r, ti] = pos[key], 0
    if not outs:
        return np.zeros((len(toks), w.m), np.float32)
    out_m = np.stack(outs)[:, None, :]
    return oracle.decode(out_m, idx_m, loc_m, g_o[:, toks], 1, w.dtype == "bf16")


def run_and_check(w, weight_seed=None, full=False, rng_seed=0):
    rng = np.random.default_rng(rng_seed)
    torch.cuda.synchronize()
    inp = dict(_WEIGHTS.get_device(w, weight_seed))
    inp.update(synth.make_inputs_device(w, "cuda", parts=("x", "wg", "bias", "dy")))
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
    slot_tok = {(int(j), int(l)): int(t) for t, j, l in zip(t_k, j_k, l_k)}

    # tokens whose output is checked, and the slots whose FFN rows are checked
    if full:
        toks = np.arange(w.s)
        slots = sorted(slot_tok)
    else:
        toks = np.sort(rng.choice(w.s, size=min(SAMPLE_TOKENS, w.s), replace=False))
        slots = {(int(idx_o[r, t]), int(loc_o[r, t])) for t in toks for r in range(w.k) if kept[r, t]}
        covered = {(j, l // TILE_ROWS) for (j, l) in slots}
        for j in np.nonzero(kept_o > 0)[0]:
            for tile in range((int(kept_o[j]) + TILE_ROWS - 1) // TILE_ROWS):
                if (int(j), tile) not in covered:
                    lo, hi = tile * TILE_ROWS, min((tile + 1) * TILE_ROWS, int(kept_o[j]))
                    slots.add((int(j), int(rng.integers(lo, hi))))
        slots = sorted(slots)
    ffn_o = _ffn_rows_by_slot(w, x_h, slots, slot_tok)

    # expert FFN output on those slots
    sj = torch.tensor([j for j, _ in slots], device="cuda", dtype=torch.long)
    sl = torch.tensor([l for _, l in slots], device="cuda", dtype=torch.long)
    got = bufs.out[sj, sl].float().cpu().numpy()
    assert_close(got, np.stack([ffn_o[s_] for s_ in slots]), w.dtype, "expert FFN rows")
    tiles = {(j, l // TILE_ROWS) for (j, l) in slots}
    want_tiles = sum((int(kj) + TILE_ROWS - 1) // TILE_ROWS for kj in kept_o)
    assert len(tiles) == want_tiles, "an FFN tile without a checked row"

    # layer output: the oracle's decode of the oracle's FFN rows
    y_want = _compact_decode(w, toks, idx_o, loc_o, kept, g_o, ffn_o)
    y_got = bufs.y[torch.from_numpy(toks).cuda().long()].float().cpu().numpy()
    assert_close(y_got, y_want, w.dtype, "layer output y")

    # decode alone, identity experts: decode the encoded buffer with the oracle's
    # gates (both sides then multiply identical values); bit-exact
    y2 = torch.empty((w.s, w.m), dtype=tdt, device="cuda")
    M.moe_decode(bufs.buf, bufs.idx, bufs.loc, torch.from_numpy(g_o).cuda(), bufs.c_dev, y2,
                 bufs.status)
    torch.cuda.synchronize()
    status_ok(bufs.status)
    x_rows = {s_: oracle.to_f32(x_h[slot_tok[s_]]) for s_ in slot_tok} if full else None
    if not full:
        x_rows = {(int(idx_o[r, t]), int(loc_o[r, t])): oracle.to_f32(x_h[t])
                  for t in toks for r in range(w.k) if kept[r, t]}
    y2_want = _compact_decode(w, toks, idx_o, loc_o, kept, g_o, x_rows)
    y2_got = y2[torch.from_numpy(toks).cuda().long()]
    want_bits = bf16_bits_of_f32(y2_want) if bf16 else y2_want.view(np.int32)
    got_bits = (y2_got.view(torch.int16) if bf16 else y2_got.view(torch.int32)).cpu().numpy()
    assert np.array_equal(got_bits, want_bits), "decode of the encoded buffer"
    del y2, y2_got

    res = dict(idx=idx_o, loc=loc_o, g=g_o, c=c_o, c_max=c_max, need=need_o)
    return inp, bufs, res


def test_tiny_fp32_full_layer():
    run_and_check(W.TINY_FP32, full=True)


def test_bf16_e8_bench_workload():
    run_and_check(W.BF16_E8, full=True)


def test_bf16_e16_forward_and_backward():
    w = W.BF16_E16_BWD
    inp, bufs, res = run_and_check(w, full=True)
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
    run_and_check(W.BF16_E256_SWIGLU)


@pytest.mark.parametrize("p", range(32))
def test_dynamic_load_sweep_point(p):
    w = W.sweep_points()[p]
    run_and_check(w, weight_seed=0, rng_seed=p)
