"""The bench's roofline arithmetic on the host: the algorithmic work of every
stage (the per-unit figures of the measurement plan, times the units a call
processes) and the binding-roofline choice, checked against numbers written
out by hand for the headline layer (s=65536, m=4096, e=64, k=2, h=8192 GELU,
bf16, all 131072 routes kept)."""

import bench
from synth import workloads as W

HEAD = W.sweep_points()[26]
R, T1, HIT = 131072, 65536, 64     # kept routes, tokens with a kept route, experts hit
PK = {"hbm": 6779.0, "bf16": 1854.9, "fp32": 78.8}


def test_headline_workload_is_the_large_sweep_point():
    w, _ = bench.CONFIGS[bench.HEADLINE]
    assert (w.s, w.m, w.e, w.k, w.h, w.act, w.capacity_factor) == (65536, 4096, 64, 2, 8192, "gelu", 2.0)


def test_stage_work_by_hand():
    work = bench.stage_work(HEAD, R, T1, HIT)
    b = 2
    assert work["gate"]["bytes"] == 65536 * 4096 * b + 4 * 4096 * 64 + 8 * 65536 * 2
    assert work["gate"]["flop"] == 2.0 * 65536 * 4096 * 64
    assert work["encode"]["bytes"] == T1 * 4096 * b + R * 4096 * b + 8 * 65536 * 2
    assert work["decode"]["bytes"] == R * 4096 * b + 65536 * 4096 * b + 12 * 65536 * 2
    # fc1 + fc2 over the kept rows only: 2 products of 2 * R * m * h
    assert work["expert_ffn"]["flop"] == 4.0 * R * 4096 * 8192 == 17592186044416.0
    # the hit experts' W1 and W2, the buffer rows read and the output rows written, the hidden both ways
    assert work["expert_ffn"]["bytes"] == HIT * 2 * 4096 * 8192 * b + 2 * R * 4096 * b + 2 * R * 8192 * b
    assert work["decode_bwd"]["bytes"] == T1 * 4096 * b + 2 * R * 4096 * b + 16 * 65536 * 2
    assert work["encode_bwd"]["bytes"] == R * 4096 * b + 65536 * 4096 * b + 8 * 65536 * 2
    assert work["ffn_bwd"]["flop"] == 8.0 * R * 4096 * 8192


def test_swiglu_counts_three_matrices():
    w = W.BF16_E256_SWIGLU
    work = bench.stage_work(w, 16417, 9000, 57)
    assert work["expert_ffn"]["flop"] == 6.0 * 16417 * w.m * w.h
    assert work["expert_ffn"]["bytes"] == 57 * 3 * w.m * w.h * 2 + 2 * 16417 * w.m * 2 + 2 * 16417 * w.h * 2
    assert work["ffn_bwd"]["flop"] == 12.0 * 16417 * w.m * w.h


def test_rate_picks_the_binding_roofline():
    work = bench.stage_work(HEAD, R, T1, HIT)
    # the FFN at 10.4 ms: tensor-bound, 1691.5 TFLOP/s = 0.912 of the bf16 peak
    d = bench.rate("expert_ffn", 10.4, work["expert_ffn"], PK)
    assert d["bound"] == "tensor"
    assert abs(d["tflops"] - 17592.186044416 / 10.4) < 1e-6
    assert abs(d["roofline_frac"] - d["tc_frac"]) < 1e-12 and abs(d["tc_frac"] - 0.91192) < 1e-4
    # the gate: fp32-bound (34.4 GFLOP is 0.44 ms at the FMA peak, its 0.54 GB 0.08 ms at HBM)
    g = bench.rate("gate", 1.0, work["gate"], PK)
    assert g["bound"] == "fp32" and abs(g["roofline_frac"] - g["fp32_frac"]) < 1e-12
    # encode: bytes only, HBM-bound
    e = bench.rate("encode", 0.27, work["encode"], PK)
    assert e["bound"] == "hbm" and abs(e["hbm_frac"] - work["encode"]["bytes"] / 0.27e-3 / 1e9 / 6779.0) < 1e-12
    c = bench.rate("capacity", 0.016, work["capacity"], PK)
    assert c["bound"] == "latency"


class _Run:
    def __init__(self, w):
        self.w = w

    def routing_summary(self):
        return 1621, 24576, 8192, 16


def test_graded_report_labels_the_backward_variants():
    w = W.BF16_E16_BWD
    extra = {"ffn_bwd": 1.08, "ffn_bwd_recompute": 1.33, "ffn_bwd_fp32_wgrad": 1.14,
             "decode_bwd": 0.045, "fwd_bwd_step": 1.83}
    d = bench.graded_report("bf16_e16", _Run(w), {"gate": 0.027, "expert_ffn": 0.52}, PK, extra)
    st = d["stages"]
    flop = 8.0 * 24576 * w.m * w.h
    for n in ("ffn_bwd", "ffn_bwd_recompute", "ffn_bwd_fp32_wgrad"):
        assert st[n]["bound"] == "tensor"
        assert abs(st[n]["tflops"] - flop / (extra[n] * 1e-3) / 1e12) < 1e-6
    assert "recomputes" in st["ffn_bwd_recompute"]["note"]
    assert "fp32" in st["ffn_bwd_fp32_wgrad"]["note"]
    assert "kept" in st["ffn_bwd"]["note"]
    assert st["fwd_bwd_step"]["tokens_per_s"] == w.s / 1.83e-3
