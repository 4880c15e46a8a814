"""Benchmark of the MoE layer hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config NAME] [--no-graded] [--no-cpu-baseline]

One step = one forward pass of the whole path (gate -> capacity/locations ->
encode -> expert FFN -> decode) over one batch of the chosen workload.  The
default workload is the largest one that fits a GPU: the dynamic-load sweep's
s=65536 point with capacity factor 2 and uniform routing (m=4096, e=64, k=2,
h=8192 GELU, c=4096, every one of the 131072 routes kept).  Inputs are seeded
synthetic tensors already resident in HBM; L2 is flushed (256 MiB write, then a 256 MiB read)
before every timed step, outside the timed interval.

value        whole-job forward tokens/s (device time, CUDA events, max over ranks)
e2e          the same metric through one C call per step with host buffers
             (moe_layer_forward_host: each step's x copied from pinned host
             memory and its y copied back, inside the timed interval; steps
             alternate over two streams with their own device buffers, so one
             step's copies overlap the previous step's compute)
stages       every stage's time on the workload, each against its binding
             roofline: HBM bytes for gate/encode/decode, fp32 FMA for the gate
             where its flops outweigh its bytes, tensor-core flops and weight
             bytes for the expert FFN
graded       the same stage breakdown on the s=8192 e=16 layer (with its whole
             forward + backward chain) and on the e=256 SwiGLU layer
roofline     the expert FFN (the dominant kernel) on the headline workload
cpu_baseline the CPU oracle timed on the host cores on a bounded token sample

With --gpus N > 1 (torchrun) every rank runs an independent replica of the
layer on its own GPU ("replicas only": the layer has no cross-GPU step).
`--impl reference` times the CPU oracle as the reference arm (rank 0 only).
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth import workloads as W  # noqa: E402

METRIC = "MoE-layer fwd tokens/s; encode/decode HBM GB/s and FFN TC util, 1×GB300"
L2_FLUSH_BYTES = 256 << 20

# name -> (workload, expert-weight seed or None for the workload's own seed)
CONFIGS = {
    "tiny_f32": (W.TINY_FP32, None),
    "bf16_e8": (W.BF16_E8, None),
    "bf16_e16": (W.BF16_E16_BWD, None),
    "bf16_e256_swiglu": (W.BF16_E256_SWIGLU, None),
    # sweep point p = 3*8 + 1*2 + 0: s=65536, f=2, uniform; the sweep shares weight seed 0
    "sweep_s65536_f2": (W.sweep_points()[26], 0),
    # the same expert shape (m=4096, h=8192, about 2048 rows per expert) with 8 experts:
    # the s=65536 layer's kernels at 1/8 of the work, small enough for multi-pass profiling
    "sweep_shape_e8": (W.sweep_points()[26].with_(s=8192, e=8), 0),
}
HEADLINE = "sweep_s65536_f2"
GRADED = ("bf16_e16", "bf16_e256_swiglu")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=HEADLINE, choices=sorted(CONFIGS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graded", action="store_true",
                    help="skip the stage breakdowns of the other graded workloads")
    ap.add_argument("--only", choices=["gate", "gate_bwd", "backward", "fp8"],
                    help="time one stage alone on the config's inputs (its own JSON line, not the "
                         "layer's): only the tensors that stage reads are drawn")
    return ap.parse_args(argv)


class L2Flush:
    """Writes a 256 MiB buffer (larger than L2), then reads another one, so that
    the written lines are back in HBM before the timed interval starts: the
    first timed kernel finds L2 holding none of its inputs and no dirty lines
    whose write-back it would otherwise pay for."""

    def __init__(self, torch, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def fill_(self, v):
        self.w.fill_(v)
        self.r.max()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d.get("bf16_tflops_sustained"),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [l for (ts, l) in self.lines if t0 - 0.06 <= ts <= t1 + 0.06] or [l for _, l in self.lines]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# -------------------------------------------------------------- multi-rank
def reduce_max(vals, device=None):
    """Max over ranks of a list of floats (identity when not distributed)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in vals]
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(world, tokens_per_rank, ms_step):
    """Whole-job tokens/s: every rank runs its own replica on its own tokens."""
    return world * tokens_per_rank / (ms_step * 1e-3)


# ------------------------------------------------------ algorithmic work
def stage_work(w, R, t1, hit):
    """Algorithmic bytes and flops per call of every stage, from the routing
    actually produced: R kept routes, t1 tokens with at least one kept route,
    `hit` experts with at least one kept row (b bytes per element)."""
    b = 4 if w.dtype == "f32" else 2
    s, m, e, k, h = w.s, w.m, w.e, w.k, w.h
    nw = 3 if w.act == "swiglu" else 2                      # weight matrices per expert
    ffn_flop = (6.0 if w.act == "swiglu" else 4.0) * R * m * h
    return {
        "gate": dict(bytes=s * m * b + 4 * m * e + 8 * s * k, flop=2.0 * s * m * e),
        "capacity": dict(bytes=8 * s * k),
        "encode": dict(bytes=t1 * m * b + R * m * b + 8 * s * k),
        "expert_ffn": dict(flop=ffn_flop,
                           bytes=hit * nw * m * h * b + 2 * R * m * b + 2 * R * h * b),
        "decode": dict(bytes=R * m * b + s * m * b + 12 * s * k),
        "decode_bwd": dict(bytes=t1 * m * b + 2 * R * m * b + 16 * s * k),
        "encode_bwd": dict(bytes=R * m * b + s * m * b + 8 * s * k),
        # dgrad and wgrad products, 2*R*m*h flop each: GELU/ReLU d_hid, d_buf,
        # d_w2, d_w1; SwiGLU adds d_b's share of d_buf and d_w3
        "ffn_bwd": dict(flop=(12.0 if w.act == "swiglu" else 8.0) * R * m * h),
        # d_logits [s, e] written and read, x read, d_x written (fp32), wg read
        "gate_bwd": dict(bytes=s * m * b + 4 * s * m + 8 * s * e + 4 * m * e + 12 * s * k,
                         flop=4.0 * s * m * e),
    }


def rate(name, ms, work, pk):
    """A stage's time against its binding roofline (the larger of its HBM and
    its arithmetic time; arithmetic is tensor-core bf16 for the FFN, fp32 FMA
    for the gate)."""
    d = {"ms": ms}
    sec = ms * 1e-3
    t_hbm = t_alu = 0.0
    if "bytes" in work:
        gbs = work["bytes"] / sec / 1e9
        d.update(gbs=gbs, hbm_frac=gbs / pk["hbm"])
        t_hbm = work["bytes"] / (pk["hbm"] * 1e9)
    if "flop" in work:
        tf = work["flop"] / sec / 1e12
        if name in ("expert_ffn", "ffn_bwd"):
            d.update(tflops=tf, tc_frac=tf / pk["bf16"])
            t_alu = work["flop"] / (pk["bf16"] * 1e12)
        elif pk.get("fp32"):
            d.update(fp32_tflops=tf, fp32_frac=tf / pk["fp32"])
            t_alu = work["flop"] / (pk["fp32"] * 1e12)
    if name == "capacity":
        d["bound"] = "latency"
    elif t_hbm or t_alu:
        d["bound"] = "hbm" if t_hbm >= t_alu else ("tensor" if "tc_frac" in d else "fp32")
        d["roofline_frac"] = max(t_hbm, t_alu) / sec
    return d


# ------------------------------------------------------------------ oracle
def oracle_sample_inputs(w, inp, s_sample):
    """The first s_sample tokens of the workload's batch (same weights)."""
    ws = w.with_(s=s_sample, name=f"{w.name}_first{s_sample}")
    sub = dict(inp)
    sub["x"] = inp["x"][:s_sample]
    return ws, sub


def time_oracle(w, inp, target_s, s_min=1):
    """Time the CPU oracle's full forward chain on the first s' tokens of the
    batch (a batch of its own: capacity by the workload's rule at s'), s'
    sized so one pass takes about target_s seconds (at least s_min, at most
    the whole batch); when the whole batch is faster than that, it is repeated
    until target_s has passed.  Returns (tokens/s, s', passes, seconds, threads)."""
    import oracle

    s1 = min(w.s, max(s_min, 16))
    ws, sub = oracle_sample_inputs(w, inp, s1)
    t = time.perf_counter()
    oracle.layer_forward(ws, sub)
    dt = time.perf_counter() - t
    s2 = int(max(s1, min(w.s, s1 * target_s / max(dt, 1e-3))))
    ws, sub = oracle_sample_inputs(w, inp, s2)
    passes, t0 = 0, time.perf_counter()
    while True:
        oracle.layer_forward(ws, sub)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= target_s or s2 < w.s:
            break
    return passes * s2 / dt, s2, passes, dt, oracle.get_threads()


def host_inputs(w, weight_seed, dev=None):
    """The workload's inputs as host arrays for the oracle: drawn on the GPU
    when one is available (the multi-GB expert weights), else on the host;
    bf16 tensors widened to fp32 values once, here, so that the oracle's calls
    do not convert them again."""
    import torch

    import oracle

    if dev is None and torch.cuda.is_available():
        dev = torch.device("cuda", torch.cuda.current_device())
    if dev is not None:
        d = synth.make_inputs_device(w, dev, weight_seed=weight_seed)
        out = {}
        for n, t in d.items():
            out[n] = None if t is None else t.float().cpu().numpy()
            d[n] = None
        del d
        torch.cuda.empty_cache()
        return out
    inp = synth.make_inputs_host(w)
    return {n: None if a is None else oracle.to_f32(a) for n, a in inp.items()}


def cpu_baseline_dict(w, inp, target_s):
    v, s2, passes, dt, thr = time_oracle(w, inp, target_s, s_min=min(w.s, 256))
    return {"value": v, "unit": "tokens/s", "cores": thr, "kind": "oracle",
            "sample": f"full forward chain (gate, capacity, encode, FFN, decode) on the first {s2} "
                      f"of {w.s} tokens as a batch of their own (capacity by the same rule), same "
                      f"weights, {passes} pass(es): {dt:.1f} s on {thr} threads"}


def ffn_traffic_from_profile(workload_name):
    """DRAM bytes per expert-FFN call on this workload from the committed ncu
    summary, or None when there is none or the forward GEMM's source has
    changed since its counters were taken.  The digest covers ffn_tc.cu up to
    its e4m3-forward marker: the GEMM kernel and the bf16 forward launcher
    (the e4m3 launcher and the backward's host code follow)."""
    import hashlib

    prof = os.path.join(ROOT, "profiles", f"expert_ffn_tcgen05_{workload_name}.md")
    src = os.path.join(ROOT, "combine_moe_gate_gb300", "csrc", "ffn_tc.cu")
    try:
        text = open(prof).read()
        data = open(src, "rb").read()
    except OSError:
        return None
    end = data.find(b"// ------------------------------------------------------------ e4m3 forward\n")
    if end < 0:
        return None
    digest = hashlib.sha256(data[:end]).hexdigest()[:16]
    fields = dict(line.split(":", 1) for line in text.splitlines() if line.startswith(
        ("source_sha256_16:", "dram_bytes_per_call:")))
    if fields.get("source_sha256_16", "").split()[0:1] != [digest]:
        return None
    return int(fields["dram_bytes_per_call"].split()[0])


# ------------------------------------------------------------------- ours
class LayerRun:
    """One workload's device inputs and buffers, and its timed passes."""

    STAGES = ["gate", "capacity", "encode", "expert_ffn", "decode"]

    def __init__(self, w, weight_seed, dev, flush):
        import torch

        import combine_moe_gate_gb300 as M

        self.M, self.torch, self.w, self.dev, self.flush = M, torch, w, dev, flush
        self.inp = synth.make_inputs_device(w, dev, weight_seed=weight_seed)
        self.tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        self.dt = M.MOE_BF16 if w.dtype == "bf16" else M.MOE_F32
        self.bufs = M.alloc_layer(w.s, w.m, w.e, w.k, w.h, w.act, w.capacity_factor,
                                  dtype=self.tdt, device=dev)
        self.flags = M.MOE_FLAG_NORMALIZE_GATES if w.normalize_gates and w.k >= 2 else 0
        b = self.bufs
        self.cap_ws = b.workspace[: M.moe_capacity_workspace_size(w.s, w.e, w.k)]
        self.ffn_ws = torch.empty(M.moe_expert_ffn_workspace_size(self.dt, w.act, w.e, b.c_max, w.m,
                                                                  w.h), dtype=torch.uint8, device=dev)

    def args(self):
        i = self.inp
        return (i["x"], i["wg"], i["bias"], i["w1"], i["b1"], i["w3"], i["w2"], i["b2"])

    def whole_step(self):
        x, wg, gb, w1, b1, w3, w2, b2 = self.args()
        self.M.run_layer(x, wg, gb, w1, b1, w3, w2, b2, self.w.act, self.w.k,
                         self.w.capacity_factor, self.bufs, normalize_gates=bool(self.flags))

    def staged_step(self, ev, pre=None):
        """The five C-ABI calls with an event after each stage (ev[0] before);
        with `pre`, the expert FFN is the training forward that also keeps its
        pre-activation there."""
        M, w, b = self.M, self.w, self.bufs
        x, wg, gb, w1, b1, w3, w2, b2 = self.args()
        ev[0].record()
        M.moe_gate_topk(x, wg, gb, w.k, b.idx, b.gates, b.status, flags=self.flags)
        ev[1].record()
        M.moe_capacity_locations(b.idx, w.e, w.capacity_factor, b.c_max, self.cap_ws, b.loc,
                                 b.counts, b.c_dev, b.status)
        ev[2].record()
        M.moe_encode(x, b.idx, b.loc, b.counts, b.c_dev, b.buf, b.status)
        ev[3].record()
        if pre is None:
            M.moe_expert_ffn(b.buf, b.counts, b.c_dev, w1, b1, w3, w2, b2, w.act, self.ffn_ws, b.out,
                             b.status)
        else:
            M.moe_expert_ffn_train(b.buf, b.counts, b.c_dev, w1, b1, w3, w2, b2, w.act, self.ffn_ws,
                                   b.out, pre, b.status)
        ev[4].record()
        M.moe_decode(b.out, b.idx, b.loc, b.gates, b.c_dev, b.y, b.status)
        ev[5].record()

    def fp8_experts(self, steps, warmup):
        """The layer with e4m3 experts (ReLU / GELU): the weights quantised per
        output channel once (untimed), then per call the encoded buffer's
        kept rows quantised and the e4m3 FFN, timed alone (L2 flushed before
        each call), and the whole e4m3 layer step (gate, capacity, encode,
        quantise, FFN, decode) through the same C calls."""
        torch, M, w, b = self.torch, self.M, self.w, self.bufs
        x, wg, gb, w1, b1, w3, w2, b2 = self.args()
        dev = self.dev
        if w.act not in ("relu", "gelu") or w.m % 16 or w.h % 16 or w.dtype != "bf16":
            return None
        st = b.status
        w1q = torch.empty(w1.shape, dtype=torch.uint8, device=dev)
        w2q = torch.empty(w2.shape, dtype=torch.uint8, device=dev)
        w1s = torch.empty(w1.shape[:-1], dtype=torch.float32, device=dev)
        w2s = torch.empty(w2.shape[:-1], dtype=torch.float32, device=dev)
        M.moe_quantize_rows_fp8(w1, w1q, w1s, st)
        M.moe_quantize_rows_fp8(w2, w2q, w2s, st)
        bq = torch.empty(b.buf.shape, dtype=torch.uint8, device=dev)
        bs = torch.empty(b.buf.shape[:-1], dtype=torch.float32, device=dev)
        ws = torch.empty(M.moe_expert_ffn_fp8_workspace_size(w.e, b.c_max, w.m, w.h),
                         dtype=torch.uint8, device=dev)
        out8 = torch.empty_like(b.out)

        def ffn():
            M.moe_quantize_rows_fp8(b.buf, bq, bs, st, counts=b.counts, c_dev=b.c_dev)
            M.moe_expert_ffn_fp8(bq, bs, b.counts, b.c_dev, w1q, w1s, b1, w2q, w2s, b2, w.act, ws,
                                 out8, st)

        def layer():
            M.moe_gate_topk(x, wg, gb, w.k, b.idx, b.gates, st, flags=self.flags)
            M.moe_capacity_locations(b.idx, w.e, w.capacity_factor, b.c_max, self.cap_ws, b.loc,
                                     b.counts, b.c_dev, st)
            M.moe_encode(x, b.idx, b.loc, b.counts, b.c_dev, b.buf, st)
            ffn()
            M.moe_decode(out8, b.idx, b.loc, b.gates, b.c_dev, b.y, st)

        layer()   # the buffer the timed FFN calls read
        res = {"expert_ffn_ms": self.time_calls(ffn, steps, warmup),
               "layer_ms": self.time_calls(layer, steps, warmup)}
        self.check_status()
        return res

    def hid(self):
        w, b = self.w, self.bufs
        n = w.e * b.c_max * w.h
        return self.ffn_ws[: n * (2 if w.dtype == "bf16" else 4)].view(self.tdt).view(w.e, b.c_max, w.h)

    def check_status(self):
        v = int(self.bufs.status.item())
        if v != 0:
            raise RuntimeError(f"{self.w.name}: device status {v} ({self.M.status_str(v)})")

    def time_calls(self, fn, steps, warmup):
        """Mean event time (ms) of fn over `steps` calls, L2 flushed before each."""
        torch = self.torch
        for _ in range(warmup):
            self.flush.fill_(1)
            fn()
        torch.cuda.synchronize()
        tot = 0.0
        for _ in range(steps):
            self.flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            tot += a.elapsed_time(b)
        return tot / steps

    def time_stages(self, steps, warmup):
        torch = self.torch
        mk = lambda: [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        for _ in range(warmup):
            self.flush.fill_(1)
            self.staged_step(mk())
        torch.cuda.synchronize()
        events = []
        for _ in range(steps):
            self.flush.fill_(1)
            ev = mk()
            self.staged_step(ev)
            events.append(ev)
        torch.cuda.synchronize()
        self.check_status()
        out = {n: 0.0 for n in self.STAGES}
        for ev in events:
            for i, n in enumerate(self.STAGES):
                out[n] += ev[i].elapsed_time(ev[i + 1])
        return {n: v / steps for n, v in out.items()}

    def routing_summary(self):
        """(c, R kept routes, t1 tokens with a kept route, experts hit), read
        back after timing."""
        b = self.bufs
        counts = b.counts.cpu().numpy().astype(np.int64)
        c = int(b.c_dev.item())
        kept = np.minimum(counts, c)
        loc = b.loc.cpu().numpy()
        return c, int(kept.sum()), int(((loc < c).any(0)).sum()), int((kept > 0).sum())

    def pipelined(self, chunks_list, steps, warmup):
        """The forward with the capacity dimension cut into d chunks (encode of
        chunk i+1 on a side stream overlapping the FFN of chunk i), d in
        chunks_list: mean ms per call, L2 flushed before each."""
        torch, M, w, b = self.torch, self.M, self.w, self.bufs
        aux = torch.cuda.Stream(device=self.dev)
        x, wg, gb, w1, b1, w3, w2, b2 = self.args()
        res = {}
        for d in chunks_list:
            events = [torch.cuda.Event() for _ in range(d + 1)]

            def fn():
                M.moe_layer_forward_pipelined(x, wg, gb, w1, b1, w3, w2, b2, w.act, w.k,
                                              w.capacity_factor, self.flags, b.idx, b.gates, b.loc,
                                              b.counts, b.c_dev, b.buf, b.out, b.y, b.workspace,
                                              b.status, d, aux, events)

            res[str(d)] = self.time_calls(fn, steps, warmup)
        self.check_status()
        return res

    def dispatch_backward(self, steps, warmup):
        """decode backward (dE, dG from dY) and encode backward (dX from dBuf
        := dE) on the forward just timed, each alone."""
        torch, M, w, b = self.torch, self.M, self.w, self.bufs
        dy = synth.normal_torch(w.seed, "dy", (w.s, w.m), 1.0, w.dtype, self.dev)
        d_out = torch.empty_like(b.out)
        d_g = torch.empty((w.k, w.s), device=self.dev, dtype=torch.float32)
        dx = torch.empty((w.s, w.m), device=self.dev, dtype=self.tdt)
        res = {
            "decode_bwd": self.time_calls(
                lambda: M.moe_decode_bwd(dy, b.out, b.idx, b.loc, b.gates, b.counts, b.c_dev, d_out,
                                         d_g, b.status), steps, warmup),
            "encode_bwd": self.time_calls(
                lambda: M.moe_encode_bwd(d_out, b.idx, b.loc, b.c_dev, dx, b.status), steps, warmup),
        }
        self.check_status()
        return res

    def backward_chain(self, steps, warmup, pk):
        """Backward of the forward just run, timed call by call and as the whole
        forward + backward chain: decode backward (dE, dG from dY), the expert
        FFN backward (d_buf and the weight gradients from dE), encode backward
        (the copy path's d_x from d_buf) and the gate backward (the gate path's
        d_logits, d_wg, d_bias, d_x from dG).  The two d_x terms are left
        separate (their sum is one elementwise add).  For bf16 experts the
        chain's forward is the training forward, which keeps the pre-activation
        (SwiGLU: a and b), and the FFN backward reads it
        (moe_expert_ffn_bwd_saved); the backward that recomputes it, and the
        one that keeps the weight gradients in fp32, are timed alone as well."""
        torch, M, w, b = self.torch, self.M, self.w, self.bufs
        x, wg, gb, w1, b1, w3, w2, b2 = self.args()
        dev, tdt = self.dev, self.tdt
        dy = self.inp["dy"] if self.inp.get("dy") is not None else synth.normal_torch(
            w.seed, "dy", (w.s, w.m), 1.0, w.dtype, dev)
        d_out = torch.empty_like(b.out)
        d_g = torch.empty((w.k, w.s), device=dev, dtype=torch.float32)
        d_buf = torch.empty_like(b.buf)
        dx = torch.empty((w.s, w.m), device=dev, dtype=tdt)
        swiglu = w.act == "swiglu"
        d_w1 = torch.empty_like(w1)
        d_w3 = torch.empty_like(w1) if swiglu else None
        d_w2 = torch.empty_like(w2)
        d_b1 = None if b1 is None else torch.empty_like(b1)
        d_b2 = None if b2 is None else torch.empty_like(b2)
        ws = torch.empty(M.moe_expert_ffn_bwd_workspace_size(self.dt, w.act, w.e, b.c_max, w.m, w.h),
                         dtype=torch.uint8, device=dev)
        d_logits = torch.empty((w.s, w.e), device=dev, dtype=torch.float32)
        d_wg = torch.empty((w.m, w.e), device=dev, dtype=torch.float32)
        d_bias = torch.empty((w.e,), device=dev, dtype=torch.float32)
        d_xg = torch.empty((w.s, w.m), device=dev, dtype=torch.float32)
        hid = self.hid()
        saved = w.dtype == "bf16"
        pre = (torch.empty((w.e, b.c_max, 2 * w.h if swiglu else w.h), device=dev, dtype=tdt)
               if saved else None)

        def dec():
            M.moe_decode_bwd(dy, b.out, b.idx, b.loc, b.gates, b.counts, b.c_dev, d_out, d_g,
                             b.status)

        def ffn_recompute():
            M.moe_expert_ffn_bwd(b.buf, hid, b.counts, b.c_dev, w1, b1, w3, w2, w.act, d_out, ws,
                                 d_buf, d_w1, d_w3, d_w2, d_b1, d_b2, b.status)

        def ffn():
            if pre is None:
                ffn_recompute()
            else:
                M.moe_expert_ffn_bwd_saved(b.buf, hid, pre, b.counts, b.c_dev, w1, w3, w2, w.act, d_out,
                                           ws, d_buf, d_w1, d_w3, d_w2, d_b1, d_b2, b.status)

        # the same with the weight and bias gradients kept in fp32
        g32 = None if pre is None else [torch.empty(t.shape, device=dev, dtype=torch.float32)
                                        if t is not None else None
                                        for t in (d_w1, d_w3, d_w2, d_b1, d_b2)]

        def ffn_f32():
            M.moe_expert_ffn_bwd_saved(b.buf, hid, pre, b.counts, b.c_dev, w1, w3, w2, w.act, d_out,
                                       ws, d_buf, *g32, b.status)

        def enc():
            M.moe_encode_bwd(d_buf, b.idx, b.loc, b.c_dev, dx, b.status)

        def gate():
            M.moe_gate_bwd(x, wg, gb, b.idx, b.gates, d_g, d_logits, b.status, d_wg=d_wg,
                           d_bias=d_bias, d_x=d_xg, flags=self.flags)

        # the forward whose buf / hid / out (/ pre) the backward reads
        self.staged_step([torch.cuda.Event() for _ in range(6)], pre)

        def chain():
            self.staged_step([torch.cuda.Event() for _ in range(6)], pre)
            dec()
            ffn()
            enc()
            gate()

        res = {}
        for name, fn in (("decode_bwd", dec), ("ffn_bwd", ffn), ("encode_bwd", enc),
                         ("gate_bwd", gate)):
            res[name] = self.time_calls(fn, steps, warmup)
        if pre is not None:
            res["ffn_bwd_recompute"] = self.time_calls(ffn_recompute, steps, warmup)
            res["ffn_bwd_fp32_wgrad"] = self.time_calls(ffn_f32, steps, warmup)
        res["fwd_bwd_step"] = self.time_calls(chain, steps, warmup)
        self.check_status()
        return res


def rank_free(run):
    del run
    import torch

    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def fp32_fma_peak(M, dev):
    """Measured fp32 FMA throughput (TFLOP/s): the better of scalar and packed
    fp32x2 fused multiply-adds over every SM, best of 5 launches."""
    import torch

    out = torch.zeros(1, dtype=torch.float32, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks, iters = sms * 8, 8192
    flop = blocks * 256 * iters * 32.0
    best = {}
    for packed in (0, 1):
        M.moe_probe_fp32_fma(packed, blocks, 64, out)
        torch.cuda.synchronize()
        t = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            M.moe_probe_fp32_fma(packed, blocks, iters, out)
            b.record()
            b.synchronize()
            t.append(a.elapsed_time(b))
        best["packed" if packed else "scalar"] = flop / (min(t) * 1e-3) / 1e12
    return best


def graded_report(name, run, stage_ms, pk, extra=None):
    w = run.w
    c, R, t1, hit = run.routing_summary()
    work = stage_work(w, R, t1, hit)
    d = {"workload": w.name, "s": w.s, "m": w.m, "e": w.e, "k": w.k, "h": w.h, "act": w.act,
         "capacity_factor": w.capacity_factor, "c": c, "kept_routes": R, "experts_hit": hit,
         "layer_ms": sum(stage_ms.values()),
         "stages": {n: rate(n, ms, work[n], pk) for n, ms in stage_ms.items()}}
    if extra:
        saved = "ffn_bwd_recompute" in extra
        for n, ms in extra.items():
            base = "ffn_bwd" if n.startswith("ffn_bwd") else n
            if base in work:
                note = "backward, timed alone"
                if base == "ffn_bwd" and saved:
                    note += {"ffn_bwd_recompute": "; recomputes the pre-activation",
                             "ffn_bwd_fp32_wgrad": "; reads the kept pre-activation, weight and bias "
                                                   "gradients stored in fp32"}.get(
                        n, "; reads the pre-activation the training forward kept")
                d["stages"][n] = dict(rate(base, ms, work[base], pk), note=note)
            else:
                d["stages"][n] = {"ms": ms, "tokens_per_s": w.s / (ms * 1e-3),
                                  "note": "forward + decode/FFN/encode/gate backward, one chain"}
    return d


def run_ours(args, rank, world, local_rank):
    import torch

    import combine_moe_gate_gb300 as M

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pk = peaks()
    flush = L2Flush(torch, dev)
    fp32 = fp32_fma_peak(M, dev)
    pk["fp32"] = max(fp32.values())
    w, wseed = CONFIGS[args.config]
    run = LayerRun(w, wseed, dev, flush)

    # ---- warm-up: staged and whole
    run.time_stages(max(1, args.warmup // 2), 1)
    for _ in range(args.warmup):
        flush.fill_(1)
        run.whole_step()
    torch.cuda.synchronize()
    run.check_status()

    # ---- timed (headline): device-resident inputs, the whole layer per step
    n_launch0 = M.launch_count()
    pairs = []
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        t_wall0 = clk.mark()
        for _ in range(args.steps):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            run.whole_step()
            b.record()
            pairs.append((a, b))
        torch.cuda.synchronize()
        t_wall1 = clk.mark()
    if world > 1:
        torch.distributed.barrier()
    launches = M.launch_count() - n_launch0
    ms_step = sum(a.elapsed_time(b) for a, b in pairs) / args.steps
    clocks = clk.summary(t_wall0, t_wall1)
    run.check_status()

    # ---- stages: the same calls with an event after every stage
    stage_ms = run.time_stages(args.steps, 2)

    # ---- e2e: one C call per step with host buffers (pinned): every step copies
    # its x from host memory and its y back inside the timed interval.  Steps
    # alternate between two streams with their own device buffers, so step
    # n+1's input copy and step n's output copy run on the copy engines while
    # step n computes (a double-buffered serving loop); the inputs are larger
    # than L2, so no flush is needed between steps.
    xx, wg, gb, w1, b1, w3, w2, b2 = run.args()
    x_host = run.inp["x"].cpu().pin_memory()
    y_hosts = [torch.empty((w.s, w.m), dtype=run.tdt).pin_memory() for _ in range(2)]
    x_devs = [torch.empty_like(run.inp["x"]) for _ in range(2)]
    bufsets = [run.bufs, M.alloc_layer(w.s, w.m, w.e, w.k, w.h, w.act, w.capacity_factor,
                                       dtype=run.tdt, device=dev, c_max=run.bufs.c_max)]
    streams = [torch.cuda.Stream(device=dev) for _ in range(2)]

    def e2e_run(n):
        main = torch.cuda.current_stream()
        for st_ in streams:
            st_.wait_stream(main)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(main)
        for st_ in streams:
            st_.wait_event(a)
        for i in range(n):
            j = i % 2
            M.run_layer_host(x_host, y_hosts[j], x_devs[j], wg, gb, w1, b1, w3, w2, b2, w.act,
                             w.k, w.capacity_factor, bufsets[j], normalize_gates=bool(run.flags),
                             stream=streams[j])
        for st_ in streams:
            main.wait_stream(st_)
        b.record(main)
        b.synchronize()
        return a.elapsed_time(b)

    e2e_run(max(3, args.warmup // 2))
    e2e_ms = e2e_run(args.steps) / args.steps
    run.check_status()
    v2 = int(bufsets[1].status.item())
    if v2 != 0:
        raise RuntimeError(f"device status {v2} ({M.status_str(v2)})")
    # the last step's output reached the host: it equals the device-resident pass's y
    last = (args.steps - 1) % 2
    if not torch.equal(y_hosts[last], bufsets[last].y.cpu()):
        raise RuntimeError("e2e: host output differs from the device output")

    # ---- decode and encode backward on this workload (timed alone, not part of
    # the step): dE and dG from a dY of the batch's shape, then dX from dBuf := dE
    bw = run.dispatch_backward(args.steps, 3)
    # ---- capacity-dimension pipelining (not the headline: the same layer, chunked)
    pipe = run.pipelined([2, 4, 8], max(5, min(args.steps, 30)), 3)
    # ---- e4m3 experts on the same layer (not the headline: another expert format)
    f8 = run.fp8_experts(max(5, min(args.steps, 20)), 3)

    c, R, t1, hit = run.routing_summary()
    work = stage_work(w, R, t1, hit)
    stages = {n: rate(n, stage_ms[n], work[n], pk) for n in run.STAGES}
    for n, ms in bw.items():
        stages[n] = dict(rate(n, ms, work[n], pk), note="backward, timed alone")
    ffn_tf = work["expert_ffn"]["flop"] / (stage_ms["expert_ffn"] * 1e-3) / 1e12

    # ---- max over ranks
    ms_step, e2e_ms = reduce_max([ms_step, e2e_ms], device=dev)
    res = {
        "metric": METRIC,
        "value": job_throughput(world, w.s, ms_step),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded counter-based normal draws; no dataset)",
        "config": {"workload": w.name, "s": w.s, "m": w.m, "e": w.e, "k": w.k, "h": w.h,
                   "act": w.act, "capacity_factor": w.capacity_factor, "c": c, "kept_routes": R,
                   "experts_hit": hit,
                   "l2": "flushed before every timed step, outside the interval (256 MiB write, then a 256 MiB read so no dirty line is left)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"kernel": "expert_ffn (tcgen05 grouped GEMM, fc1+fc2; duration from the "
                               "stage-bracketed timed pass)", "bound": "tensor",
                     "achieved": ffn_tf, "peak": pk["bf16"], "unit": "TFLOP/s",
                     "frac": ffn_tf / pk["bf16"], "peak_source": f"{pk['src']} bf16 burst",
                     "traffic": ffn_traffic_from_profile(w.name), "traffic_unit": "bytes per call"},
        "stages": stages,
        "fp32_fma_tflops": dict(fp32, source="moe_probe_fp32_fma on this GPU, best of 5"),
        "fp8_experts": None if f8 is None else {
            "expert_ffn_ms": f8["expert_ffn_ms"],
            "expert_ffn_tflops": work["expert_ffn"]["flop"] / (f8["expert_ffn_ms"] * 1e-3) / 1e12,
            "fp8_peak_tflops": 2 * pk["bf16"],
            "tc_frac": work["expert_ffn"]["flop"] / (f8["expert_ffn_ms"] * 1e-3) / 1e12 / (2 * pk["bf16"]),
            "layer_ms": f8["layer_ms"], "tokens_per_s": w.s / (f8["layer_ms"] * 1e-3),
            "note": "e4m3 operands, one fp32 scale per row (moe_quantize_rows_fp8 + "
                    "moe_expert_ffn_fp8, the buffer's quantisation included in the FFN time); "
                    "fp8 peak = 2 x the measured bf16 burst peak (dense e4m3 : bf16 = 2 : 1)"},
        "pipelining": dict({"single_pass_ms": ms_step}, **{f"chunks_{d}_ms": v for d, v in pipe.items()},
                           note="moe_layer_forward_pipelined: encode of capacity chunk i+1 on a side "
                                "stream overlaps the FFN of chunk i; results bit-identical"),
        "e2e": {"value": job_throughput(world, w.s, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
                "d2h_bytes_per_step": y_hosts[0].numel() * y_hosts[0].element_size(),
                "ms_per_step": e2e_ms,
                "api": "moe_layer_forward_host (one C call per step), steps alternating over two "
                       "streams with their own buffers, inputs larger than L2 (no flush)"},
        "clocks": clocks,
        "gpu_launches": launches,
    }
    del x_host, y_hosts, x_devs, bufsets, streams
    rank_free(run)
    run = None

    # ---- the other graded workloads: stage breakdowns (and the e=16 layer's backward)
    if not args.no_graded:
        graded = {}
        gsteps = max(5, min(args.steps, 30))
        for name in GRADED:
            if name == args.config:
                continue
            gw, gseed = CONFIGS[name]
            g = LayerRun(gw, gseed, dev, flush)
            sm = g.time_stages(gsteps, 3)
            extra = g.backward_chain(gsteps, 3, pk) if gw.backward else None
            graded[name] = graded_report(name, g, sm, pk, extra)
            if gw.backward:
                single = g.time_calls(g.whole_step, gsteps, 3)
                graded[name]["pipelining"] = dict({"single_pass_ms": single},
                                                  **{f"chunks_{d}_ms": v for d, v in
                                                     g.pipelined([2, 4, 8], gsteps, 3).items()})
            rank_free(g)
            g = None
        res["graded"] = graded

    if rank == 0 and not args.no_cpu_baseline:
        inp = host_inputs(w, wseed, dev)
        res["cpu_baseline"] = cpu_baseline_dict(w, inp, args.cpu_seconds)
    return res


def run_only_backward(args):
    """The backward chain alone on the config's layer (one forward first):
    decode backward, expert FFN backward, encode backward and gate backward,
    each timed call by call (L2 flushed before each), plus the whole forward +
    backward chain."""
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w, wseed = CONFIGS[args.config]
    run = LayerRun(w, wseed, dev, L2Flush(torch, dev))
    ms = run.backward_chain(args.steps, args.warmup, None)
    return {"stage": "backward", "workload": w.name, "steps": args.steps,
            "ms": {k: round(v, 5) for k, v in ms.items()}}


def run_only_fp8(args):
    """The config's layer with e4m3 experts (ReLU / GELU) alone: one whole
    e4m3 layer step first (its tensor-core GEMM launches are the first two),
    then the e4m3 FFN call by call (buffer quantisation, fc1, hidden
    quantisation, fc2; L2 flushed before each), then the whole e4m3 layer."""
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w, wseed = CONFIGS[args.config]
    run = LayerRun(w, wseed, dev, L2Flush(torch, dev))
    r = run.fp8_experts(args.steps, args.warmup)
    if r is None:
        return {"stage": "fp8", "workload": w.name, "unsupported": "e4m3 experts: ReLU / GELU only"}
    R = int(torch.clamp(run.bufs.counts, max=int(run.bufs.c_dev.item())).sum())
    flop = 4.0 * R * w.m * w.h
    return {"stage": "fp8", "workload": w.name, "steps": args.steps, "kept_rows": R,
            "expert_ffn_ms": r["expert_ffn_ms"], "layer_ms": r["layer_ms"],
            "expert_ffn_tflops": flop / (r["expert_ffn_ms"] * 1e-3) / 1e12,
            "tokens_per_s": w.s / (r["layer_ms"] * 1e-3)}


def run_only_gate(args):
    """The gate (or, with --only gate_bwd, the gate backward: d_logits, d_wg,
    d_bias and d_x from unit-normal d_gates) alone on the config's x, gate
    weight and bias: mean event time over args.steps calls, L2 flushed before
    each."""
    import torch

    import combine_moe_gate_gb300 as M

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w, _ = CONFIGS[args.config]
    inp = synth.make_inputs_device(w, dev, parts=("x", "wg", "bias"))
    idx = torch.empty((w.k, w.s), dtype=torch.int32, device=dev)
    g = torch.empty((w.k, w.s), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = L2Flush(torch, dev)
    flags = M.MOE_FLAG_NORMALIZE_GATES if w.normalize_gates and w.k >= 2 else 0
    fn = lambda: M.moe_gate_topk(inp["x"], inp["wg"], inp["bias"], w.k, idx, g, st, flags=flags)
    flop = 2.0 * w.s * w.m * w.e
    if args.only == "gate_bwd":
        fn()
        d_g = synth.normal_torch(w.seed, "d_gates", (w.k, w.s), 1.0, "f32", dev)
        d_logits = torch.empty((w.s, w.e), device=dev, dtype=torch.float32)
        d_wg = torch.empty((w.m, w.e), device=dev, dtype=torch.float32)
        d_bias = torch.empty((w.e,), device=dev, dtype=torch.float32)
        d_x = torch.empty((w.s, w.m), device=dev, dtype=torch.float32)
        fn = lambda: M.moe_gate_bwd(inp["x"], inp["wg"], inp["bias"], idx, g, d_g, d_logits, st,
                                    d_wg=d_wg, d_bias=d_bias, d_x=d_x, flags=flags)
        flop *= 2.0
    for _ in range(args.warmup):
        flush.fill_(1)
        fn()
    torch.cuda.synchronize()
    tot = 0.0
    for _ in range(args.steps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        tot += a.elapsed_time(b)
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")
    ms = tot / args.steps
    return {"stage": args.only, "workload": w.name, "ms": ms, "steps": args.steps,
            "fp32_tflops": flop / (ms * 1e-3) / 1e12}


def run_reference(args):
    """The CPU oracle as the reference arm: each step is a bounded token sample."""
    import oracle

    w, wseed = CONFIGS[args.config]
    inp = host_inputs(w, wseed)
    per_step = max(0.25, min(2.0, 90.0 / max(1, args.steps)))
    _, s2, _, _, thr = time_oracle(w, inp, per_step)
    ws, sub = oracle_sample_inputs(w, inp, s2)
    for _ in range(min(args.warmup, 1)):
        oracle.layer_forward(ws, sub)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.layer_forward(ws, sub)
    dt = (time.perf_counter() - t) / args.steps
    v = s2 / dt
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded counter-based normal draws; no dataset)",
        "config": {"workload": w.name, "s": w.s, "m": w.m, "e": w.e, "k": w.k, "h": w.h,
                   "act": w.act, "capacity_factor": w.capacity_factor},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": thr, "kind": "oracle",
                         "sample": f"each step: the CPU oracle's forward chain on the first {s2} "
                                   f"tokens of the batch as a batch of their own"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return
    if args.only:
        if rank == 0:
            print(json.dumps(run_only_backward(args) if args.only == "backward" else
                             run_only_fp8(args) if args.only == "fp8" else run_only_gate(args)))
        return
    if world > 1:
        import torch

        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch

        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
