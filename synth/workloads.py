"""The synthetic MoE-layer workloads and their seeded input recipe.

Shapes follow the workloads the pages measure: the DeepSpeed index-dispatch
change (PR #8195, "Results") times s=8192 m=2048 e=16 k=3 in bf16, and the Tutel
blog (DeepSpeed-MoE vs Tutel, section 3.5, memory example) uses 32K tokens with
D=H=4K and top-2.  No dataset is involved: every tensor is drawn from `synth.rng`.

Input recipe (all N(0, .) draws are `normal_host` streams named below):

* x   [s, m]      N(0, 1)               stream "x"     (dtype of the layer)
* wg  [m, e]      N(0, 1/m)             stream "wg"    (fp32 always)
* gate bias [e]   -alpha * ln(e_i + 1)  (skewed workloads only; Zipf-like ranking,
                                         expert 0 most popular), fp32
* w1  [e, h, m]   N(0, 1/m)             stream "w1"    (row j = fc1 weights of hidden unit j)
* w3  [e, h, m]   N(0, 1/m)             stream "w3"    (SwiGLU "up" projection only)
* w2  [e, m, h]   N(0, 1/h)             stream "w2"    (row i = fc2 weights of output i)
* b1  [e, h], b2 [e, m]  0.01 * N(0,1)  streams "b1", "b2" (ReLU/GELU experts only)
* dy  [s, m]      N(0, 1)               stream "dy"    (upstream gradient, backward runs)
"""

from dataclasses import dataclass, field
import math

import numpy as np

from .rng import normal_host

ACT_RELU, ACT_GELU, ACT_SWIGLU = "relu", "gelu", "swiglu"


@dataclass(frozen=True)
class Workload:
    name: str
    s: int
    m: int
    e: int
    k: int
    h: int
    act: str
    capacity_factor: float
    dtype: str = "bf16"          # 'f32' or 'bf16' for x / buffers / expert weights
    skew_alpha: float = 0.0      # gate bias -alpha*ln(rank); 0 = none
    normalize_gates: bool = True  # renormalise the k selected gates (k >= 2)
    backward: bool = False
    seed: int = 0
    biases: bool = field(default=True)

    @property
    def has_bias(self) -> bool:
        return self.biases and self.act != ACT_SWIGLU

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        if "name" not in kw:
            d["name"] = _auto_name(d)
        return Workload(**d)


def _auto_name(d) -> str:
    f = d["capacity_factor"]
    fs = ("m" if f < 0 else "") + f"{abs(f):g}"
    sk = f"_zipf{d['skew_alpha']:g}" if d["skew_alpha"] else ""
    return (f"{d['dtype']}_s{d['s']}_m{d['m']}_e{d['e']}_k{d['k']}_h{d['h']}_{d['act']}"
            f"_f{fs}{sk}")


def _w(**kw) -> Workload:
    kw.setdefault("name", "")
    d = dict(kw)
    if not d["name"]:
        d["name"] = _auto_name({**dict(dtype="bf16", skew_alpha=0.0), **d})
    return Workload(**d)


#: Tiny fp32 layer (k=1: raw softmax probability as gate; ties -> lower index).
TINY_FP32 = _w(s=256, m=64, e=4, k=1, h=128, act=ACT_RELU, capacity_factor=1.0,
               dtype="f32", normalize_gates=False)
#: bf16 layer with fixed capacity c = ceil(1.25*k*s/e) = 1280 -- the bench workload.
BF16_E8 = _w(s=4096, m=1024, e=8, k=2, h=4096, act=ACT_GELU, capacity_factor=1.25)
#: The PR #8195 shape, capacity 0 (no drop), forward + backward of encode/decode.
BF16_E16_BWD = _w(s=8192, m=2048, e=16, k=3, h=4096, act=ACT_GELU, capacity_factor=0.0,
                  backward=True)
#: Fine-grained layer with capped adaptive capacity and Zipf-like skew, SwiGLU experts.
BF16_E256_SWIGLU = _w(s=16384, m=7168, e=256, k=8, h=2048, act=ACT_SWIGLU,
                      capacity_factor=-1.5, skew_alpha=2.0)

SWEEP_S = (1024, 4096, 16384, 65536)
SWEEP_F = (1.0, 2.0, 0.0, -1.25)
SWEEP_SKEW = (0.0, 1.2)


def sweep_points():
    """The 32-point dynamic-load sweep (e=64, k=2, m=4096, h=8192 GELU).

    Point p (row-major over s, capacity factor, skew) uses seed p.
    """
    pts = []
    p = 0
    for s in SWEEP_S:
        for f in SWEEP_F:
            for a in SWEEP_SKEW:
                pts.append(_w(s=s, m=4096, e=64, k=2, h=8192, act=ACT_GELU, capacity_factor=f,
                              skew_alpha=a, seed=p))
                p += 1
    return pts


WORKLOADS = {w.name: w for w in [TINY_FP32, BF16_E8, BF16_E16_BWD, BF16_E256_SWIGLU]}


def gate_bias_host(w: Workload):
    """Skew bias b_e = -alpha*ln(e+1) in fp32, or None for uniform routing."""
    if not w.skew_alpha:
        return None
    r = np.arange(1, w.e + 1, dtype=np.float64)
    return (-w.skew_alpha * np.log(r)).astype(np.float32)


def make_inputs_host(w: Workload, parts=("x", "wg", "bias", "w1", "w3", "w2", "b1", "b2", "dy")):
    """Draw the requested input tensors on the host (numpy).

    bf16 tensors come back as uint16 bit patterns; fp32 as float32.
    """
    dt, sd = w.dtype, w.seed
    out = {}
    if "x" in parts:
        out["x"] = normal_host(sd, "x", (w.s, w.m), 1.0, dt)
    if "wg" in parts:
        out["wg"] = normal_host(sd, "wg", (w.m, w.e), 1.0 / math.sqrt(w.m), "f32")
    if "bias" in parts:
        out["bias"] = gate_bias_host(w)
    if "w1" in parts:
        out["w1"] = normal_host(sd, "w1", (w.e, w.h, w.m), 1.0 / math.sqrt(w.m), dt)
    if "w3" in parts:
        out["w3"] = (normal_host(sd, "w3", (w.e, w.h, w.m), 1.0 / math.sqrt(w.m), dt)
                     if w.act == ACT_SWIGLU else None)
    if "w2" in parts:
        out["w2"] = normal_host(sd, "w2", (w.e, w.m, w.h), 1.0 / math.sqrt(w.h), dt)
    if "b1" in parts:
        out["b1"] = normal_host(sd, "b1", (w.e, w.h), 0.01, dt) if w.has_bias else None
    if "b2" in parts:
        out["b2"] = normal_host(sd, "b2", (w.e, w.m), 0.01, dt) if w.has_bias else None
    if "dy" in parts:
        out["dy"] = normal_host(sd, "dy", (w.s, w.m), 1.0, dt) if w.backward else None
    return out


def make_inputs_device(w: Workload, device="cuda", weight_seed=None,
                       parts=("x", "wg", "bias", "w1", "w3", "w2", "b1", "b2", "dy")):
    """The same recipe drawn with torch on `device` (for multi-GB workloads).

    bf16 tensors come back as torch.bfloat16, fp32 as torch.float32.  Expert
    weights use `weight_seed` when given (the sweep shares one weight set across
    its points), otherwise the workload's seed.  Only the requested parts are
    drawn.
    """
    import torch

    from .rng import normal_torch

    dt, sd = w.dtype, w.seed
    wsd = sd if weight_seed is None else weight_seed
    draw = {
        "x": lambda: normal_torch(sd, "x", (w.s, w.m), 1.0, dt, device),
        "wg": lambda: normal_torch(sd, "wg", (w.m, w.e), 1.0 / math.sqrt(w.m), "f32", device),
        "bias": lambda: None,
        "w1": lambda: normal_torch(wsd, "w1", (w.e, w.h, w.m), 1.0 / math.sqrt(w.m), dt, device),
        "w3": lambda: (normal_torch(wsd, "w3", (w.e, w.h, w.m), 1.0 / math.sqrt(w.m), dt, device)
                       if w.act == ACT_SWIGLU else None),
        "w2": lambda: normal_torch(wsd, "w2", (w.e, w.m, w.h), 1.0 / math.sqrt(w.h), dt, device),
        "b1": lambda: normal_torch(wsd, "b1", (w.e, w.h), 0.01, dt, device) if w.has_bias else None,
        "b2": lambda: normal_torch(wsd, "b2", (w.e, w.m), 0.01, dt, device) if w.has_bias else None,
        "dy": lambda: normal_torch(sd, "dy", (w.s, w.m), 1.0, dt, device) if w.backward else None,
    }
    out = {n: draw[n]() for n in parts}
    b = gate_bias_host(w)
    if "bias" in parts and b is not None:
        out["bias"] = torch.from_numpy(b).to(device)
    return out
