"""Device buffers for one MoE layer forward, allocated with torch (plumbing only).

The layer itself runs in libmoe_gate.so (`moe_layer_forward`); this module
sizes and allocates the tensors the C ABI writes into.
"""

from dataclasses import dataclass
from typing import Optional

import torch

from . import (MOE_BF16, MOE_F32, MOE_FLAG_NORMALIZE_GATES, moe_capacity_bound,
               moe_layer_forward, moe_layer_forward_host, moe_layer_workspace_size)


@dataclass
class MoELayerBuffers:
    idx: torch.Tensor      # [k, s] int32
    gates: torch.Tensor    # [k, s] fp32
    loc: torch.Tensor      # [k, s] int32
    counts: torch.Tensor   # [e] int32
    c_dev: torch.Tensor    # [1] int32
    buf: torch.Tensor      # [e, c_max, m]
    out: torch.Tensor      # [e, c_max, m]
    y: torch.Tensor        # [s, m]
    workspace: torch.Tensor
    status: torch.Tensor   # [1] int32

    @property
    def c_max(self) -> int:
        return self.buf.shape[1]


def alloc_layer(s, m, e, k, h, act, capacity_factor, dtype=torch.bfloat16, device="cuda",
                c_max: Optional[int] = None) -> MoELayerBuffers:
    """Allocate every output and scratch tensor of one layer forward.

    c_max defaults to the capacity bound, which can never overflow."""
    if c_max is None:
        c_max = moe_capacity_bound(capacity_factor, s, e, k)
    dt = MOE_BF16 if dtype == torch.bfloat16 else MOE_F32
    ws = moe_layer_workspace_size(dt, act, s, m, e, k, c_max, h)
    i32 = dict(dtype=torch.int32, device=device)
    return MoELayerBuffers(
        idx=torch.empty((k, s), **i32),
        gates=torch.empty((k, s), dtype=torch.float32, device=device),
        loc=torch.empty((k, s), **i32),
        counts=torch.empty((e,), **i32),
        c_dev=torch.empty((1,), **i32),
        buf=torch.empty((e, c_max, m), dtype=dtype, device=device),
        out=torch.empty((e, c_max, m), dtype=dtype, device=device),
        y=torch.empty((s, m), dtype=dtype, device=device),
        workspace=torch.empty((ws,), dtype=torch.uint8, device=device),
        status=torch.zeros((1,), **i32),
    )


def run_layer_host(x_host, y_host, x, wg, gate_bias, w1, b1, w3, w2, b2, act, k, capacity_factor,
                   bufs: MoELayerBuffers, normalize_gates=True, flags=0, stream=None):
    """Enqueue host-to-device copy of x_host, the whole forward layer and the
    copy of y back to y_host (one C call); the caller synchronises."""
    if normalize_gates:
        flags |= MOE_FLAG_NORMALIZE_GATES
    moe_layer_forward_host(x_host, y_host, x, wg, gate_bias, w1, b1, w3, w2, b2, act, k,
                           capacity_factor, flags, bufs.idx, bufs.gates, bufs.loc, bufs.counts,
                           bufs.c_dev, bufs.buf, bufs.out, bufs.y, bufs.workspace, bufs.status,
                           stream=stream)
    return y_host


def run_layer(x, wg, gate_bias, w1, b1, w3, w2, b2, act, k, capacity_factor, bufs: MoELayerBuffers,
              normalize_gates=True, flags=0, stream=None):
    """Enqueue the whole forward layer; returns bufs.y (no host synchronisation)."""
    if normalize_gates:
        flags |= MOE_FLAG_NORMALIZE_GATES
    moe_layer_forward(x, wg, gate_bias, w1, b1, w3, w2, b2, act, k, capacity_factor, flags,
                      bufs.idx, bufs.gates, bufs.loc, bufs.counts, bufs.c_dev, bufs.buf, bufs.out,
                      bufs.y, bufs.workspace, bufs.status, stream=stream)
    return bufs.y
