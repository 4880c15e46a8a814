"""Dense one-hot formulation of dispatch and combine (test infrastructure only).

This is the formulation the pages start from and then replace:

* "DeepSpeed-MoE vs Tutel" blog, section 3.5: dispatch as
  einsum("TEC,TM->ECM", mask, input), cost O(T*E*Cg*D), mostly multiplications
  by zero; section 1.4 gives the same S*E*M*ce cost for sparse einsum.
* DeepSpeed PR #8195, change 3: the native path built a dense [s, e, c] one-hot
  and ran einsum("sec,sm->ecm"); combine is its transpose with gate weights.

All sums here are in float64 (numpy einsum through BLAS).  Masks are built from
route tables (idx, loc, gates) of shape [k, s]; a route is kept iff loc < c.
"""

import numpy as np


def dispatch_mask(idx, loc, c, e):
    """D[t, j, l] = 1 iff some kept route of token t goes to expert j, slot l."""
    k, s = idx.shape
    D = np.zeros((s, e, c), np.float64)
    for r in range(k):
        for t in range(s):
            if loc[r, t] < c:
                D[t, idx[r, t], loc[r, t]] = 1.0
    return D


def combine_weights(idx, loc, g, c, e):
    """C[t, j, l] = gate of the kept route of token t that landed at (j, l)."""
    k, s = idx.shape
    C = np.zeros((s, e, c), np.float64)
    for r in range(k):
        for t in range(s):
            if loc[r, t] < c:
                C[t, idx[r, t], loc[r, t]] = float(g[r, t])
    return C


def encode(D, x):
    """buf[j, l, :] = sum_t D[t, j, l] * x[t, :]  ('sec,sm->ecm')."""
    return np.einsum("sec,sm->ecm", D, np.asarray(x, np.float64), optimize=True)


def decode(C, out):
    """y[t, :] = sum_{j,l} C[t, j, l] * out[j, l, :]  ('sec,ecm->sm'); out is [e, c, m]."""
    return np.einsum("sec,ecm->sm", C, np.asarray(out, np.float64), optimize=True)


def decode_bwd(C, D, dy, out):
    """Adjoint of decode: d_out = 'sec,sm->ecm'(C, dy); gate gradient per slot
    dC[t, j, l] = D[t, j, l] * <dy[t], out[j, l]>."""
    dy = np.asarray(dy, np.float64)
    d_out = np.einsum("sec,sm->ecm", C, dy, optimize=True)
    dC = D * np.einsum("sm,ecm->sec", dy, np.asarray(out, np.float64), optimize=True)
    return d_out, dC


def encode_bwd(D, d_buf):
    """Adjoint of encode: dx = 'sec,ecm->sm'(D, d_buf)."""
    return np.einsum("sec,ecm->sm", D, np.asarray(d_buf, np.float64), optimize=True)
