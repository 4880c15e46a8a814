"""FP8 (e4m3) experts on the GPU against the oracle, step by step: the row
quantiser bit for bit; fc1 (hidden) within the fp32-accumulation and bf16
rounding bound; the hidden's quantisation bit for bit (on the kernel's own
hidden); fc2 within the same bound (on the kernel's own codes)."""

import numpy as np
import pytest
import torch

import combine_moe_gate_gb300 as M
import oracle
import synth

from gpu_util import status_ok

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def _bf16(shape, seed, name, scale=1.0):
    bits = synth.normal_host(seed, name, shape, scale, "bf16")
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def _q(x, counts=None, c_dev=None):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = torch.full(x.shape, 0xAA, dtype=torch.uint8, device="cuda")
    sc = torch.full(x.shape[:-1], -1.0, dtype=torch.float32, device="cuda")
    M.moe_quantize_rows_fp8(x, q, sc, st, counts=counts, c_dev=c_dev)
    torch.cuda.synchronize()
    status_ok(st)
    return q, sc


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


# row widths for each register layout of the kernel (one, two, four or eight
# warps per row; a chunk count just past a layout's capacity) and the loop
# form beyond 16384 columns
@pytest.mark.parametrize("rows,cols", [(1, 16), (37, 80), (600, 4096), (5, 2064), (9, 8192),
                                       (3, 16384), (2, 16400)])
def test_quantize_rows_fp8_is_bit_exact(rows, cols):
    x = _bf16((rows, cols), 21, f"q{rows}", 3.0)
    x[0] = 0                                   # an all-zero row: scale 1
    if rows > 2:
        x[2, 5] = -1000.0                          # a row whose amax is negative
        x[1] *= 1e-30                              # tiny values (e4m3 subnormals after scaling)
    q, sc = _q(x)
    qo, so = oracle.quantize_rows_fp8(_bits(x))
    assert np.array_equal(sc.cpu().numpy(), so)
    assert np.array_equal(q.cpu().numpy(), qo)


@pytest.mark.parametrize("m", [64, 4096])
def test_quantize_rows_fp8_writes_kept_rows_only(m):
    e, c_max = 3, 50
    x = _bf16((e, c_max, m), 22, f"qk{m}")
    counts = torch.tensor([50, 0, 17], dtype=torch.int32, device="cuda")
    c_dev = torch.tensor([40], dtype=torch.int32, device="cuda")
    q, sc = _q(x, counts, c_dev)
    qo, so = oracle.quantize_rows_fp8(_bits(x).reshape(e * c_max, m))
    qo, so = qo.reshape(e, c_max, m), so.reshape(e, c_max)
    qn, sn = q.cpu().numpy(), sc.cpu().numpy()
    for j, kept in enumerate([40, 0, 17]):
        assert np.array_equal(qn[j, :kept], qo[j, :kept]) and np.array_equal(sn[j, :kept], so[j, :kept])
        assert np.all(qn[j, kept:] == 0xAA) and np.all(sn[j, kept:] == -1.0)


def _tol(qa, sa, qw, sw, want):
    """|err| bound: one bf16 rounding of the result (2^-8 relative, with margin
    2^-7) plus fp32 accumulation over K terms of the scaled products."""
    dec = np.array([oracle.fp8_decode(c) if (c & 0x7F) != 0x7F else 0.0 for c in range(256)])
    mag = np.abs(dec[qa]) @ np.abs(dec[qw]).T * np.abs(sa)[:, None] * np.abs(sw)[None, :]
    K = qa.shape[1]
    return 2.0 ** -7 * np.abs(want) + 2 * K * U * mag + 1e-30


CASES = [
    # e, c_max, m, h, act, kept rows per expert, c
    (3, 300, 256, 384, "gelu", [300, 0, 129], 300),
    (2, 260, 128, 256, "relu", [7, 260], 200),
    (4, 512, 2048, 1024, "gelu", [512, 300, 1, 256], 512),   # 16 K blocks in fc1
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"e{c[0]}_m{c[2]}_h{c[3]}_{c[4]}")
def test_expert_ffn_fp8_matches_oracle(case):
    e, c_max, m, h, act, kept, c = case
    dev = "cuda"
    buf = _bf16((e, c_max, m), 31, f"b{m}", 1.0)
    w1 = _bf16((e, h, m), 32, f"w1{m}", m ** -0.5)
    w2 = _bf16((e, m, h), 33, f"w2{h}", h ** -0.5)
    b1 = _bf16((e, h), 34, f"b1{h}", 0.1)
    b2 = _bf16((e, m), 35, f"b2{m}", 0.1)
    counts = torch.tensor(kept, dtype=torch.int32, device=dev)
    c_dev = torch.tensor([c], dtype=torch.int32, device=dev)
    eff = [min(k_, c) for k_ in kept]
    bq, bs = _q(buf, counts, c_dev)
    w1q, w1s = _q(w1)
    w2q, w2s = _q(w2)
    ws = torch.zeros(M.moe_expert_ffn_fp8_workspace_size(e, c_max, m, h), dtype=torch.uint8, device=dev)
    out = torch.full((e, c_max, m), float("nan"), dtype=torch.bfloat16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    M.moe_expert_ffn_fp8(bq, bs, counts, c_dev, w1q, w1s, b1, w2q, w2s, b2, act, ws, out, st)
    torch.cuda.synchronize()
    status_ok(st)
    rows = e * c_max
    up = lambda n: (n + 255) // 256 * 256
    hid = ws[: rows * h * 2].view(torch.bfloat16).view(e, c_max, h)
    hq = ws[up(rows * h * 2): up(rows * h * 2) + rows * h].view(e, c_max, h)
    hs = ws[up(rows * h * 2) + up(rows * h): up(rows * h * 2) + up(rows * h) + rows * 4].view(torch.float32).view(e, c_max)
    to = lambda t: t.cpu().numpy()
    for j in range(e):
        r = eff[j]
        if r == 0:
            continue
        qa, sa = to(bq[j, :r]), to(bs[j, :r])
        # fc1
        want = oracle.fc_fp8(qa, sa, to(w1q[j]), to(w1s[j]), _bits(b1[j]), act)
        got = oracle.to_f32(_bits(hid[j, :r]))
        assert np.all(np.abs(got - want) <= _tol(qa, sa, to(w1q[j]), to(w1s[j]), want)), j
        # the hidden's quantisation, on the kernel's own hidden
        qh, sh = oracle.quantize_rows_fp8(_bits(hid[j, :r]))
        assert np.array_equal(to(hq[j, :r]), qh) and np.array_equal(to(hs[j, :r]), sh), j
        # fc2 on the kernel's codes
        want2 = oracle.fc_fp8(qh, sh, to(w2q[j]), to(w2s[j]), _bits(b2[j]), None)
        got2 = oracle.to_f32(_bits(out[j, :r]))
        assert np.all(np.abs(got2 - want2) <= _tol(qh, sh, to(w2q[j]), to(w2s[j]), want2)), j
