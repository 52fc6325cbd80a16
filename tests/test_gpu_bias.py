"""Additive attention bias on the GPU against the float64 oracle.

The score of (i, j) gains bias[b, h, i, j] after the scale; -inf entries mask
pairs out. Covered: every dtype path, d = 64 and 128, causal / window / none,
dropout, both dQ modes, broadcast shapes ([1, H], [B, 1], [B, H] planes),
padded row strides, a ragged N (bias tiles and rows past N), a row with every
key masked, and a bias equal to ALiBi's against the ALiBi path.
"""
import numpy as np
import pytest
import torch

import flashattention_backward_fa_gb300 as fa
import oracle
from flashattention_backward_fa_gb300.inputs import Workload, make_inputs
from gpu_check import DQ_IDS, DQ_MODES, LSE_ATOL, to_np, within

pytestmark = pytest.mark.gpu


def make_bias(B, H, N, dtype, seed, neg_inf_frac=0.15, row_pad=0, dead_row=None):
    """Seeded bias [B, H, N, N] (size-1 dims broadcast) of the workload dtype;
    -inf entries off the diagonal. 16-bit rows are padded to a multiple of 8
    elements (the library's alignment rule), plus row_pad more."""
    g = torch.Generator().manual_seed(seed)
    width = (N + 7) // 8 * 8 + row_pad if dtype != "f32" else N + row_pad
    b = torch.randn((B, H, N, width), generator=g) * 2.0
    if neg_inf_frac:
        m = torch.rand((B, H, N, width), generator=g) < neg_inf_frac
        idx = torch.arange(N)
        m[:, :, idx, idx] = False
        b = b.masked_fill(m, float("-inf"))
    if dead_row is not None:
        b[:, :, dead_row, :] = float("-inf")
    b = b.to({"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[dtype])
    return b[..., :N]  # a view with the padded row stride


def to_device(bias):
    """The bias on the GPU with its (padded) strides kept."""
    return torch.empty_strided(bias.shape, bias.stride(), dtype=bias.dtype, device="cuda").copy_(bias)


def _run(w, bias, deterministic):
    q, k, v, do = make_inputs(w)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    bd = to_device(bias)
    kw = dict(scale=w.scale, causal=w.causal, window=w.window, dropout_p=w.dropout_p, seed=w.philox_seed,
              offset=w.philox_offset, attn_bias=bd)
    o, lse = fa.attention_forward(qd, kd, vd, **kw)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, dod, lse, **kw, deterministic=deterministic)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(clear=True) == 0
    return (q, k, v, do), (o, lse, dq, dk, dv)


def _check(w, bias, inputs, outs):
    q, k, v, do = (to_np(t) for t in inputs)
    o, lse, dq, dk, dv = outs
    bn = bias.float().numpy().astype(np.float64)
    args = (w.scale, w.causal, w.window, w.dropout_p, w.philox_seed, w.philox_offset)
    ro, rl = oracle.forward(q, k, v, *args, bias=bn)
    ok, rep = within(to_np(o), ro, w.dtype)
    assert ok, ("o", rep)
    lg = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(lg)) and np.all(lg[~fin] == -np.inf)
    assert np.abs(lg[fin] - rl[fin]).max() <= LSE_ATOL
    rq, rk, rv, _ = oracle.backward(q, k, v, to_np(o), do, lg, *args, bias=bn)
    floor = float(np.linalg.norm(rv))
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        gn = to_np(g)
        assert np.all(np.isfinite(gn)), name
        ok, rep = within(gn, r, w.dtype, norm_floor=floor if name != "dv" else 0.0)
        assert ok, (name, rep)


CASES = [
    # dtype, d, N, causal, window, dropout, bias batch, bias heads, row pad
    ("bf16", 128, 300, True, 0, 0.0, 1, 3, 0),
    ("f16", 64, 257, False, 0, 0.0, 2, 1, 8),  # 16-bit pads: multiples of 8
    ("bf16", 64, 200, True, 60, 0.1, 2, 3, 0),
    ("f16", 128, 129, False, 40, 0.0, 1, 1, 16),
    ("bf16", 128, 64, True, 0, 0.2, 2, 3, 0),
    ("f32", 64, 150, True, 0, 0.0, 2, 3, 1),
    ("f32", 40, 97, False, 0, 0.1, 1, 3, 0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
@pytest.mark.parametrize("deterministic", DQ_MODES, ids=DQ_IDS)
def test_bias_against_oracle(case, deterministic):
    dtype, d, N, causal, window, p, bb, bh, pad = case
    if dtype == "f32" and not deterministic:
        pytest.skip("fp32 has one dQ path")
    B, H = 2, 3
    w = Workload("bias", B, H, N, d, dtype, causal=causal, window=window, dropout_p=p, philox_seed=6,
                 philox_offset=2, input_seed=N + d + bb)
    bias = make_bias(bb, bh, N, dtype, seed=N * 7 + d, row_pad=pad)
    inputs, outs = _run(w, bias, deterministic)
    _check(w, bias, inputs, outs)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 64), ("f32", 64)])
def test_bias_dead_row(dtype, d):
    """A query row with every key masked: O = 0, L = -inf, zero dQ, no NaN anywhere."""
    w = Workload("dead", 1, 2, 200, d, dtype, causal=True, input_seed=9)
    bias = make_bias(1, 1, 200, dtype, seed=10, neg_inf_frac=0.0, dead_row=77)
    inputs, outs = _run(w, bias, True)
    o, lse, dq = outs[0], outs[1], outs[2]
    assert torch.count_nonzero(o[0, 77]).item() == 0
    assert torch.all(lse[0, :, 77] == float("-inf"))
    assert torch.count_nonzero(dq[0, 77]).item() == 0
    _check(w, bias, inputs, outs)


def test_bias_long_sequence_large_values():
    """N = 2048 causal with a [1, H] bias of large magnitude (|bias| up to ~20)."""
    w = Workload("bias_long", 1, 2, 2048, 128, "bf16", causal=True, input_seed=12)
    bias = make_bias(1, 2, 2048, "bf16", seed=13, neg_inf_frac=0.05)
    bias = (bias.float() * 4).to(torch.bfloat16)
    inputs, outs = _run(w, bias, True)
    _check(w, bias, inputs, outs)


def test_bias_equal_to_alibi_matches_alibi_path():
    N, H = 333, 4
    w = Workload("bias_alibi", 1, H, N, 128, "bf16", causal=True, input_seed=14)
    slopes = 2.0 ** (-8.0 * (torch.arange(H) + 1) / H)
    pos = torch.arange(N, dtype=torch.float64)
    ab = (-slopes.double()[:, None, None] * (pos[:, None] - pos[None, :]).abs())[None]
    q, k, v, do = (t.cuda() for t in make_inputs(w))
    # the bias path sees ALiBi rounded to bf16 (rows padded to 336); the oracle takes the same rounded bias
    padded = torch.zeros((1, H, N, 336), dtype=torch.bfloat16)
    padded[..., :N] = ab.to(torch.bfloat16)
    bias = padded.cuda()[..., :N]
    o1, l1 = fa.attention_forward(q, k, v, causal=True, attn_bias=bias)
    g1 = fa.attention_backward(q, k, v, o1, do, l1, causal=True, attn_bias=bias)
    o2, l2 = fa.attention_forward(q, k, v, causal=True, alibi_slopes=slopes.float().cuda())
    torch.cuda.synchronize()
    # both against the oracle of their own bias
    _check(w, bias.cpu(), [t.cpu() for t in (q, k, v, do)], (o1, l1) + tuple(g1))
    assert (l1 - l2).abs().max().item() < 0.05  # bf16 rounding of the ALiBi bias only


def test_bias_autograd_function():
    w = Workload("bias_ag", 2, 2, 140, 64, "f16", causal=True, input_seed=15)
    q, k, v, do = (t.cuda() for t in make_inputs(w))
    bias = to_device(make_bias(2, 1, 140, "f16", seed=16))
    qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = fa.flash_attn_func(qa, ka, va, causal=True, attn_bias=bias)
    out.backward(do)
    o, lse = fa.attention_forward(q, k, v, causal=True, attn_bias=bias)
    g = fa.attention_backward(q, k, v, o, do, lse, causal=True, attn_bias=bias)
    torch.cuda.synchronize()
    assert torch.equal(out.detach(), o)
    for a, b in zip((qa.grad, ka.grad, va.grad), g):
        assert torch.equal(a, b)
