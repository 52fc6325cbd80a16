"""ALiBi position bias on the GPU against the float64 oracle.

The score of (i, j) gains -m_h |i - j| after the scale. The slopes follow the
usual geometric ladder m_h = 2^(-8 (h + 1) / H), either shared over the batch
([H]) or per batch entry ([B, H]). Every dtype path runs: the tcgen05 kernels
(bf16, fp16; d = 64, 128; causal, window, none; with and without dropout; both
dQ modes), the fp32 CUDA-core kernels, and packed sequences.
"""
import numpy as np
import pytest
import torch

import flashattention_backward_fa_gb300 as fa
import oracle
from flashattention_backward_fa_gb300.inputs import Workload, make_inputs, make_varlen_inputs
from gpu_check import DQ_IDS, DQ_MODES, LSE_ATOL, to_np, within

pytestmark = pytest.mark.gpu


def ladder(H, B=None, shift=0.0):
    m = 2.0 ** (-8.0 * (np.arange(H) + 1) / H)
    if B is not None:
        m = np.stack([m * (1.0 + shift * b) for b in range(B)])
    return torch.tensor(m, dtype=torch.float32)


CASES = [
    # dtype, d, N, causal, window, dropout, per-batch slopes
    ("bf16", 128, 333, True, 0, 0.0, False),
    ("f16", 64, 257, False, 0, 0.0, True),
    ("bf16", 64, 300, True, 70, 0.0, True),
    ("f16", 128, 200, True, 0, 0.15, False),
    ("bf16", 128, 190, False, 50, 0.1, True),
    ("f32", 64, 150, True, 0, 0.0, True),
    ("f32", 128, 97, False, 0, 0.2, False),
]


def _run(w, slopes, deterministic):
    q, k, v, do = make_inputs(w)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    sd = slopes.cuda()
    kw = dict(scale=w.scale, causal=w.causal, window=w.window, dropout_p=w.dropout_p, seed=w.philox_seed,
              offset=w.philox_offset, alibi_slopes=sd)
    o, lse = fa.attention_forward(qd, kd, vd, **kw)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, dod, lse, **kw, deterministic=deterministic)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(clear=True) == 0
    return (q, k, v, do), (o, lse, dq, dk, dv)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
@pytest.mark.parametrize("deterministic", DQ_MODES, ids=DQ_IDS)
def test_alibi_against_oracle(case, deterministic):
    dtype, d, N, causal, window, p, per_batch = case
    if dtype == "f32" and not deterministic:
        pytest.skip("fp32 has one dQ path")
    B, H = 2, 3
    w = Workload("alibi", B, H, N, d, dtype, causal=causal, window=window, dropout_p=p, philox_seed=9,
                 philox_offset=4, input_seed=N + d)
    slopes = ladder(H, B if per_batch else None, shift=0.5)
    inputs, (o, lse, dq, dk, dv) = _run(w, slopes, deterministic)
    q, k, v, do = (to_np(t) for t in inputs)
    sl = slopes.numpy().astype(np.float64)
    args = (w.scale, causal, window, p, w.philox_seed, w.philox_offset)
    ro, rl = oracle.forward(q, k, v, *args, alibi=sl)
    ok, rep = within(to_np(o), ro, dtype)
    assert ok, ("o", rep)
    lg = lse.cpu().numpy().astype(np.float64)
    assert np.abs(lg - rl).max() <= LSE_ATOL
    rq, rk, rv, _ = oracle.backward(q, k, v, to_np(o), do, lg, *args, alibi=sl)
    floor = float(np.linalg.norm(rv))
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        ok, rep = within(to_np(g), r, dtype, norm_floor=floor if name != "dv" else 0.0)
        assert ok, (name, rep)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 64)])
def test_alibi_long_sequence_steep_slopes(dtype, d):
    """N = 2048 with slopes up to 0.5: most of each row's mass sits near the
    diagonal, and far keys underflow to zero probability."""
    B, H, N = 1, 4, 2048
    w = Workload("alibi_long", B, H, N, d, dtype, causal=True, input_seed=21)
    slopes = ladder(H)
    inputs, (o, lse, dq, dk, dv) = _run(w, slopes, True)
    q, k, v, do = (to_np(t) for t in inputs)
    sl = slopes.numpy().astype(np.float64)
    lg = lse.cpu().numpy().astype(np.float64)
    ro, rl = oracle.forward(q, k, v, w.scale, True, alibi=sl)
    assert within(to_np(o), ro, dtype)[0]
    assert np.abs(lg - rl).max() <= LSE_ATOL
    rq, rk, rv, _ = oracle.backward(q, k, v, to_np(o), do, lg, w.scale, True, alibi=sl)
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        ok, rep = within(to_np(g), r, dtype)
        assert ok, (name, rep)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 64), ("f32", 64)])
def test_alibi_zero_slopes_bit_identical_to_plain(dtype, d):
    """Zero slopes add exact zeros to every score, so the backward kernels (and the
    fp32 forward) reproduce the plain ones bit for bit. The 16-bit ALiBi forward
    visits key blocks outward from the diagonal instead of in ascending order, so
    its O and L agree with the plain forward up to summation order."""
    w = Workload("alibi0", 2, 2, 321, d, dtype, causal=True, input_seed=3)
    q, k, v, do = (t.cuda() for t in make_inputs(w))
    z = torch.zeros(2, dtype=torch.float32, device="cuda")
    o1, l1 = fa.attention_forward(q, k, v, causal=True)
    o2, l2 = fa.attention_forward(q, k, v, causal=True, alibi_slopes=z)
    g1 = fa.attention_backward(q, k, v, o1, do, l1, causal=True)
    g2 = fa.attention_backward(q, k, v, o1, do, l1, causal=True, alibi_slopes=z)
    torch.cuda.synchronize()
    if dtype == "f32":
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    else:
        assert torch.allclose(o1.float(), o2.float(), rtol=8e-3, atol=1e-3)
        assert torch.allclose(l1, l2, rtol=0, atol=1e-5)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_alibi_deterministic_bit_identical():
    w = Workload("alibi_det", 2, 4, 777, 128, "bf16", causal=True, input_seed=4)
    slopes = ladder(4, 2, 0.25)
    a = _run(w, slopes, True)[1]
    b = _run(w, slopes, True)[1]
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("per_seq", [False, True])
def test_alibi_varlen(per_seq):
    lengths = [129, 1, 300, 64, 0, 255]
    H, d = 3, 128
    q, k, v, do, cu = make_varlen_inputs(lengths, H, d, "bf16", seed=31)
    slopes = ladder(H, len(lengths) if per_seq else None, shift=0.3)
    qd, kd, vd, dod, cud, sd = (t.cuda() for t in (q, k, v, do, cu, slopes))
    msl = max(lengths)
    o, lse = fa.varlen_attention_forward(qd, kd, vd, cud, msl, causal=True, alibi_slopes=sd)
    dq, dk, dv = fa.varlen_attention_backward(qd, kd, vd, o, dod, lse, cud, msl, causal=True, alibi_slopes=sd)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(clear=True) == 0
    qn, kn, vn, don = (to_np(t) for t in (q, k, v, do))
    sl = slopes.numpy().astype(np.float64)
    scale = fa.default_scale(d)
    ro, rl = oracle.varlen_forward(qn, kn, vn, cu.numpy(), scale, True, alibi=sl)
    assert within(to_np(o), ro, "bf16")[0]
    rq, rk, rv = oracle.varlen_backward(qn, kn, vn, to_np(o), don, lse.cpu().numpy(), cu.numpy(), scale, True,
                                        alibi=sl)
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        ok, rep = within(to_np(g), r, "bf16")
        assert ok, (name, rep)


def test_alibi_autograd_function():
    w = Workload("alibi_ag", 1, 2, 130, 64, "bf16", causal=True, input_seed=5)
    q, k, v, do = (t.cuda() for t in make_inputs(w))
    slopes = ladder(2).cuda()
    qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = fa.flash_attn_func(qa, ka, va, causal=True, alibi_slopes=slopes)
    out.backward(do)
    o, lse = fa.attention_forward(q, k, v, causal=True, alibi_slopes=slopes)
    g = fa.attention_backward(q, k, v, o, do, lse, causal=True, alibi_slopes=slopes)
    torch.cuda.synchronize()
    assert torch.equal(out.detach(), o)
    for a, b in zip((qa.grad, ka.grad, va.grad), g):
        assert torch.equal(a, b)
