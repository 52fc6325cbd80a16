"""Packed variable-length forward and backward against the float64 oracle.

Sequences of ragged lengths (1, under one tile, exactly one tile, one past a
tile, several tiles, empty) are packed into [total, H, d] tensors with int32
cu_seqlens; the oracle runs each sequence on its own. Both dQ modes, causal
and windowed masks, d = 64 and 128, both 16-bit dtypes. A pack holding one
sequence must give the same bits as the fixed-length entry points.
"""
import numpy as np
import pytest
import torch

import flashattention_backward_fa_gb300 as fa
import oracle
from flashattention_backward_fa_gb300.inputs import make_varlen_inputs, varlen_lengths
from gpu_check import DQ_IDS, DQ_MODES, LSE_ATOL, to_np, within

pytestmark = pytest.mark.gpu

RAGGED = [1, 127, 128, 129, 300, 64, 513, 0, 257]


def _run(lengths, H, d, dtype, causal, window, deterministic, seed=0, max_seqlen=None):
    q, k, v, do, cu = make_varlen_inputs(lengths, H, d, dtype, seed)
    msl = max(lengths) if max_seqlen is None else max_seqlen
    qd, kd, vd, dod, cud = (t.cuda() for t in (q, k, v, do, cu))
    o, lse = fa.varlen_attention_forward(qd, kd, vd, cud, msl, causal=causal, window=window)
    dq, dk, dv = fa.varlen_attention_backward(qd, kd, vd, o, dod, lse, cud, msl, causal=causal, window=window,
                                              deterministic=deterministic)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(clear=True) == 0
    return (q, k, v, do, cu), (o, lse, dq, dk, dv)


def _check(inputs, outs, dtype, causal, window):
    q, k, v, do = (to_np(t) for t in inputs[:4])
    cu = inputs[4].numpy()
    o, lse, dq, dk, dv = (to_np(t) for t in outs)
    scale = fa.default_scale(q.shape[2])
    ro, rl = oracle.varlen_forward(q, k, v, cu, scale, causal, window)
    ok, rep = within(o, ro, dtype)
    assert ok, ("o", rep)
    live = np.isfinite(rl)
    assert np.array_equal(live, np.isfinite(lse))
    assert np.abs(lse[live] - rl[live]).max() <= LSE_ATOL
    # gradients in function mode: the oracle is fed the O and L the kernels produced
    rq, rk, rv = oracle.varlen_backward(q, k, v, o, do, lse, cu, scale, causal, window)
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        ok, rep = within(g, r, dtype)
        assert ok, (name, rep)


@pytest.mark.parametrize("dtype,d,causal,window", [("bf16", 128, True, 0), ("f16", 64, True, 0),
                                                   ("bf16", 64, False, 0), ("f16", 128, True, 100),
                                                   ("bf16", 128, False, 200)])
@pytest.mark.parametrize("deterministic", DQ_MODES, ids=DQ_IDS)
def test_varlen_ragged(dtype, d, causal, window, deterministic):
    inputs, outs = _run(RAGGED, 3, d, dtype, causal, window, deterministic, seed=d + window)
    _check(inputs, outs, dtype, causal, window)


def test_varlen_many_short_sequences():
    lengths = varlen_lengths(40, 200, seed=5)
    inputs, outs = _run(lengths, 2, 128, "bf16", True, 0, True, seed=6)
    _check(inputs, outs, "bf16", True, 0)


def test_varlen_long_sequence_with_short_neighbours():
    inputs, outs = _run([5, 2048, 3, 700], 2, 128, "bf16", True, 0, False, seed=7)
    _check(inputs, outs, "bf16", True, 0)


def test_varlen_max_seqlen_above_longest():
    # a max_seqlen larger than every length only adds CTAs with no work
    inputs, outs = _run([200, 90, 333], 2, 64, "f16", True, 0, True, seed=8, max_seqlen=1024)
    _check(inputs, outs, "f16", True, 0)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 64)])
def test_varlen_deterministic_bit_identical(dtype, d):
    inputs, a = _run(RAGGED, 2, d, dtype, True, 0, True, seed=9)
    _, b = _run(RAGGED, 2, d, dtype, True, 0, True, seed=9)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0), (True, 64)])
def test_single_sequence_matches_fixed_length_bits(causal, window):
    """One sequence in the pack is the fixed-length problem with B = 1: same kernels, same bits."""
    N, H, d = 777, 2, 128
    (q, k, v, do, cu), (o, lse, dq, dk, dv) = _run([N], H, d, "bf16", causal, window, True, seed=10)
    qd, kd, vd, dod = (t.cuda()[None] for t in (q, k, v, do))
    o2, lse2 = fa.attention_forward(qd, kd, vd, causal=causal, window=window)
    dq2, dk2, dv2 = fa.attention_backward(qd, kd, vd, o2, dod, lse2, causal=causal, window=window,
                                          deterministic=True)
    torch.cuda.synchronize()
    assert torch.equal(o, o2[0]) and torch.equal(lse, lse2[0])
    for x, y in ((dq, dq2), (dk, dk2), (dv, dv2)):
        assert torch.equal(x, y[0])


def test_varlen_rejects_unsupported():
    q = torch.zeros((16, 2, 64), dtype=torch.float32, device="cuda")
    cu = torch.tensor([0, 16], dtype=torch.int32, device="cuda")
    lse = torch.empty((2, 16), dtype=torch.float32, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_varlen_fwd(q, q, q, torch.empty_like(q), lse, cu, 16)
    assert e.value.code == -2
    qh = q.half()
    qh96 = torch.zeros((16, 2, 96), dtype=torch.float16, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_varlen_fwd(qh96, qh96, qh96, torch.empty_like(qh96), lse, cu, 16)
    assert e.value.code == -2
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_varlen_bwd(qh, qh, qh, qh, qh, lse, qh.clone(), qh.clone(), qh.clone(), cu, 16, ws)
    assert e.value.code == -4


def test_varlen_autograd_function():
    lengths = [100, 1, 257, 64]
    H, d = 2, 64
    q, k, v, do, cu = (t.cuda() for t in make_varlen_inputs(lengths, H, d, "f16", seed=41))
    msl = max(lengths)
    qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = fa.flash_attn_varlen_func(qa, ka, va, cu, msl, causal=True)
    out.backward(do)
    o, lse = fa.varlen_attention_forward(q, k, v, cu, msl, causal=True)
    g = fa.varlen_attention_backward(q, k, v, o, do, lse, cu, msl, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(out.detach(), o)
    for a, b in zip((qa.grad, ka.grad, va.grad), g):
        assert torch.equal(a, b)
