"""Degenerate and boundary cases of the method on the GPU.

* causal with window = 1: each query sees only itself, so P = 1 on the
  diagonal, O = V, dV = dO, and dS = P (dP - D) = dO.V - dO.O = 0: dQ and dK
  vanish (up to the rounding of D against dP). Without the causal mask the
  window is one-sided (keys j >= i), checked against the oracle.
* a window at least as long as the sequence is no window;
* dO = 0 gives exactly zero gradients;
* scores far beyond exp's range (Q, K scaled up) stay finite and match the oracle;
* lengths on and next to the 128-row tile boundaries, and many small units.
"""
import numpy as np
import pytest
import torch

import flashattention_backward_fa_gb300 as fa
from flashattention_backward_fa_gb300.inputs import Workload, make_inputs
from gpu_check import DQ_IDS, DQ_MODES, check_against_oracle, run_gpu, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 64), ("f32", 64)])
def test_window_one_is_identity_attention(dtype, d):
    w = Workload("w1", 2, 2, 300, d, dtype, causal=True, window=1, input_seed=41)
    res = run_gpu(w)
    o, v = to_np(res["o"]), to_np(res["v"])
    dv, do = to_np(res["dv"]), to_np(res["do"])
    if dtype == "f32":
        # P = 1 up to the rounding of L
        np.testing.assert_allclose(o, v, rtol=1e-6, atol=1e-7)
        np.testing.assert_allclose(dv, do, rtol=1e-6, atol=1e-7)
    else:
        # P rounds to exactly 1 in 16 bits: O = V and dV = dO bit for bit
        np.testing.assert_array_equal(o, v)
        np.testing.assert_array_equal(dv, do)
    for name in ("dq", "dk"):
        g = np.abs(to_np(res[name]))
        assert g.max() <= 1e-3, (name, g.max())       # rounding of D against dP only
    fails, _ = check_against_oracle(w, res, exact=False)
    assert not fails, fails


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 64), ("f32", 64)])
def test_one_sided_window_one_without_causal(dtype, d):
    w = Workload("w1nc", 1, 2, 260, d, dtype, causal=False, window=1, input_seed=46)
    res = run_gpu(w)
    fails, _ = check_against_oracle(w, res, exact=False)
    assert not fails, fails


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 64)])
def test_window_longer_than_sequence_is_no_window(dtype, d):
    w = Workload("wlong", 1, 2, 260, d, dtype, causal=True, window=10000, input_seed=42)
    res = run_gpu(w)
    ref = run_gpu(w.with_(window=0))
    for name in ("o", "lse", "dq", "dk", "dv"):
        a, b = res[name].float(), ref[name].float()
        assert torch.allclose(a, b, rtol=0, atol=0) or torch.allclose(a, b, rtol=1e-2, atol=1e-3), name
    fails, _ = check_against_oracle(w, res, exact=False)
    assert not fails, fails


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 64), ("f32", 64)])
@pytest.mark.parametrize("deterministic", DQ_MODES, ids=DQ_IDS)
def test_zero_upstream_gradient_gives_zero_gradients(dtype, d, deterministic):
    if dtype == "f32" and not deterministic:
        pytest.skip("fp32 has one dQ path")
    w = Workload("dozero", 1, 2, 200, d, dtype, causal=True, input_seed=43)
    q, k, v, _ = (t.cuda() for t in make_inputs(w))
    do = torch.zeros_like(q)
    o, lse = fa.attention_forward(q, k, v, causal=True)
    dq, dk, dv = fa.attention_backward(q, k, v, o, do, lse, causal=True, deterministic=deterministic)
    torch.cuda.synchronize()
    for g in (dq, dk, dv):
        assert torch.count_nonzero(g).item() == 0


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 64)])
def test_large_scores_stay_finite(dtype, d):
    """Q and K scaled so that |S| reaches thousands of nats: the row maximum and
    L keep every exponent in range."""
    w = Workload("big", 1, 2, 333, d, dtype, causal=True, input_seed=44)
    q, k, v, do = make_inputs(w)
    big = 30.0 if dtype == "bf16" else 12.0        # fp16 tops out at 65504
    q = (q.float() * big).to(q.dtype)
    k = (k.float() * big).to(k.dtype)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=True)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, dod, lse, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(clear=True) == 0
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    res = dict(q=q, k=k, v=v, do=do, o=o.cpu(), lse=lse.cpu(), dq=dq.cpu(), dk=dk.cpu(), dv=dv.cpu())
    fails, _ = check_against_oracle(w, res, exact=False)
    assert not fails, fails


@pytest.mark.parametrize("N", [127, 128, 129, 255, 256, 257, 511])
def test_tile_boundaries(N):
    w = Workload(f"tb{N}", 1, 2, N, 128, "bf16", causal=True, input_seed=N)
    for det in DQ_MODES:
        res = run_gpu(w, deterministic=det)
        fails, _ = check_against_oracle(w, res, exact=False)
        assert not fails, (det, fails)


def test_many_small_units():
    """B * H = 256 units of 96 rows: one partial tile each, groups of units in the grid."""
    w = Workload("many", 16, 16, 96, 64, "f16", causal=True, input_seed=45)
    res = run_gpu(w)
    fails, _ = check_against_oracle(w, res, exact=False)
    assert not fails, fails
