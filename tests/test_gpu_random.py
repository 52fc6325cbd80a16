"""Seeded random configurations against the float64 oracle.

Forty problems drawn from a fixed seed across every option the library takes
at once: dtype, head dimension, ragged N, batch and heads, causal, window,
dropout, ALiBi slopes or an additive bias, and the dQ mode. Each is checked
in function mode (the oracle fed the kernels' O and L) under the dtype's
gate, plus the forward's O and L.
"""
import numpy as np
import pytest
import torch

import flashattention_backward_fa_gb300 as fa
import oracle
from flashattention_backward_fa_gb300.inputs import Workload, make_inputs
from gpu_check import LSE_ATOL, to_np, within

pytestmark = pytest.mark.gpu


def _configs(n=40, seed=2026):
    r = np.random.default_rng(seed)
    out = []
    for t in range(n):
        dtype = r.choice(["bf16", "f16", "f32"], p=[0.45, 0.35, 0.2])
        d = int(r.choice([64, 128])) if dtype != "f32" else int(r.choice([16, 40, 64, 128]))
        N = int(r.integers(1, 700))
        B, H = int(r.integers(1, 4)), int(r.integers(1, 5))
        causal = bool(r.random() < 0.6)
        window = int(r.integers(1, N + 40)) if r.random() < 0.3 else 0
        p = float(r.choice([0.0, 0.0, 0.1, 0.25]))
        extra = str(r.choice(["none", "none", "alibi", "bias"]))
        det = bool(r.random() < 0.6) or dtype == "f32"
        # the accumulating dQ modes alternate: atomic on odd t, ordered on even t
        mode = True if det else (False if t % 2 else fa.FA_DQ_ORDERED)
        out.append((t, dtype, d, N, B, H, causal, window, p, extra, mode))
    return out


@pytest.mark.parametrize("cfg", _configs(), ids=lambda c: f"r{c[0]}-{c[1]}-d{c[2]}-n{c[3]}-{c[9]}")
def test_random_configuration(cfg):
    t, dtype, d, N, B, H, causal, window, p, extra, det = cfg
    w = Workload(f"rand{t}", B, H, N, d, dtype, causal=causal, window=window, dropout_p=p, philox_seed=100 + t,
                 philox_offset=t, input_seed=5000 + t)
    q, k, v, do = make_inputs(w)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    kw = dict(scale=w.scale, causal=causal, window=window, dropout_p=p, seed=w.philox_seed, offset=w.philox_offset)
    alibi = bias = None
    g = torch.Generator().manual_seed(9000 + t)
    if extra == "alibi":
        alibi = (torch.rand((B, H) if t % 2 else (H,), generator=g) * 0.5).float()
        kw["alibi_slopes"] = alibi.cuda()
    elif extra == "bias":
        width = (N + 7) // 8 * 8 if dtype != "f32" else N
        bt = torch.randn((1 if t % 2 else B, H if t % 3 else 1, N, width), generator=g)
        bt = bt.masked_fill(torch.rand(bt.shape, generator=g) < 0.1, float("-inf"))
        bt = bt.to(q.dtype)[..., :N]
        bias = bt
        kw["attn_bias"] = torch.empty_strided(bt.shape, bt.stride(), dtype=bt.dtype, device="cuda").copy_(bt)
    o, lse = fa.attention_forward(qd, kd, vd, **kw)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, dod, lse, **kw, deterministic=det)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(clear=True) == 0
    qn, kn, vn, don = (to_np(x) for x in (q, k, v, do))
    ok_args = dict(alibi=None if alibi is None else alibi.numpy().astype(np.float64),
                   bias=None if bias is None else bias.float().numpy().astype(np.float64))
    args = (w.scale, causal, window, p, w.philox_seed, w.philox_offset)
    ro, rl = oracle.forward(qn, kn, vn, *args, **ok_args)
    good, rep = within(to_np(o), ro, dtype)
    assert good, ("o", rep)
    lg = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(lg))
    if fin.any():
        assert np.abs(lg[fin] - rl[fin]).max() <= LSE_ATOL
    rq, rk, rv, _ = oracle.backward(qn, kn, vn, to_np(o), don, lg, *args, **ok_args)
    floor = float(np.linalg.norm(rv))
    for name, gt, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        gn = to_np(gt)
        assert np.all(np.isfinite(gn)), name
        good, rep = within(gn, r, dtype, norm_floor=floor if name != "dv" else 0.0)
        assert good, (name, rep)
