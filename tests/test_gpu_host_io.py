"""fa_bwd_host: the backward from host buffers with overlapped copies.

The call cuts the problem into groups (heads when B = 1, batch entries
otherwise), uploads, computes and downloads them on three streams. Every group
runs the same kernels on the same rows as one fa_bwd over the whole problem,
with the dropout masks keyed by the full (batch * H + head) index, so in
deterministic mode the host results must equal fa_bwd's bit for bit.
"""
import numpy as np
import pytest
import torch

import flashattention_backward_fa_gb300 as fa
import oracle
from flashattention_backward_fa_gb300.inputs import Workload, make_inputs
from gpu_check import to_np, within

pytestmark = pytest.mark.gpu


def _device_reference(w, deterministic=True):
    q, k, v, do = (t.cuda() for t in make_inputs(w))
    kw = dict(scale=w.scale, causal=w.causal, window=w.window, dropout_p=w.dropout_p, seed=w.philox_seed,
              offset=w.philox_offset)
    o, lse = fa.attention_forward(q, k, v, **kw)
    g = fa.attention_backward(q, k, v, o, do, lse, **kw, deterministic=deterministic)
    torch.cuda.synchronize()
    return (q, k, v, o, do, lse), g, kw


def _host_run(w, dev_tensors, kw, deterministic=True, pin=True, layout="bnhd"):
    q, k, v, o, do, lse = dev_tensors

    def host(t):
        t = t.cpu()
        if layout == "bhnd":  # [B, H, N, d] storage viewed as [B, N, H, d]
            t = t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
        return t.pin_memory() if pin else t

    hin = [host(t) for t in (q, k, v, o, do)]
    hl = lse.cpu().contiguous()
    hl = hl.pin_memory() if pin else hl
    hout = [torch.full_like(hin[0], float("nan")) for _ in range(3)]
    if pin:
        hout = [t.pin_memory() for t in hout]
    B, N, H, d = q.shape
    nbytes = fa.fa_bwd_host_buffer_size(B, H, N, d, q.dtype, deterministic)
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    fa.fa_bwd_host(*hin, hl, *hout, buf, **kw, deterministic=deterministic, stream=s)
    s.synchronize()
    assert fa.fa_get_device_status(clear=True) == 0
    return hout


CASES = [
    # name, B, H, N, d, dtype, extra
    ("heads_bf16_causal", 1, 6, 700, 128, "bf16", dict(causal=True)),
    ("heads_f16_window_dropout", 1, 5, 333, 64, "f16", dict(causal=True, window=90, dropout_p=0.2, philox_seed=3)),
    ("batch_bf16_dropout", 3, 2, 257, 128, "bf16", dict(dropout_p=0.1, philox_seed=8, philox_offset=5)),
    ("batch_f16_many", 6, 1, 130, 64, "f16", dict(causal=True)),
    ("f32_head_dim_33_unsplit", 1, 3, 97, 33, "f32", dict(causal=True)),  # 33 * 4 B: one group
    ("f32_batch", 2, 2, 64, 64, "f32", dict(dropout_p=0.3, philox_seed=1)),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_host_backward_bit_identical_to_device_call(case):
    name, B, H, N, d, dt, kw = case
    w = Workload(name, B, H, N, d, dt, input_seed=B * 100 + N, **kw)
    dev, ref, kw2 = _device_reference(w)
    out = _host_run(w, dev, kw2)
    for a, b in zip(out, ref):
        assert torch.equal(a, b.cpu())


def test_host_backward_strided_host_layout_and_pageable_memory():
    w = Workload("strided", 1, 4, 300, 64, "bf16", causal=True, input_seed=77)
    dev, ref, kw = _device_reference(w)
    for pin, layout in ((True, "bhnd"), (False, "bnhd"), (False, "bhnd")):
        out = _host_run(w, dev, kw, pin=pin, layout=layout)
        for a, b in zip(out, ref):
            assert torch.equal(a.contiguous(), b.cpu())


def test_host_backward_atomic_mode_against_oracle():
    w = Workload("atomic", 1, 4, 400, 128, "bf16", causal=True, input_seed=78)
    dev, ref, kw = _device_reference(w, deterministic=False)
    out = _host_run(w, dev, kw, deterministic=False)
    q, k, v, o, do, lse = (to_np(t) for t in dev)
    rq, rk, rv, _ = oracle.backward(q, k, v, o, do, lse, w.scale, True)
    for name, g, r in zip(("dq", "dk", "dv"), out, (rq, rk, rv)):
        ok, rep = within(to_np(g), r, "bf16")
        assert ok, (name, rep)
    # dK and dV do not go through atomics: equal to the device call's
    assert torch.equal(out[1], ref[1].cpu()) and torch.equal(out[2], ref[2].cpu())


def test_host_backward_repeated_calls_on_one_stream():
    """Back-to-back calls reuse the staging buffer; each must see its own inputs."""
    w1 = Workload("rep1", 1, 4, 256, 128, "bf16", causal=True, input_seed=1)
    w2 = w1.with_(input_seed=2)
    d1, r1, kw = _device_reference(w1)
    d2, r2, _ = _device_reference(w2)
    B, N, H, d = d1[0].shape
    buf = torch.empty(fa.fa_bwd_host_buffer_size(B, H, N, d, torch.bfloat16, True), dtype=torch.uint8,
                      device="cuda")
    s = torch.cuda.Stream()
    outs = []
    for dev in (d1, d2, d1, d2):
        hin = [t.cpu().pin_memory() for t in dev[:5]]
        hl = dev[5].cpu().pin_memory()
        hout = [torch.empty_like(hin[0]).pin_memory() for _ in range(3)]
        fa.fa_bwd_host(*hin, hl, *hout, buf, **kw, stream=s)
        outs.append((hin, hl, hout))  # keep the host buffers alive until the stream is done
    s.synchronize()
    for (_, _, hout), ref in zip(outs, (r1, r2, r1, r2)):
        for a, b in zip(hout, ref):
            assert torch.equal(a, b.cpu())
