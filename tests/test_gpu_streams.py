"""Stream behaviour of the deterministic backward.

The deterministic 16-bit ``fa_bwd`` runs its dQ kernel on a library-owned
side stream and joins it back into the caller's stream before returning.
These tests check that the caller still sees one stream-ordered operation:
work queued after ``fa_bwd`` on the caller's stream observes all three
gradients, and concurrent calls from two host threads on two streams give
the same bits as a lone call.
"""
import threading

import pytest
import torch

import flashattention_backward_fa_gb300 as fa
from flashattention_backward_fa_gb300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

W = WORKLOADS["bf16_causal_b4h16_n2048_d128"].with_(B=2, H=4, N=1024)


def _setup(seed_shift=0):
    q, k, v, do = (t.cuda() for t in make_inputs(W))
    if seed_shift:
        q, do = q.roll(seed_shift, dims=1).contiguous(), do.roll(seed_shift, dims=1).contiguous()
    o, lse = fa.attention_forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    return q, k, v, o, do, lse


def _bwd(args, stream):
    q, k, v, o, do, lse = args
    dq, dk, dv = (torch.empty_like(t) for t in (q, k, v))
    ws = fa.alloc_workspace(q, True)
    fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, causal=True, deterministic=True, stream=stream)
    return dq, dk, dv, ws


def test_work_after_fa_bwd_on_caller_stream_sees_all_gradients():
    args = _setup()
    ref = _bwd(args, None)[:3]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        # Poison the outputs on s, then overwrite them with the backward on s and
        # copy them out on s: the copies must see the join of the side stream.
        dq, dk, dv = (torch.full_like(t, float("nan")) for t in ref)
        ws = fa.alloc_workspace(args[0], True)
        q, k, v, o, do, lse = args
        fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, causal=True, deterministic=True, stream=s)
        copies = [t.clone() for t in (dq, dk, dv)]
    s.synchronize()
    assert fa.fa_get_device_status(clear=True) == 0
    for a, b in zip(ref, copies):
        assert torch.equal(a, b)


def test_two_host_threads_two_streams_bit_identical():
    a1, a2 = _setup(), _setup(seed_shift=7)
    r1, r2 = _bwd(a1, None)[:3], _bwd(a2, None)[:3]
    torch.cuda.synchronize()
    out, errors = {}, []

    def worker(name, args, n):
        try:
            s = torch.cuda.Stream()
            res = []
            for _ in range(n):
                res.append(_bwd(args, s)[:3])
            s.synchronize()
            out[name] = res
        except Exception as e:  # surfaced below
            errors.append(e)

    t1 = threading.Thread(target=worker, args=("a", a1, 6))
    t2 = threading.Thread(target=worker, args=("b", a2, 6))
    t1.start(); t2.start(); t1.join(); t2.join()
    assert not errors, errors
    assert fa.fa_get_device_status(clear=True) == 0
    for res in out["a"]:
        for x, y in zip(r1, res):
            assert torch.equal(x, y)
    for res in out["b"]:
        for x, y in zip(r2, res):
            assert torch.equal(x, y)


def test_calls_from_a_fresh_host_thread():
    """A thread whose first CUDA work is a library call (no context bound to it
    yet) gets the same forward and backward as the main thread: the entry points
    bind the device's context before encoding their tensor maps."""
    q, k, v, o, do, lse = _setup()
    ref = _bwd((q, k, v, o, do, lse), torch.cuda.current_stream())[:3]
    torch.cuda.synchronize()
    out = {}

    def worker():
        try:
            o2 = torch.empty_like(o)
            lse2 = torch.empty_like(lse)
            fa.fa_fwd(q, k, v, o2, lse2, causal=True)
            dq, dk, dv = (torch.empty_like(t) for t in (q, k, v))
            ws = fa.alloc_workspace(q, True)
            fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, causal=True, deterministic=True)
            torch.cuda.synchronize()
            out["r"] = (o2, lse2, dq, dk, dv)
        except Exception as e:  # reported in the main thread
            out["e"] = e

    t = threading.Thread(target=worker)
    t.start()
    t.join()
    assert "e" not in out, out.get("e")
    o2, lse2, dq, dk, dv = out["r"]
    assert torch.equal(o2, o) and torch.equal(lse2, lse)
    for a, b in zip((dq, dk, dv), ref):
        assert torch.equal(a, b)
