"""Guard bands: no kernel writes a byte outside the outputs it declares.

Comparing results with the oracle only sees the elements it reads. A store one
row past a tile, into the padding between rows or heads of a strided layout,
past the end of a packed sequence, or past the end of the workspace, would
pass such a check unseen. Here every tensor is a view into a larger buffer
whose other bytes hold a sentinel:

* before and after each tensor, a guard band of 4096 elements;
* inside it, stride padding: each head row of d elements is followed by 16
  padding elements (h stride d + 16), each sequence position by 8 more (n
  stride H * (d + 16) + 8), each batch entry by 64 more;
* the workspace sits between two 4096-byte guard bands, and the forward's
  L between two 1024-element bands.

For floating-point buffers the sentinel is a NaN pattern, so an input read
that strayed into padding would also show up as a non-finite or wrong
gradient. After each call every byte outside the declared outputs must still
hold the sentinel, and the outputs must match the float64 oracle under the
usual gate. Cases: a ragged tail (N = 333), a sliding window with dropout,
non-causal d = 64, the fp32 path, and packed variable-length sequences, each
in every dQ mode the path has (query-major recompute, atomic, ordered).
"""
import numpy as np
import pytest
import torch

import flashattention_backward_fa_gb300 as fa
import oracle
from flashattention_backward_fa_gb300.inputs import Workload, make_inputs, make_varlen_inputs
from gpu_check import DQ_IDS, DQ_MODES, LSE_ATOL, to_np, within

pytestmark = pytest.mark.gpu

GUARD = 4096
# NaN bit patterns per element size (bf16 / fp16 share 0x7FA5: all-ones
# exponent, nonzero mantissa in both formats).
_SENT = {2: (torch.int16, 0x7FA5), 4: (torch.int32, 0x7FA5A5A5)}
_WS_BYTE = 0xA5


class Guarded:
    """A strided tensor view inside a sentinel-filled buffer."""

    def __init__(self, shape, dtype, pad_h=16, pad_n=8, pad_b=64):
        esz = torch.tensor([], dtype=dtype).element_size()
        self.int_dtype, self.sent = _SENT[esz]
        if len(shape) == 4:
            B, N, H, d = shape
            sh = d + pad_h
            sn = H * sh + pad_n
            sb = N * sn + pad_b
            strides, span = (sb, sn, sh, 1), B * sb
        else:  # packed [total, H, d]
            T, H, d = shape
            sh = d + pad_h
            sn = H * sh + pad_n
            strides, span = (sn, sh, 1), T * sn
        self.raw = torch.full((GUARD + span + GUARD,), self.sent, dtype=self.int_dtype, device="cuda")
        self.view = torch.as_strided(self.raw.view(dtype), shape, strides, GUARD)
        self.mask = torch.zeros(self.raw.shape, dtype=torch.bool, device="cuda")
        torch.as_strided(self.mask, shape, strides, GUARD).fill_(True)

    def fill_from(self, t):
        self.view.copy_(t)
        return self.view

    def untouched_outside(self):
        return bool((self.raw[~self.mask] == self.sent).all())


class GuardedFlat:
    """A contiguous tensor between two guard bands (L, the workspace)."""

    def __init__(self, numel, dtype, guard, sentinel):
        self.raw = torch.full((guard + numel + guard,), sentinel, dtype=dtype, device="cuda")
        self.guard, self.numel, self.sentinel = guard, numel, sentinel
        self.view = self.raw[guard:guard + numel]

    def untouched_outside(self):
        g, n = self.guard, self.numel
        return bool((self.raw[:g] == self.sentinel).all() and (self.raw[g + n:] == self.sentinel).all())


def _run_fixed(w, deterministic):
    q0, k0, v0, do0 = make_inputs(w)
    shape = tuple(q0.shape)
    ins = [Guarded(shape, w.torch_dtype) for _ in range(4)]
    q, k, v, do = (g.fill_from(t.cuda()) for g, t in zip(ins, (q0, k0, v0, do0)))
    go, gq, gk, gv = (Guarded(shape, w.torch_dtype) for _ in range(4))
    lse_g = GuardedFlat(w.B * w.H * w.N, torch.int32, 1024, _SENT[4][1])
    lse = lse_g.view.view(torch.float32).view(w.B, w.H, w.N)
    kw = dict(scale=w.scale, causal=w.causal, window=w.window, dropout_p=w.dropout_p, seed=w.philox_seed,
              offset=w.philox_offset)
    fa.fa_fwd(q, k, v, go.view, lse, **kw)
    nbytes = fa.fa_bwd_workspace_size(w.B, w.H, w.N, w.d, w.torch_dtype, deterministic)
    ws_g = GuardedFlat(nbytes, torch.uint8, GUARD, _WS_BYTE)
    fa.fa_bwd(q, k, v, go.view, do, lse, gq.view, gk.view, gv.view, ws_g.view, **kw, deterministic=deterministic)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(clear=True) == 0
    for name, g in (("q", ins[0]), ("k", ins[1]), ("v", ins[2]), ("do", ins[3]), ("o", go), ("dq", gq),
                    ("dk", gk), ("dv", gv)):
        assert g.untouched_outside(), f"bytes outside {name} changed"
    assert lse_g.untouched_outside(), "bytes outside L changed"
    assert ws_g.untouched_outside(), "bytes outside the workspace changed"
    # the outputs themselves, against the oracle (function mode)
    args = (w.scale, w.causal, w.window, w.dropout_p, w.philox_seed, w.philox_offset)
    o_np, lse_np = to_np(go.view), lse.double().cpu().numpy()
    ro, rl = oracle.forward(to_np(q0), to_np(k0), to_np(v0), *args)
    ok, rep = within(o_np, ro, w.dtype)
    assert ok, ("o", rep)
    assert np.abs(lse_np - rl).max() <= LSE_ATOL
    rq, rk, rv, _ = oracle.backward(to_np(q0), to_np(k0), to_np(v0), o_np, to_np(do0), lse_np, *args)
    floor = float(np.linalg.norm(rv))
    for name, g, r in (("dq", gq, rq), ("dk", gk, rk), ("dv", gv, rv)):
        ok, rep = within(to_np(g.view), r, w.dtype, floor)
        assert ok, (name, rep)


CASES = {
    "bf16_d128_causal_tail333": Workload("canary_tail", 2, 3, 333, 128, "bf16", causal=True, input_seed=71),
    "f16_d64_window96_dropout": Workload("canary_win", 2, 2, 300, 64, "f16", causal=True, window=96,
                                         dropout_p=0.1, philox_seed=99, philox_offset=7, input_seed=72),
    "bf16_d64_noncausal_129": Workload("canary_nc", 1, 3, 129, 64, "bf16", input_seed=73),
    "f32_d64_causal_200": Workload("canary_f32", 1, 2, 200, 64, "f32", causal=True, input_seed=74),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("deterministic", DQ_MODES, ids=DQ_IDS)
def test_guard_bands_fixed_length(case, deterministic):
    w = CASES[case]
    if w.dtype == "f32" and deterministic is not True:
        pytest.skip("fp32 has one dQ path")
    _run_fixed(w, deterministic)


@pytest.mark.parametrize("deterministic", DQ_MODES, ids=DQ_IDS)
@pytest.mark.parametrize("dtype,d,causal,window", [("bf16", 128, True, 0), ("f16", 64, True, 100)])
def test_guard_bands_varlen(dtype, d, causal, window, deterministic):
    lengths = [1, 127, 300, 0, 129, 64]
    H = 2
    q0, k0, v0, do0, cu = make_varlen_inputs(lengths, H, d, dtype, seed=75)
    tdt = q0.dtype
    shape = tuple(q0.shape)
    ins = [Guarded(shape, tdt) for _ in range(4)]
    q, k, v, do = (g.fill_from(t.cuda()) for g, t in zip(ins, (q0, k0, v0, do0)))
    go, gq, gk, gv = (Guarded(shape, tdt) for _ in range(4))
    total = shape[0]
    lse_g = GuardedFlat(H * total, torch.int32, 1024, _SENT[4][1])
    lse = lse_g.view.view(torch.float32).view(H, total)
    cud = cu.cuda()
    msl = max(lengths)
    fa.fa_varlen_fwd(q, k, v, go.view, lse, cud, msl, causal=causal, window=window)
    nbytes = fa.fa_varlen_bwd_workspace_size(len(lengths), msl, total, H, d, tdt, deterministic)
    ws_g = GuardedFlat(nbytes, torch.uint8, GUARD, _WS_BYTE)
    fa.fa_varlen_bwd(q, k, v, go.view, do, lse, gq.view, gk.view, gv.view, cud, msl, ws_g.view, causal=causal,
                     window=window, deterministic=deterministic)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(clear=True) == 0
    for name, g in (("q", ins[0]), ("k", ins[1]), ("v", ins[2]), ("do", ins[3]), ("o", go), ("dq", gq),
                    ("dk", gk), ("dv", gv)):
        assert g.untouched_outside(), f"bytes outside {name} changed"
    assert lse_g.untouched_outside(), "bytes outside L changed"
    assert ws_g.untouched_outside(), "bytes outside the workspace changed"
    scale = fa.default_scale(d)
    qn, kn, vn, don = (to_np(t) for t in (q0, k0, v0, do0))
    o_np, lse_np = to_np(go.view), lse.double().cpu().numpy()
    ro, rl = oracle.varlen_forward(qn, kn, vn, cu.numpy(), scale, causal, window)
    ok, rep = within(o_np, ro, dtype)
    assert ok, ("o", rep)
    live = np.isfinite(rl)
    assert np.abs(lse_np[live] - rl[live]).max() <= LSE_ATOL
    rq, rk, rv = oracle.varlen_backward(qn, kn, vn, o_np, don, lse_np, cu.numpy(), scale, causal, window)
    for name, g, r in (("dq", gq, rq), ("dk", gk, rk), ("dv", gv, rv)):
        ok, rep = within(to_np(g.view), r, dtype)
        assert ok, (name, rep)
