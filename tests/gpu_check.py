"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and compare against the float64 oracle with the gate's tolerances.

Tolerances (fixed by the library's acceptance gate):
  * fp32: relative L2 error <= 1e-5 per tensor;
  * fp16 / bf16: elementwise |g - r| <= 5e-3 + 5e-3 * |r|.
The forward's L is held to max |err| <= 1e-4 (it is fp32 arithmetic either way).
"""
from __future__ import annotations

import numpy as np
import torch

import flashattention_backward_fa_gb300 as fa
import oracle
from flashattention_backward_fa_gb300.inputs import Workload, make_inputs

ATOL = RTOL = 5e-3
F32_REL_L2 = 1e-5
LSE_ATOL = 1e-4
EXACT_REL_L2 = 1e-2  # composed forward -> backward, 16-bit dtypes (secondary bar)

# The dQ algorithms every parity test runs: the deterministic default (query-major
# recompute), atomic accumulation, and the ordered (deterministic) accumulation.
DQ_MODES = [True, False, fa.FA_DQ_ORDERED]
DQ_IDS = ["det", "atomic", "ordered"]


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def within(g: np.ndarray, r: np.ndarray, dtype: str, norm_floor: float = 0.0):
    """(ok, report) under the gate's tolerance for ``dtype``.

    For fp32 the relative L2 error is taken against max(||r||, norm_floor):
    dQ and dK pass the norm of dV of the same problem as the floor, which only
    matters where the exact dQ / dK vanish (a single key, identical keys) and
    a plain relative error would divide rounding noise by zero.
    """
    err = np.abs(g - r)
    rel_l2 = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), norm_floor, 1e-300))
    rep = {"max_abs": float(err.max()) if err.size else 0.0, "rel_l2": rel_l2}
    if dtype == "f32":
        return rel_l2 <= F32_REL_L2, rep
    bad = err > ATOL + RTOL * np.abs(r)
    rep["violations"] = int(bad.sum())
    return not bad.any(), rep


def run_gpu(w: Workload, deterministic=True, layout="bnhd", device="cuda"):
    """Inputs on the GPU, fa_fwd then fa_bwd; returns dict of CPU tensors and the inputs."""
    q, k, v, do = make_inputs(w)

    def place(t):
        t = t.to(device)
        if layout == "bhnd":  # [B, H, N, d] storage viewed as [B, N, H, d]
            t = t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
        return t

    qd, kd, vd, dod = (place(t) for t in (q, k, v, do))
    kw = dict(scale=w.scale, causal=w.causal, window=w.window, dropout_p=w.dropout_p, seed=w.philox_seed,
              offset=w.philox_offset)
    o = torch.empty_like(qd)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=device)
    fa.fa_fwd(qd, kd, vd, o, lse, **kw)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = fa.alloc_workspace(qd, deterministic)
    fa.fa_bwd(qd, kd, vd, o, dod, lse, dq, dk, dv, ws, **kw, deterministic=deterministic)
    torch.cuda.synchronize()
    status = fa.fa_get_device_status(clear=True)
    assert status == 0, f"device status {status}"
    return dict(q=q, k=k, v=v, do=do, o=o.cpu(), lse=lse.cpu(), dq=dq.cpu(), dk=dk.cpu(), dv=dv.cpu())


def check_against_oracle(w: Workload, res, exact=True):
    """Compare GPU results with the oracle in function mode (and exact mode)."""
    q, k, v, do = (to_np(res[n]) for n in ("q", "k", "v", "do"))
    o_g, lse_g = to_np(res["o"]), res["lse"].numpy().astype(np.float64)
    args = (w.scale, w.causal, w.window, w.dropout_p, w.philox_seed, w.philox_offset)
    report = {}
    failures = []
    rq, rk, rv, _ = oracle.backward(q, k, v, o_g, do, lse_g, *args)
    floor = float(np.linalg.norm(rv))
    for name, r in (("dq", rq), ("dk", rk), ("dv", rv)):
        ok, rep = within(to_np(res[name]), r, w.dtype, floor)
        report[f"fn_{name}"] = rep
        if not ok:
            failures.append(f"function-mode {name}: {rep}")
    if exact:
        O, L, eq, ek, ev, _ = oracle.reference_grads(q, k, v, do, *args)
        ok, rep = within(o_g, O, w.dtype)
        report["o"] = rep
        if not ok:
            failures.append(f"forward O: {rep}")
        lerr = float(np.abs(lse_g - L).max())
        report["lse_max_abs"] = lerr
        if not lerr <= LSE_ATOL:
            failures.append(f"forward L max abs {lerr}")
        # Composed forward -> backward. For 16-bit dtypes the forward's O is
        # rounded to 16 bits, which moves D_i = sum_k dO_ik O_ik by up to
        # sum_k |dO_ik| 2^-9 |O_ik|; no backward can undo that, so the composed
        # result is held to relative L2 <= 1e-2 and the elementwise gate applies
        # to the backward as a function of its inputs (above).
        floor = float(np.linalg.norm(ev))
        for name, r in (("dq", eq), ("dk", ek), ("dv", ev)):
            ok, rep = within(to_np(res[name]), r, w.dtype, floor)
            report[f"exact_{name}"] = rep
            if w.dtype != "f32":
                ok = rep["rel_l2"] <= EXACT_REL_L2
            if not ok:
                failures.append(f"exact-mode {name}: {rep}")
    return failures, report
