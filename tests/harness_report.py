"""Writes harness_report.json: the correctness report of "Lecture 7 — Backward
Pass and Validation" (sections "Build it", "Measure it", "Ship it") for this
library.

Rows: the page's shape sweep, (B, H, N, D) in {(1, 8, 512, 64), (2, 16, 2048,
128), (1, 4, 8192, 64)} x {fp16, bf16} x {causal, not}, run through this
library's forward and deterministic backward on the GPU. Each row reports the
forward's and each gradient's max-abs error and relative L2 error against the
float64 oracle (gradients in function mode, i.e. fed the O and L the kernels
produced), whether the library's gate passes (|g - r| <= 5e-3 + 5e-3 |r|), and
whether the page's own tolerance band for the dtype (its DTYPE_TOL table:
fp16 1e-3 / 1e-3, bf16 5e-3 / 5e-3 as atol / rtol) holds as well. A
determinism block runs forward + backward ten times per dtype and checks the
gradients bit for bit.

Run on a GPU:  python tests/harness_report.py [output.json]
"""
import json
import os
import sys
import time

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import flashattention_backward_fa_gb300 as fa  # noqa: E402
import oracle  # noqa: E402
from flashattention_backward_fa_gb300.inputs import Workload, make_inputs  # noqa: E402

SHAPES = [(1, 8, 512, 64), (2, 16, 2048, 128), (1, 4, 8192, 64)]
PAGE_BAND = {"f16": (1e-3, 1e-3), "bf16": (5e-3, 5e-3)}   # (atol, rtol)
GATE = (5e-3, 5e-3)


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _errs(g, r, band):
    d = np.abs(g - r)
    atol, rtol = band
    return {"max_abs": float(d.max()), "rel_l2": float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300)),
            "ok": bool(np.all(d <= atol + rtol * np.abs(r)))}


def row(B, H, N, D, dtype, causal, seed):
    w = Workload(f"page_{B}x{H}x{N}x{D}_{dtype}_{'causal' if causal else 'full'}", B, H, N, D, dtype,
                 causal=causal, input_seed=seed)
    q, k, v, do = make_inputs(w)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, dod, lse, causal=causal, deterministic=True)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(clear=True) == 0
    qn, kn, vn, don = (_np(t) for t in (q, k, v, do))
    on, ln = _np(o), lse.cpu().numpy().astype(np.float64)
    t0 = time.time()
    ro, rl = oracle.forward(qn, kn, vn, w.scale, causal)
    rq, rk, rv, _ = oracle.backward(qn, kn, vn, on, don, ln, w.scale, causal)
    out = {"name": w.name, "shape_BHND": [B, H, N, D], "dtype": dtype, "causal": causal,
           "oracle_seconds": round(time.time() - t0, 2), "lse_max_abs": float(np.abs(ln - rl).max())}
    for name, g, r in (("fwd", on, ro), ("dq", _np(dq), rq), ("dk", _np(dk), rk), ("dv", _np(dv), rv)):
        gate, page = _errs(g, r, GATE), _errs(g, r, PAGE_BAND[dtype])
        out[f"{name}_max_abs"] = gate["max_abs"]
        out[f"{name}_rel_l2"] = gate["rel_l2"]
        out[f"{name}_pass_gate"] = gate["ok"]
        out[f"{name}_pass_page_band"] = page["ok"]
    out["atol_band_page"], out["rtol_band_page"] = PAGE_BAND[dtype]
    out["pass"] = all(out[f"{n}_pass_gate"] for n in ("fwd", "dq", "dk", "dv")) and out["lse_max_abs"] <= 1e-4
    out["pass_page_band"] = all(out[f"{n}_pass_page_band"] for n in ("fwd", "dq", "dk", "dv"))
    return out


def determinism(dtype, runs=10):
    w = Workload(f"det_{dtype}", 2, 16, 2048, 128, dtype, causal=True, input_seed=7)
    q, k, v, do = (t.cuda() for t in make_inputs(w))
    ref = None
    same = True
    for _ in range(runs):
        o, lse = fa.attention_forward(q, k, v, causal=True)
        g = fa.attention_backward(q, k, v, o, do, lse, causal=True, deterministic=True)
        if ref is None:
            ref = (o,) + tuple(g)
        else:
            same &= all(torch.equal(a, b) for a, b in zip(ref, (o,) + tuple(g)))
    torch.cuda.synchronize()
    return {"shape_BHND": [2, 16, 2048, 128], "dtype": dtype, "causal": True, "runs": runs,
            "bit_identical": bool(same)}


def main(path):
    rows, seed = [], 0
    for (B, H, N, D) in SHAPES:
        for dtype in ("f16", "bf16"):
            for causal in (False, True):
                rows.append(row(B, H, N, D, dtype, causal, seed))
                seed += 1
                print(json.dumps({k: rows[-1][k] for k in ("name", "pass", "pass_page_band")}), flush=True)
    report = {
        "source": "Lecture 7 — Backward Pass and Validation: harness shapes, per-tensor max-abs, tolerance bands",
        "gpu": torch.cuda.get_device_name(0),
        "library_version": fa.load_library().fa_version(),
        "gate": "|g - r| <= 5e-3 + 5e-3 |r| (16-bit), against the float64 oracle; L max-abs <= 1e-4",
        "rows": rows,
        "determinism": [determinism("f16"), determinism("bf16")],
        "all_pass": all(r["pass"] for r in rows),
    }
    with open(path, "w") as f:
        json.dump(report, f, indent=1)
    print("wrote", path, "all_pass", report["all_pass"])


if __name__ == "__main__":
    main(sys.argv[1] if len(sys.argv) > 1 else os.path.join(os.path.dirname(HERE), "harness_report.json"))
