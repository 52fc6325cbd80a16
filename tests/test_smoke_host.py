"""The smoke check's comparison path, run on the host.

``__graft_entry__.smoke()`` needs a GPU. Its comparison against the oracle
does not: feeding it the oracle's own forward and backward must pass, and a
gradient with a planted error must fail. This keeps the smoke entry point
callable (signatures, tolerances) on machines without a GPU.
"""
import numpy as np
import pytest

import __graft_entry__ as entry
import oracle
from flashattention_backward_fa_gb300.inputs import make_inputs


@pytest.mark.parametrize("w", entry.smoke_workloads(), ids=lambda w: w.name)
def test_smoke_check_accepts_oracle_results(w):
    q, k, v, do = (t.double().numpy() for t in make_inputs(w))
    o, lse = oracle.forward(q, k, v, w.scale, w.causal, w.window, w.dropout_p, w.philox_seed, w.philox_offset)
    dq, dk, dv, _ = oracle.backward(q, k, v, o, do, lse, w.scale, w.causal, w.window, w.dropout_p, w.philox_seed,
                                    w.philox_offset)
    entry.check_smoke_case(w, (q, k, v, do), o, lse, (dq, dk, dv))


def test_smoke_check_rejects_a_planted_error():
    w = entry.smoke_workloads()[0]
    q, k, v, do = (t.double().numpy() for t in make_inputs(w))
    o, lse = oracle.forward(q, k, v, w.scale, w.causal, w.window)
    dq, dk, dv, _ = oracle.backward(q, k, v, o, do, lse, w.scale, w.causal, w.window)
    dk = dk.copy()
    dk[0, 5, 1, 7] += 0.1 + 0.1 * abs(dk[0, 5, 1, 7])
    with pytest.raises(AssertionError):
        entry.check_smoke_case(w, (q, k, v, do), o, lse, (dq, dk, dv))
