"""Failure detection on the GPU without a fault.

The tensor-core kernels bound every mbarrier wait by wall-clock time; a wait
that gives up sets the timeout bit of the device status word, raises its CTA's
abort flag, drains (with a bound) and frees TMEM, so the context stays usable.
fa_selftest_timeout launches one CTA whose waits can never complete (an
mbarrier that nothing arrives on), through the same wait and drain functions.
This test checks that both wait styles give up, that the host reads
FA_ERR_TIMEOUT, that clearing works, and that a normal backward afterwards still
matches the oracle with a clean status.
"""
import ctypes
import time

import pytest
import torch

import flashattention_backward_fa_gb300 as fa
from flashattention_backward_fa_gb300 import binding
from flashattention_backward_fa_gb300.inputs import Workload
from gpu_check import check_against_oracle, run_gpu

pytestmark = pytest.mark.gpu

FA_ERR_TIMEOUT = -6


def _status_code():
    s = ctypes.c_uint(0)
    code = binding.load_library().fa_get_device_status(ctypes.byref(s), 0)
    return code, int(s.value)


def test_bounded_wait_gives_up_and_context_survives():
    torch.cuda.synchronize()
    fa.fa_get_device_status(clear=True)            # start from a clean word
    assert _status_code() == (0, 0)

    t0 = time.monotonic()
    outcome = fa.fa_selftest_timeout()            # synchronises through .item()
    elapsed = time.monotonic() - t0
    assert outcome == 3, outcome                  # both the polling and the blocking wait gave up
    # one wait limit (4 s) plus the bounded drain (4 s); well under a minute
    assert 7.0 <= elapsed <= 60.0, elapsed

    code, bits = _status_code()
    assert code == FA_ERR_TIMEOUT and bits & 1, (code, bits)
    assert fa.fa_get_device_status(clear=True) & 1   # read and clear
    assert _status_code() == (0, 0)

    # The context is still usable: a backward on the tensor cores matches the oracle.
    w = Workload("after_timeout", 1, 2, 300, 128, "bf16", causal=True, input_seed=7)
    res = run_gpu(w)
    fails, _ = check_against_oracle(w, res, exact=False)
    assert not fails, fails
    assert _status_code() == (0, 0)


def test_host_pointers_are_refused_before_any_launch():
    """The C ABI checks that every buffer is memory of the current device before it
    launches anything (a host pointer would make the kernels fault); the binding
    refuses CPU tensors itself."""
    w = Workload("ptr_check", 1, 2, 256, 64, "bf16", causal=True, input_seed=3)
    from flashattention_backward_fa_gb300.inputs import make_inputs
    q, k, v, do = (t.cuda() for t in make_inputs(w))
    o, lse = fa.attention_forward(q, k, v, causal=True)
    dq, dk, dv = (torch.full_like(q, 7.0) for _ in range(3))
    ws = fa.alloc_workspace(q, True)
    torch.cuda.synchronize()
    fa.fa_get_device_status(clear=True)
    lib = binding.load_library()
    base = list(binding._bwd_args(q, k, v, o, do, lse, dq, dk, dv, None, True, 0, 0.0, 0, 0, True, ws, None))
    nbytes = base[23]
    host_ws = torch.empty(nbytes + 256, dtype=torch.uint8)           # pageable host memory
    host_dq = torch.empty(q.shape, dtype=q.dtype)                    # a CPU tensor
    host_lse = torch.empty(lse.shape, dtype=lse.dtype)
    for idx, ptr in ((22, (host_ws.data_ptr() + 255) & ~255), (6, host_dq.data_ptr()), (5, host_lse.data_ptr())):
        args = list(base)
        args[idx] = ptr
        assert lib.fa_bwd(*args) == -1, idx                          # FA_ERR_INVALID_ARG
    # the forward refuses a host L buffer the same way
    st = binding._layout(q)[1]
    assert lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), host_lse.data_ptr(), 1, 2, 256, 64,
                      st, 2, binding.default_scale(64), 1, 0, 0.0, 0, 0, binding._stream(None)) == -1
    torch.cuda.synchronize()
    assert bool((dq == 7.0).all()) and bool((dk == 7.0).all())       # nothing ran
    assert fa.fa_get_device_status(clear=True) == 0
    # the binding refuses CPU tensors before calling the library
    with pytest.raises(ValueError):
        fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, host_ws, causal=True)
    with pytest.raises(ValueError):
        fa.fa_bwd(q, k, v, o, do, lse.cpu(), dq, dk, dv, ws, causal=True)
