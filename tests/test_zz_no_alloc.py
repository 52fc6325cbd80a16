"""fa_bwd_noalloc: the deterministic backward without a caller-supplied workspace.

It exists for callers that cannot allocate device memory when they run the
backward (a pre-planned memory arena, a runtime recording work before any
allocator exists, an embedding that only hands over tensors). It takes its
scratch from one fixed device array inside the library, so these tests check
that its results equal the workspace entry point's on two calls in a row (the
array keeps the previous call's contents, which must not leak into the next
result), and that problems beyond the array's size are refused before any
launch. The file is named to be collected last.
"""
import ctypes

import pytest
import torch

import flashattention_backward_fa_gb300 as fa
from flashattention_backward_fa_gb300.inputs import Workload, make_inputs

MAX_ROWS = 1 << 20  # B * H * roundup(N, 128) the fixed scratch holds


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,d,causal,window", [("bf16", 128, True, 0), ("f16", 64, True, 96), ("f32", 64, False, 0)])
def test_noalloc_matches_workspace_entry_point_twice(dtype, d, causal, window):
    # Two different problems in a row through the no-allocation entry point. The
    # first covers more scratch rows (2*3*768 padded rows) than the second
    # (2*3*256), so the second call runs over rows the first one left behind and
    # must not see anything of them. Both calls run the same deterministic
    # kernels as fa_bwd, so their outputs must be bit-identical to fa_bwd's; the
    # second call is also held to the float64 oracle under the usual gate.
    import numpy as np

    import oracle
    from gpu_check import to_np, within

    for call, (N, seed) in enumerate(((700, 5), (130, 6))):
        w = Workload(f"noalloc_{dtype}_{call}", 2, 3, N, d, dtype, causal=causal, window=window,
                     input_seed=4000 + seed)
        q, k, v, do = (t.cuda() for t in make_inputs(w))
        o, lse = fa.attention_forward(q, k, v, scale=w.scale, causal=causal, window=window)
        ref = fa.attention_backward(q, k, v, o, do, lse, scale=w.scale, causal=causal, window=window,
                                    deterministic=True)
        out = [torch.full_like(q, float("nan")) for _ in range(3)]
        fa.fa_bwd_noalloc(q, k, v, o, do, lse, *out, scale=w.scale, causal=causal, window=window)
        torch.cuda.synchronize()
        assert fa.fa_get_device_status(clear=True) == 0
        for name, a, r in zip(("dq", "dk", "dv"), out, ref):
            assert torch.equal(a, r), (call, name)
        if call == 1:
            rq, rk, rv, _ = oracle.backward(to_np(q), to_np(k), to_np(v), to_np(o), to_np(do),
                                            lse.double().cpu().numpy(), w.scale, causal, window)
            floor = float(np.linalg.norm(rv))
            for name, a, r in zip(("dq", "dk", "dv"), out, (rq, rk, rv)):
                ok, rep = within(to_np(a), r, dtype, floor)
                assert ok, (name, rep)


def test_noalloc_rejects_problems_beyond_its_scratch():
    """Sizes beyond the fixed array are refused before any CUDA call (runs without a GPU)."""
    lib = fa.load_library()
    B, H, d = 1, 1, 128
    N = MAX_ROWS + 1  # one padded block more than the scratch holds
    st = fa.FaStrides(N * H * d, H * d, d)
    P = 0x10000
    rc = lib.fa_bwd_noalloc(*([P] * 9), B, H, N, d, st, fa.FA_BF16, 0.1, 1, 0, 0.0, 0, 0, None)
    assert rc == -4  # FA_ERR_WORKSPACE
    rc = lib.fa_bwd_noalloc(*([P] * 9), 0, H, 64, d, st, fa.FA_BF16, 0.1, 1, 0, 0.0, 0, 0, None)
    assert rc == -1  # invalid size
    # Beyond the library's size limits the answer is fa_bwd's, not the scratch's.
    N = (1 << 30) + 1
    st = fa.FaStrides(N * H * d, H * d, d)
    rc = lib.fa_bwd_noalloc(*([P] * 9), B, H, N, d, st, fa.FA_BF16, 0.1, 1, 0, 0.0, 0, 0, None)
    assert rc == -2  # FA_ERR_UNSUPPORTED, as fa_bwd returns
    assert lib.fa_bwd_workspace_size(B, H, N, d, fa.FA_BF16, 1) == 0
