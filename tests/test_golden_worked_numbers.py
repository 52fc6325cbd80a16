"""The pages' worked numbers for the backward's memory and work, against the
library's own accounting (CPU only).

Fixture: tests/golden/worked_numbers_saved_state.txt ("FlashAttention backward",
section "Worked numbers: why O(N^2) was never an option").
"""
import os

import pytest

import flashattention_backward_fa_gb300 as fa
from flashattention_backward_fa_gb300 import binding

HERE = os.path.dirname(os.path.abspath(__file__))


def _fixture():
    rows, ratio = [], None
    with open(os.path.join(HERE, "golden", "worked_numbers_saved_state.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == "ratio_bwd_fwd":
                ratio = float(parts[1])
            else:
                rows.append((int(parts[0]), float(parts[1]), float(parts[2]), float(parts[3])))
    return rows, ratio


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(binding.LIB_PATH):
        from flashattention_backward_fa_gb300.build import build_library
        build_library()
    return fa.load_library()


def test_printed_figures_follow_from_the_sizes():
    rows, _ = _fixture()
    d = 128
    for N, p_printed, saved_printed, ratio_printed in rows:
        p_bytes = N * N * 2
        saved = N * d * 2 + N * 4 * 2
        # the page rounds to two significant figures (decimal or binary units)
        assert abs(p_bytes - p_printed) / p_printed < 0.08, N
        assert abs(saved - saved_printed) / saved_printed < 0.08, N
        assert abs(p_bytes / saved - ratio_printed) / ratio_printed < 0.08, N


def test_library_keeps_linear_state(lib):
    """What the backward holds besides the inputs is O, L and the workspace; it
    grows linearly in N (plus a constant block) and stays within 2% of the
    page's O + L + D."""
    rows, _ = _fixture()
    d = 128
    for N, p_printed, saved_printed, ratio_printed in rows:
        ws = fa.fa_bwd_workspace_size(1, 1, N, d, fa.FA_BF16, True)
        # -L*log2(e) and -D, fp32, padded rows, plus a constant 256-byte block of unit counters
        assert ws == 2 * 4 * ((N + 127) // 128 * 128) + 256
        ours = N * d * 2 + N * 4 + ws                    # O + L + workspace
        page = N * d * 2 + N * 4 * 2
        assert ours <= 1.02 * page
        assert N * N * 2 / ours > 0.95 * ratio_printed


def test_backward_counts_two_and_a_half_forwards():
    import bench
    from flashattention_backward_fa_gb300.inputs import Workload
    _, ratio = _fixture()
    for causal, window in ((False, 0), (True, 0), (True, 300), (False, 300)):
        w = Workload("flops", 2, 3, 1000, 64, "bf16", causal=causal, window=window)
        # forward: 4*d per allowed pair (S and P V); backward: 10*d (S, dP, dV, dK, dQ)
        pairs = sum(1 for i in range(w.N) for j in range(w.N)
                    if (not causal or j <= i) and (window == 0 or j > i - window))
        if window:
            assert bench.counted_flops(w) == pytest.approx(10 * w.d * pairs * w.B * w.H)
        assert bench.counted_flops(w) / (4 * w.d * pairs * w.B * w.H) == pytest.approx(ratio, rel=0.01 if not window else 1e-12)
