"""Host logic of bench.py that needs no GPU: FLOP counting and the multi-rank
timing reduction (max over ranks) on two gloo ranks."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from flashattention_backward_fa_gb300.inputs import WORKLOADS  # noqa: E402


def test_counted_flops():
    assert bench.counted_flops(WORKLOADS["bf16_causal_b1h32_n8192_d128"]) == pytest.approx(1.374389534720e12)
    assert bench.counted_flops(WORKLOADS["bf16_causal_b4h16_n2048_d128"]) == pytest.approx(1.717986918e11)
    assert bench.counted_flops(WORKLOADS["bf16_causal_b1h8_n32768_d128"]) == pytest.approx(5.497558e12, rel=1e-6)
    w5 = WORKLOADS["fp16_window1024_drop0.1_b2h16_n4096_d64"]
    pairs_per_head = sum(min(i + 1, 1024) for i in range(4096))
    assert pairs_per_head == 3670528
    assert bench.counted_flops(w5) == pytest.approx(10 * 64 * pairs_per_head * 32)
    assert bench.counted_flops(WORKLOADS["fp32_n128_d64"]) == 10 * 128 * 128 * 64


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    m = bench.max_over_ranks(1.0 + rank, world)
    dist.destroy_process_group()
    q.put((rank, m))


def test_max_over_ranks_gloo_two_ranks():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.0), (1, 2.0)]


def test_reference_arm_runs_warmup_and_timed_steps():
    """--impl reference: W warm-up and K timed steps of the oracle, one head each."""
    w = WORKLOADS["fp32_n128_d64"]
    tf, sample, cores, sec = bench.run_reference_steps(w, steps=3, warmup=2)
    assert tf > 0 and sec > 0 and cores >= 1
    assert sample.startswith("3 timed step(s) after 2 warm-up step(s)")
    # A budget too small for K + W steps keeps at least one of each and says so.
    tf, sample, _, _ = bench.run_reference_steps(w, steps=50, warmup=10, budget_s=1e-9)
    assert tf > 0
    assert sample.startswith("1 timed step(s) after 1 warm-up step(s)")
