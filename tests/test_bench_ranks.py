"""The bench's replica path on CPU: two gloo ranks, each with its own step
time; the job's time is the slowest rank's and its throughput counts every
rank's tokens."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [3.0, 5.0][rank]
    job_ms = bench.max_over_ranks(ms, torch.device("cpu"), world)
    q.put((rank, job_ms, bench.replica_throughput(1000, job_ms, world)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, job_ms, value in got:
        assert job_ms == 5.0
        assert value == pytest.approx(2 * 1000 / 5e-3)


def test_single_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.0, None, 1) == 4.0
    assert bench.replica_throughput(16384, 8.0, 1) == pytest.approx(16384 / 8e-3)


def test_algorithmic_work_matches_the_hand_counts():
    """The roofline numerators: per-forward work of the Mixtral-shaped layer
    (T=16384, d=4096, f=14336, E=8, k=2, SwiGLU, bf16, no drops), counted by
    hand from the shapes."""
    sys.path.insert(0, ROOT)
    import bench
    import seeded_inputs as si
    cfg = si.CONFIGS["mixtral_swiglu_bf16"]
    T, d, f, E, k = 16384, 4096, 14336, 8, 2
    A = T * k
    w = bench.algorithmic(cfg, A)
    assert w["gemm1_flop"] == 2 * A * d * f * 2            # x W1 and x W3
    assert w["gemm2_flop"] == 2 * A * f * d
    assert abs(w["gemm1_flop"] + w["gemm2_flop"] - 11.54e12) < 0.01e12
    assert w["router_bytes"] == T * d * 2 + d * E * 2 + T * k * 8
    assert w["gather_bytes"] == T * d * 2 + A * d * 2      # x read once, one copy per kept slot
    assert w["combine_bytes"] == A * d * 4 + T * d * 2     # O (fp32) read, y (bf16) written
    # FP8 experts: one code per element and one scale per grouped row
    w8 = bench.algorithmic(cfg.replace(fp8_experts=True), A)
    assert w8["gather_bytes"] == T * d * 2 + A * (d + 4)
    assert w8["quantize_h_bytes"] == A * (f * 3 + 4)
