"""The bench's multi-rank arithmetic on CPU: two gloo ranks (127.0.0.1) report
different durations; both must see the slowest, and the job throughput counts
every rank's tokens over that time."""
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


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms = [12.5, 20.0][rank]
        slow = bench.slowest_rank(ms, world, "cpu")
        out[rank] = (slow, bench.job_tokens_per_s(world, 64, 10, slow / 1e3))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_and_job_throughput_two_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    slow, value = res[0]
    assert slow == 20.0
    assert value == pytest.approx(2 * 64 * 10 / 0.020)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank(3.5, 1, "cpu") == 3.5
    assert bench.job_tokens_per_s(1, 64, 100, 2.0) == 3200.0


def test_extra_workloads_exist_and_share_weights_where_bench_reuses_them():
    """Every workload the default run measures is a known configuration, and
    with_tokens (used to reuse expert weights between neighbouring workloads)
    gives exactly the inputs make_inputs draws for the new configuration."""
    sys.path.insert(0, ROOT)
    import torch
    import bench
    from sparse_moe_layer_router_gb300.synthetic import CONFIGS, make_inputs, with_tokens
    for n in bench.EXTRA_WORKLOADS:
        assert n in CONFIGS, n
    base = CONFIGS["tiny"]
    other = base.with_(name="tiny_skewed", T=96, zipf_s=1.2, zipf_alpha=0.9)
    a = with_tokens(make_inputs(base), other)
    b = make_inputs(other)
    for f in ("x", "w_router", "bias", "w_gate_up", "w_down", "ws_gate_up", "ws_down"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f
    with pytest.raises(ValueError):
        with_tokens(make_inputs(base), base.with_(name="tiny_e8", E=8))


def test_step_launch_count_follows_the_dispatch_and_split_rules():
    """One block of dispatch up to 4096 (token, slot) pairs, else three; the
    hot/cold split (bf16, 256-row tiles, under 512 rows per expert) adds a plan
    kernel and a second grid to each of the two GEMMs."""
    sys.path.insert(0, ROOT)
    import bench
    from sparse_moe_layer_router_gb300.synthetic import CONFIGS
    want = {"decode": 8, "prefill": 10, "skewed": 14, "w4a16": 10, "dense_e64": 10,
            "w4a16_dense_e64": 10, "skewed_e64": 14, "tiny": 8}
    for name, n in want.items():
        assert bench.step_launches(CONFIGS[name]) == n, name
