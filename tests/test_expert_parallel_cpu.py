"""Expert-parallel sharding (host logic) on two gloo ranks on the CPU.

Each rank owns half of the tokens and half of the routed experts.  It routes
its own tokens, the tokens and the packed int32 routing blobs are all-gathered
(two collectives), each rank computes the pairs routed to its own experts plus
the shared expert on its own tokens, and the fp32 partial outputs are
reduce-scattered back.  The per-rank compute here is the oracle (fp64, CPU), so
the test checks the partition and the exchange: the gathered blob must equal
the single-device routing bit for bit, and each rank's output must equal the
single-device oracle layer for its tokens.
"""
import os
import socket
import tempfile

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from sparse_moe_layer_router_gb300 import expert_parallel as ep
from sparse_moe_layer_router_gb300.synthetic import MoEConfig, as_u16, make_inputs

CFG = MoEConfig("ep_cpu", T=48, D=128, E=8, I=64, Is=64, k=3)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _route_fn(inp):
    wr = as_u16(inp.w_router)

    def f(x_local):
        ids, w = oracle.route(as_u16(x_local), wr, CFG.k)
        return torch.from_numpy(oracle.pack_blob(ids, w))
    return f


def _experts_fn(inp):
    """Routed experts [e0, e1) over every token plus the shared expert on [s0, s1)."""
    def f(x_all, blob_all, e0, e1, s0, s1):
        ids, w = oracle.unpack_blob(blob_all.numpy())
        x = as_u16(x_all)
        y = np.zeros((x.shape[0], CFG.D))
        for t in range(x.shape[0]):
            for j in range(CFG.k):
                e = int(ids[t, j])
                if e0 <= e < e1:
                    h = oracle.expert_hidden(x[t:t + 1], as_u16(inp.w_gate_up[e]))
                    y[t] += float(w[t, j]) * oracle.expert_down(h, as_u16(inp.w_down[e]))[0]
        if s1 > s0:
            h = oracle.expert_hidden(x[s0:s1], as_u16(inp.ws_gate_up))
            y[s0:s1] += oracle.expert_down(h, as_u16(inp.ws_down))
        return torch.from_numpy(y)
    return f


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = make_inputs(CFG)
        n = CFG.T // world
        x_local = inp.x[rank * n:(rank + 1) * n]
        y_local, blob_all = ep.ep_forward(x_local, CFG.E, _route_fn(inp), _experts_fn(inp))
        np.save(os.path.join(out_dir, f"y{rank}.npy"), y_local.numpy())
        np.save(os.path.join(out_dir, f"blob{rank}.npy"), blob_all.numpy())
    finally:
        dist.destroy_process_group()


def test_block_ranges_partition():
    for n in (1, 7, 8, 512, 513):
        for world in (1, 2, 3, 8):
            if world > n:
                continue
            parts = [ep.block_range(n, world, r) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(parts, parts[1:]))
            sizes = [e - b for b, e in parts]
            assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1
    with pytest.raises(ValueError):
        ep.expert_range(4, 8, 0)


def test_two_rank_expert_parallel_matches_single_device():
    oracle.build()
    world = 2
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_worker, args=(world, _free_port(), d), nprocs=world, join=True)
        ys = [np.load(os.path.join(d, f"y{r}.npy")) for r in range(world)]
        blobs = [np.load(os.path.join(d, f"blob{r}.npy")) for r in range(world)]
    inp = make_inputs(CFG)
    x = as_u16(inp.x)
    ids_ref, w_ref = oracle.route(x, as_u16(inp.w_router), CFG.k)
    blob_ref = oracle.pack_blob(ids_ref, w_ref)
    for b in blobs:                       # the all-gathered routing, on every rank
        assert b.dtype == np.int32 and np.array_equal(b, blob_ref)
    _, w32 = oracle.unpack_blob(blob_ref)  # the weights as the blob carries them
    experts = {e: (as_u16(inp.w_gate_up[e]), as_u16(inp.w_down[e])) for e in range(CFG.E)}
    y_ref = oracle.forward(x, ids_ref, w32.astype(np.float64), experts,
                           (as_u16(inp.ws_gate_up), as_u16(inp.ws_down)), E=CFG.E, I=CFG.I,
                           Is=CFG.Is)
    y = np.concatenate(ys)
    assert y.shape == y_ref.shape
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12 * np.abs(y_ref).max())
