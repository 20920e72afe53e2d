"""moe_forward_experts (the expert-parallel slice of the layer) on one GPU.

The routed experts are cut into contiguous ranges, as the ranks of an
expert-parallel group would hold them, and the shared expert's tokens into
disjoint ranges.  One call per range, each given only its own experts'
weights; the fp32 partial outputs summed must equal the oracle layer within
the layer tolerance, and ranges that own no routed row must contribute nothing.
"""
import numpy as np
import pytest
import torch

from sparse_moe_layer_router_gb300 import binding as B
from sparse_moe_layer_router_gb300.build import build
from sparse_moe_layer_router_gb300.synthetic import MoEConfig, make_inputs

from helpers import blob_parts, oracle_layer_rows, oracle_route, tol_check

pytestmark = pytest.mark.gpu

CASES = {
    "ep_bf16": MoEConfig("ep_bf16", T=96, D=256, E=12, I=128, Is=128, k=3),
    # hot experts and empty experts (Zipf-biased router), 256-row token tiles
    "ep_hot": MoEConfig("ep_hot", T=2100, D=256, E=16, I=64, Is=64, k=2, zipf_s=1.2,
                        zipf_alpha=3.0),
    # T >= 2048: the split bf16 launch (hot and cold grids) inside each range
    "ep_split": MoEConfig("ep_split", T=2100, D=256, E=64, I=64, Is=64, k=4, zipf_s=1.2,
                          zipf_alpha=0.3),
    "ep_w4": MoEConfig("ep_w4", T=64, D=512, E=10, I=256, Is=256, k=3, quant=1),
    "ep_w4_channel": MoEConfig("ep_w4_channel", T=64, D=512, E=10, I=256, Is=256, k=3,
                               quant=1, group=0),
}


@pytest.fixture(scope="module", autouse=True)
def built(cuda_ok):
    build()
    B.lib()


def local_weights(inp, e0, e1):
    """The weights a rank holding experts [e0, e1) would have (no router)."""
    def sl(t):
        return None if t is None else t[e0:e1].contiguous()
    return B.MoeWeights(None, None, B._p(sl(inp.w_gate_up)), B._p(sl(inp.w_down)),
                        B._p(sl(inp.s_gate_up)), B._p(sl(inp.s_down)), B._p(inp.ws_gate_up),
                        B._p(inp.ws_down), B._p(inp.ss_gate_up), B._p(inp.ss_down)), \
        [sl(inp.w_gate_up), sl(inp.w_down), sl(inp.s_gate_up), sl(inp.s_down)]


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("parts", [2, 3])
def test_expert_ranges_sum_to_the_layer(name, parts):
    cfg = CASES[name]
    host = make_inputs(cfg, device="cpu")
    dev = host.to("cuda")
    blob = B.route(cfg, dev.x, dev.w_router, dev.bias)
    ws = B.workspace(cfg, B.MOE_ENTRY_FORWARD_EXPERTS)
    total = torch.zeros((cfg.T, cfg.D), dtype=torch.float32, device="cuda")
    keep = []
    for r in range(parts):
        e0, e1 = r * cfg.E // parts, (r + 1) * cfg.E // parts
        s0, s1 = r * cfg.T // parts, (r + 1) * cfg.T // parts
        w, tensors = local_weights(dev, e0, e1)
        keep.append(tensors)
        y = B.forward_experts(cfg, dev.x, blob, w, e0, e1, s0, s1, ws=ws)
        total += y
    torch.cuda.synchronize()
    assert B.get_status(ws) == B.MOE_OK
    ids_ref, w_ref = oracle_route(host)
    ids, _ = blob_parts(blob)
    assert np.array_equal(ids, ids_ref)
    ref = oracle_layer_rows(host, np.arange(cfg.T), ids_ref, w_ref)
    tol_check(total.double().cpu().numpy(), ref, what=f"{name}: sum of {parts} expert ranges")


def test_range_without_routed_rows_gives_only_the_shared_expert():
    cfg = CASES["ep_hot"]
    host = make_inputs(cfg, device="cpu")
    dev = host.to("cuda")
    blob = B.route(cfg, dev.x, dev.w_router, dev.bias)
    ids, _ = blob_parts(blob)
    empty = sorted(set(range(cfg.E)) - set(np.unique(ids).tolist()))
    assert empty, "the Zipf bias leaves some experts without tokens"
    e = empty[0]
    w, keep = local_weights(dev, e, e + 1)
    y_none = B.forward_experts(cfg, dev.x, blob, w, e, e + 1, 0, 0)
    y_sh = B.forward_experts(cfg, dev.x, blob, w, e, e + 1, 5, 9)
    torch.cuda.synchronize()
    assert torch.count_nonzero(y_none).item() == 0
    assert torch.count_nonzero(y_sh[:5]).item() == 0 and torch.count_nonzero(y_sh[9:]).item() == 0
    ids_ref, w_ref = oracle_route(host)
    zero_w = np.zeros_like(w_ref)  # routed weights zero: the oracle layer is the shared expert
    ref = oracle_layer_rows(host, np.arange(5, 9), ids_ref, zero_w)
    tol_check(y_sh[5:9].double().cpu().numpy(), ref, what="shared expert on tokens 5..8")


def test_bad_ranges_rejected():
    cfg = CASES["ep_bf16"]
    d = torch.zeros(16, dtype=torch.int32, device="cuda")
    w = B.MoeWeights(None, None, B._p(d), B._p(d), None, None, B._p(d), B._p(d), None, None)
    ws = B.workspace(cfg, B.MOE_ENTRY_FORWARD_EXPERTS)
    p = d.data_ptr()  # raw pointers: the library's own range checks, not the binding's
    for e0, e1, s0, s1 in [(3, 3, 0, 0), (-1, 2, 0, 0), (0, cfg.E + 1, 0, 0), (0, 2, 5, 4),
                           (0, 2, 0, cfg.T + 1)]:
        with pytest.raises(B.MoeError) as ex:
            B.forward_experts(cfg, p, p, w, e0, e1, s0, s1, y_partial=p, ws=ws)
        assert ex.value.code == B.MOE_ERR_INVALID_ARG


@pytest.mark.timeout(300)
def test_ep_forward_one_rank_through_the_library():
    """The expert-parallel step (route, the two all-gathers, the expert slice,
    the reduce-scatter) with this library's kernels on a one-rank NCCL group:
    the collectives are identities, so the result must match moe_forward's
    layer output within the layer tolerance."""
    import socket
    import torch.distributed as dist
    from sparse_moe_layer_router_gb300 import expert_parallel as ep

    cfg = CASES["ep_bf16"]
    host = make_inputs(cfg, device="cpu")
    dev = host.to("cuda")
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    store = dist.TCPStore("127.0.0.1", port, 1, True)
    dist.init_process_group("nccl", store=store, rank=0, world_size=1)
    try:
        route_fn, experts_fn = ep.library_fns(
            cfg, cfg, dev.w_router, dev.bias,
            {"w_gate_up": dev.w_gate_up, "w_down": dev.w_down},
            {"ws_gate_up": dev.ws_gate_up, "ws_down": dev.ws_down})
        y_local, blob_all = ep.ep_forward(dev.x, cfg.E, route_fn, experts_fn)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    y_ref = B.forward(cfg, dev.x, dev)
    ids_ref, w_ref = oracle_route(host)
    ids, _ = blob_parts(blob_all)
    assert np.array_equal(ids, ids_ref)
    ref = oracle_layer_rows(host, np.arange(cfg.T), ids_ref, w_ref)
    tol_check(y_local.double().cpu().numpy(), ref, what="expert-parallel step, one rank")
    tol_check(y_ref.double().cpu().numpy(), y_local.double().cpu().numpy(), what="vs moe_forward")
