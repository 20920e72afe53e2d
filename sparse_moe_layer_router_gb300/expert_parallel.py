"""Expert-parallel sharding of the MoE layer over the ranks of a process group.

"Systems engineering playbook: optimizing Qwen 3.5-397B MoE on Ironwood
(TPU7x)", section 3, "Option B": every device holds E / G of the routed
experts; all tokens and their routing reach every device; each device filters
the (token, slot) pairs routed to its own experts and computes them; the
partial outputs are reduce-scattered back to the devices that own the tokens.
Same section, "3-to-2 All-Gather optimisation": the routing ids and weights
travel as one int32 blob (the layout ``moe_route`` writes), so the exchange
is two all-gathers (tokens, blob) instead of three.

This module is host logic only: the partition of experts and tokens over the
ranks and the three collectives.  The per-rank compute is passed in:
``route_fn`` (``binding.route`` on a GPU) and ``experts_fn``
(``binding.forward_experts`` on a GPU, which also applies the shared expert to
the rank's own tokens).  The shared expert is data-parallel: each rank applies
it to the tokens it owns, so every token gets it exactly once.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def block_range(n: int, world: int, rank: int) -> tuple[int, int]:
    """[begin, end) of part ``rank`` when n items are cut into ``world``
    contiguous parts whose sizes differ by at most one."""
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside [0, {world})")
    return rank * n // world, (rank + 1) * n // world


def expert_range(E: int, world: int, rank: int) -> tuple[int, int]:
    """The routed experts [e_begin, e_end) that rank ``rank`` holds."""
    if world > E:
        raise ValueError(f"{world} ranks for {E} experts: every rank needs one")
    return block_range(E, world, rank)


def all_gather_rows(local: torch.Tensor, group=None) -> torch.Tensor:
    """Every rank's ``local`` rows stacked in rank order (equal row counts).
    The bytes travel unchanged: rows are sent as raw bytes, whatever their type."""
    world = dist.get_world_size(group)
    send = local.contiguous().view(torch.uint8)
    out = torch.empty((world * send.shape[0],) + tuple(send.shape[1:]), dtype=torch.uint8,
                      device=send.device)
    dist.all_gather_into_tensor(out, send, group=group)
    return out.view(local.dtype)


def reduce_scatter_rows(partial: torch.Tensor, group=None) -> torch.Tensor:
    """Sum of every rank's ``partial`` [world * n, ...], rank r receiving rows
    [r * n, (r + 1) * n)."""
    world = dist.get_world_size(group)
    if partial.shape[0] % world:
        raise ValueError("rows not divisible by the world size")
    out = torch.empty((partial.shape[0] // world,) + tuple(partial.shape[1:]),
                      dtype=partial.dtype, device=partial.device)
    dist.reduce_scatter_tensor(out, partial.contiguous(), op=dist.ReduceOp.SUM, group=group)
    return out


def ep_forward(x_local: torch.Tensor, E: int, route_fn, experts_fn, group=None):
    """One expert-parallel layer step on this rank.

    x_local      bf16 [T_local, D], the tokens this rank owns (equal on every rank).
    route_fn     x_local -> int32 blob [T_local, 2, k] (softmax, top-k, renormalised).
    experts_fn   (x_all, blob_all, e_begin, e_end, s_begin, s_end) -> fp32 [T, D]:
                 the routed experts [e_begin, e_end) over every token plus the
                 shared expert on tokens [s_begin, s_end).
    Returns (y_local fp32 [T_local, D], blob_all int32 [T, 2, k]): this rank's
    tokens' layer output before the final bf16 rounding, and the gathered routing.
    """
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    blob_local = route_fn(x_local)
    x_all = all_gather_rows(x_local, group)          # collective 1: tokens
    blob_all = all_gather_rows(blob_local, group)    # collective 2: ids + weights in one blob
    e0, e1 = expert_range(E, world, rank)
    n = x_local.shape[0]
    y_partial = experts_fn(x_all, blob_all, e0, e1, rank * n, (rank + 1) * n)
    return reduce_scatter_rows(y_partial, group), blob_all   # collective 3: outputs home


def library_fns(cfg_local, cfg_all, w_router, bias, local_weights, shared_weights=None):
    """(route_fn, experts_fn) for ep_forward backed by this library's kernels.

    cfg_local     shapes of one rank's call to the router (T = tokens per rank).
    cfg_all       shapes of the expert slice (T = all ranks' tokens, E = all experts).
    w_router      bf16 [E, D] router weight (every rank holds it); bias fp32 [E] or None.
    local_weights dict with this rank's experts: w_gate_up, w_down (and, for W4A16,
                  s_gate_up, s_down), leading dimension e_end - e_begin.
    shared_weights dict with ws_gate_up, ws_down (ss_gate_up, ss_down for W4A16).
    """
    from . import binding as B

    sw = shared_weights or {}
    weights = B.MoeWeights(None, None, B._p(local_weights["w_gate_up"]),
                           B._p(local_weights["w_down"]), B._p(local_weights.get("s_gate_up")),
                           B._p(local_weights.get("s_down")), B._p(sw.get("ws_gate_up")),
                           B._p(sw.get("ws_down")), B._p(sw.get("ss_gate_up")),
                           B._p(sw.get("ss_down")))

    def route_fn(x_local):
        return B.route(cfg_local, x_local, w_router, bias)

    def experts_fn(x_all, blob_all, e0, e1, s0, s1):
        return B.forward_experts(cfg_all, x_all, blob_all, weights, e0, e1, s0, s1)

    return route_fn, experts_fn
