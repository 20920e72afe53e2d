"""Shared helpers of the GPU parity tests (inputs come from the seeded generator;
expected values come from the oracle only)."""
import numpy as np
import torch

import oracle
from sparse_moe_layer_router_gb300.synthetic import as_u16

# Output tolerance of the layer (bf16 output, fp32 accumulation):
#   max|y - ref| <= 2e-2 * max|ref|  and  sum|y - ref| / sum|ref| <= 5e-3.
MAX_REL = 2e-2
MEAN_REL = 5e-3
WEIGHT_ABS = 1e-5


def tol_check(y, ref, max_rel=MAX_REL, mean_rel=MEAN_REL, what="output"):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    assert np.isfinite(y).all(), f"{what}: non-finite values"
    err = np.abs(y - ref)
    scale = np.abs(ref).max()
    emax = err.max() / max(scale, 1e-30)
    emean = err.sum() / max(np.abs(ref).sum(), 1e-30)
    assert emax <= max_rel, f"{what}: max err {emax:.3e} of max|ref| > {max_rel}"
    assert emean <= mean_rel, f"{what}: mean rel err {emean:.3e} > {mean_rel}"
    return emax, emean


def to_np_u16(t):
    return as_u16(t)


def blob_parts(blob):
    b = blob.detach().cpu().numpy().astype(np.int32)
    ids = b[:, 0, :].copy()
    w = b[:, 1, :].copy().view(np.float32)
    return ids, w


def expert_host(inp, e):
    """Host copies of one expert's weights in the oracle's tuple form."""
    cfg = inp.cfg
    if e == cfg.E:
        if cfg.quant == 0:
            return as_u16(inp.ws_gate_up), as_u16(inp.ws_down)
        return (inp.ws_gate_up.cpu().numpy(), as_u16(inp.ss_gate_up),
                inp.ws_down.cpu().numpy(), as_u16(inp.ss_down))
    if cfg.quant == 0:
        return as_u16(inp.w_gate_up[e]), as_u16(inp.w_down[e])
    return (inp.w_gate_up[e].cpu().numpy(), as_u16(inp.s_gate_up[e]),
            inp.w_down[e].cpu().numpy(), as_u16(inp.s_down[e]))


def oracle_route(inp):
    bias = None if inp.bias is None else inp.bias.cpu().numpy()
    return oracle.route(as_u16(inp.x), as_u16(inp.w_router), inp.cfg.k, bias)


def oracle_layer_rows(inp, rows, ids, w):
    """Oracle y for the token indices ``rows`` given the oracle's routing."""
    cfg = inp.cfg
    rows = np.asarray(rows)
    need = sorted(set(ids[rows].ravel().tolist()))
    experts = {e: expert_host(inp, e) for e in need}
    x = as_u16(inp.x)[rows]
    return oracle.forward(x, ids[rows], w[rows], experts, expert_host(inp, cfg.E), E=cfg.E,
                          I=cfg.I, Is=cfg.Is, quant=cfg.quant, group=cfg.group)


def y_host(y):
    return y.detach().float().cpu().numpy().astype(np.float64)


def sync():
    torch.cuda.synchronize()
