"""Index data from the caller that lies outside its range.

Expert ids in a blob, grouped-GEMM offsets and pair indices, gather rows and
combine rows are clamped into range on the device: every access stays inside
the buffers, and the entries that take a workspace record MOE_ERR_INVALID_ARG
in its status word.  Where the clamped result is defined (permute, combine)
it is compared with the oracle on the clamped indices; elsewhere the test
checks the status and that guard rows past the output are untouched.
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_moe_layer_router_gb300 import binding as B
from sparse_moe_layer_router_gb300.build import build
from sparse_moe_layer_router_gb300.synthetic import MoEConfig, make_inputs

from helpers import oracle_route, tol_check, y_host

pytestmark = pytest.mark.gpu

GUARD = 32


@pytest.fixture(scope="module", autouse=True)
def built(cuda_ok):
    build()
    B.lib()


def bad_blob(cfg, seed):
    """A routing blob of valid ids with some replaced by out-of-range values."""
    host = make_inputs(cfg, device="cpu")
    ids, w = oracle_route(host)
    rng = np.random.default_rng(seed)
    bad = ids.copy()
    flat = bad.reshape(-1)
    where = rng.choice(flat.size, size=max(3, flat.size // 50), replace=False)
    vals = np.array([-1, -7, cfg.E, cfg.E + 3, 1 << 30, -(1 << 30)], np.int32)
    flat[where] = vals[np.arange(where.size) % vals.size]
    return host, bad, w, np.clip(bad, 0, cfg.E - 1)


@pytest.mark.parametrize("T,E,k", [(37, 24, 3), (1000, 50, 5)])
def test_permute_clamps_expert_ids(T, E, k):
    """One-block (T*k <= 4096) and count/scan/scatter (T*k > 4096) paths."""
    cfg = MoEConfig(f"badperm{T}", T=T, D=128, E=E, I=64, Is=64, k=k)
    _, bad, w, clamped = bad_blob(cfg, 1)
    blob = torch.from_numpy(oracle.pack_blob(bad, w)).cuda()
    ws = B.workspace(cfg, B.MOE_ENTRY_PERMUTE)
    counts, offsets, perm, inv = B.permute(cfg, blob, ws=ws)
    torch.cuda.synchronize()
    assert B.get_status(ws) == B.MOE_ERR_INVALID_ARG
    assert B.get_status(ws) == B.MOE_OK  # reading clears it
    c_ref, o_ref, p_ref, i_ref = oracle.permute(clamped, cfg.E)
    assert (counts.cpu().numpy() == c_ref).all()
    assert (offsets.cpu().numpy() == o_ref).all()
    assert (perm.cpu().numpy() == p_ref).all()
    assert (inv.cpu().numpy() == i_ref).all()
    # the fixed-scratch entry clamps the same way (it has no status word)
    s_counts, s_offsets, s_perm, s_inv = B.permute_static(cfg, blob)
    torch.cuda.synchronize()
    assert (s_perm.cpu().numpy() == p_ref).all() and (s_inv.cpu().numpy() == i_ref).all()


def test_combine_clamps_rows():
    cfg = MoEConfig("badcomb", T=40, D=256, E=16, I=64, Is=64, k=3)
    P = cfg.T * cfg.k
    g = torch.Generator().manual_seed(3)
    o = torch.randn((P, cfg.D), generator=g)
    osh = torch.randn((cfg.T, cfg.D), generator=g)
    inv = np.random.default_rng(4).permutation(P).astype(np.int32)
    inv[[0, 5, 17, P - 1]] = [-1, P, 1 << 30, -(1 << 30)]
    y = B.combine(cfg, o.cuda(), osh.cuda(), torch.from_numpy(inv).cuda())
    torch.cuda.synchronize()
    ref = oracle.combine(o.numpy().astype(np.float64), osh.numpy().astype(np.float64),
                         np.clip(inv, 0, P - 1), cfg.k)
    tol_check(y_host(y), ref, max_rel=4e-3, mean_rel=2e-3, what="y")


def gemm_case():
    cfg = MoEConfig("badgemm", T=37, D=256, E=24, I=192, Is=128, k=3)
    host = make_inputs(cfg, device="cpu")
    dev = host.to("cuda")
    ids, w = oracle_route(host)
    counts, offsets, perm, inv = oracle.permute(ids, cfg.E)
    return cfg, host, dev, ids, w, offsets, perm


def test_grouped_gemm_clamps_offsets():
    """Offsets below 0, above T*k and decreasing: no write outside the P
    output rows (guard rows keep their values), status MOE_ERR_INVALID_ARG."""
    cfg, host, dev, ids, w, offsets, perm = gemm_case()
    P = cfg.T * cfg.k
    bad = offsets.copy()
    bad[3] = -7
    bad[5] = P + 100
    bad[9] = bad[8] - 5
    bad[cfg.E] = P + 1
    tok = torch.from_numpy((perm // cfg.k).astype(np.int32)).cuda()
    xp = dev.x[tok.long()].contiguous()
    h = torch.full((P + GUARD, cfg.I), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = B.workspace(cfg, B.MOE_ENTRY_GROUPED_GEMM)
    B.grouped_gemm(cfg, B.MOE_OP_GATE_UP_SWIGLU, xp, torch.from_numpy(bad).cuda(), dev.w_gate_up,
                   h, ws=ws)
    torch.cuda.synchronize()
    assert B.get_status(ws) == B.MOE_ERR_INVALID_ARG
    assert (h[P:].float() == 7.0).all()
    # valid offsets on the same workspace: no error
    B.grouped_gemm(cfg, B.MOE_OP_GATE_UP_SWIGLU, xp, torch.from_numpy(offsets).cuda(),
                   dev.w_gate_up, h, ws=ws)
    torch.cuda.synchronize()
    assert B.get_status(ws) == B.MOE_OK


def test_grouped_gemm_clamps_pair_indices_and_row_indices():
    """Down: perm_pair entries outside [0, T*k) (the routing-weight lookup);
    gate/up: a_row_index entries outside [0, T) (the row gather)."""
    cfg, host, dev, ids, w, offsets, perm = gemm_case()
    P = cfg.T * cfg.k
    blob = torch.from_numpy(oracle.pack_blob(ids, w)).cuda()
    g = torch.Generator().manual_seed(6)
    h = (torch.randn((P, cfg.I), generator=g) * 0.5).to(torch.bfloat16).cuda()
    bad_perm = perm.copy()
    bad_perm[[1, 4, P - 2]] = [-3, P, 1 << 29]
    o = torch.full((P + GUARD, cfg.D), 5.0, dtype=torch.float32, device="cuda")
    ws = B.workspace(cfg, B.MOE_ENTRY_GROUPED_GEMM)
    B.grouped_gemm(cfg, B.MOE_OP_DOWN_WEIGHTED, h, torch.from_numpy(offsets).cuda(), dev.w_down,
                   o, perm_pair=torch.from_numpy(bad_perm).cuda(), blob=blob, ws=ws)
    torch.cuda.synchronize()
    assert B.get_status(ws) == B.MOE_ERR_INVALID_ARG
    assert (o[P:] == 5.0).all() and torch.isfinite(o[:P]).all()

    tok = (perm // cfg.k).astype(np.int32)
    tok[[0, 7]] = [-1, cfg.T + 2]
    hh = torch.empty((P, cfg.I), dtype=torch.bfloat16, device="cuda")
    B.grouped_gemm(cfg, B.MOE_OP_GATE_UP_SWIGLU, dev.x, torch.from_numpy(offsets).cuda(),
                   dev.w_gate_up, hh, a_row_index=torch.from_numpy(tok).cuda(), ws=ws)
    torch.cuda.synchronize()
    assert B.get_status(ws) == B.MOE_ERR_INVALID_ARG
    assert torch.isfinite(hh.float()).all()


def test_forward_experts_clamps_blob_ids():
    cfg = MoEConfig("badep", T=64, D=256, E=12, I=128, Is=128, k=3)
    host, bad, w, _ = bad_blob(cfg, 2)
    dev = host.to("cuda")
    blob = torch.from_numpy(oracle.pack_blob(bad, w)).cuda()
    ws = B.workspace(cfg, B.MOE_ENTRY_FORWARD_EXPERTS)
    y = B.forward_experts(cfg, dev.x, blob, dev, 0, cfg.E, 0, cfg.T, ws=ws)
    torch.cuda.synchronize()
    assert B.get_status(ws) == B.MOE_ERR_INVALID_ARG
    assert torch.isfinite(y).all()
