"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Routing ids, counts, offsets and permutations must match bit for bit; blob
weights within 1e-5; layer outputs within max|err| <= 2e-2 max|ref| and
sum|err| / sum|ref| <= 5e-3.  Inputs come from the seeded generator; expected
values come only from the oracle, computed on host copies of the same inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_moe_layer_router_gb300 import binding as B
from sparse_moe_layer_router_gb300.build import build
from sparse_moe_layer_router_gb300.synthetic import (CONFIGS, MoEConfig, as_u16, make_inputs,
                                                     normal_bf16)

from helpers import (WEIGHT_ABS, blob_parts, expert_host, oracle_layer_rows, oracle_route,
                     tol_check, y_host)

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": CONFIGS["tiny"],
    # the largest k the entry points accept (32 experts per token)
    "k32": MoEConfig("k32", T=40, D=256, E=48, I=64, Is=64, k=32),
    # several tiles in every direction with a ragged tail
    "ragged": MoEConfig("ragged", T=37, D=256, E=24, I=192, Is=128, k=3),
    # k = E: every token uses every expert
    "all_experts": MoEConfig("all_experts", T=50, D=128, E=4, I=64, Is=64, k=4),
    "one_token": MoEConfig("one_token", T=1, D=384, E=32, I=128, Is=64, k=5),
    # hot experts (> 64 rows: several token tiles) and a 200-row shared group
    "hot": MoEConfig("hot", T=200, D=256, E=16, I=128, Is=128, k=2, zipf_s=1.2, zipf_alpha=3.0),
    # the 256-row token tile variant
    "wide": MoEConfig("wide", T=2100, D=256, E=8, I=64, Is=64, k=2),
    # top-1 routing (weight 1), and a single routed expert
    "top1": MoEConfig("top1", T=50, D=256, E=8, I=128, Is=128, k=1),
    "single_expert": MoEConfig("single_expert", T=20, D=128, E=1, I=64, Is=64, k=1),
    # T >= 2048 with a Zipf bias: 15 experts of >= 64 rows and 42 smaller ones, so
    # the split bf16 launch runs both its hot and its cold grid
    "split": MoEConfig("split", T=2100, D=256, E=64, I=64, Is=64, k=4, zipf_s=1.2,
                       zipf_alpha=0.3),
}

# W4A16: symmetric int4 weights, group 128 along K, bf16 scales
W4 = {
    "w4_tiny": MoEConfig("w4_tiny", T=64, D=256, E=16, I=256, Is=256, k=2, quant=1),
    "w4_ragged": MoEConfig("w4_ragged", T=37, D=512, E=24, I=768, Is=256, k=3, quant=1),
    "w4_hot": MoEConfig("w4_hot", T=200, D=256, E=16, I=256, Is=512, k=2, quant=1, zipf_s=1.2,
                        zipf_alpha=3.0),
    "w4_wide": MoEConfig("w4_wide", T=2100, D=256, E=8, I=256, Is=256, k=2, quant=1),
    # K = 1024 / 2048: exercises the TMA scale tables (K multiple of 1024)
    "w4_table": MoEConfig("w4_table", T=96, D=2048, E=12, I=1024, Is=1024, k=3, quant=1),
    # channel-wise scales (group 0): 64-row kernel (TMEM restore) and 256-row kernel
    "w4c_ragged": MoEConfig("w4c_ragged", T=37, D=512, E=24, I=768, Is=256, k=3, quant=1,
                            group=0),
    "w4c_table": MoEConfig("w4c_table", T=96, D=2048, E=12, I=1024, Is=1024, k=3, quant=1,
                           group=0),
    "w4c_wide": MoEConfig("w4c_wide", T=2100, D=256, E=8, I=256, Is=256, k=2, quant=1,
                          group=0),
}


@pytest.fixture(scope="module", autouse=True)
def built(cuda_ok):
    build()
    B.lib()


def gpu_inputs(cfg):
    host = make_inputs(cfg, device="cpu")
    return host, host.to("cuda")


def check_route(cfg, host, dev, expect_refine=None):
    ws = B.workspace(cfg, B.MOE_ENTRY_ROUTE)
    blob = B.route(cfg, dev.x, dev.w_router, dev.bias, ws=ws)
    torch.cuda.synchronize()
    ids, w = blob_parts(blob)
    ids_ref, w_ref = oracle_route(host)
    mism = np.argwhere(ids != ids_ref)
    assert mism.size == 0, f"{len(mism)} id mismatches, first at {mism[:3].tolist()}"
    np.testing.assert_allclose(w, w_ref, rtol=0, atol=WEIGHT_ABS)
    refined = int(ws[4:8].view(torch.int32).item())
    if expect_refine is not None:
        assert (refined > 0) == expect_refine, refined
    return blob, ids_ref, w_ref, refined


@pytest.mark.parametrize("name", list(SMALL))
def test_route_bit_exact(name):
    cfg = SMALL[name]
    host, dev = gpu_inputs(cfg)
    check_route(cfg, host, dev)


def test_route_zero_router_ties_go_to_lower_index():
    cfg = SMALL["ragged"]
    host, dev = gpu_inputs(cfg)
    host.w_router.zero_()
    dev.w_router.zero_()
    blob, ids_ref, w_ref, _ = check_route(cfg, host, dev)
    assert (ids_ref == np.arange(cfg.k)).all()


def test_route_near_ties_refined_exactly():
    """Router rows that differ in one element by one bf16 step: fp32 cannot
    certify the boundary, so the fp64 re-decision must reproduce the oracle."""
    cfg = MoEConfig("near_tie", T=64, D=512, E=64, I=64, Is=64, k=6)
    host, dev = gpu_inputs(cfg)
    base = host.w_router[0].clone()
    wr = base.repeat(cfg.E, 1)
    for e in range(cfg.E):
        d = (7 * e) % cfg.D
        wr[e, d] = torch.nextafter(base[d].float(), torch.tensor(float("inf"))).to(torch.bfloat16) \
            if e % 2 else base[d]
    wr[5] = wr[3]  # an exact duplicate: exact tie decided by index
    host.w_router.copy_(wr)
    dev.w_router.copy_(wr.cuda())
    _, _, _, refined = check_route(cfg, host, dev, expect_refine=True)
    assert refined > 0


def _route_poisoned(cfg, dev):
    """moe_route into a blob filled with -1 first: every entry must be written."""
    blob = torch.full((cfg.T, 2, cfg.k), -1, dtype=torch.int32, device="cuda")
    ws = B.workspace(cfg, B.MOE_ENTRY_ROUTE)
    B.route(cfg, dev.x, dev.w_router, dev.bias, blob=blob, ws=ws)
    torch.cuda.synchronize()
    assert B.get_status(ws) == B.MOE_OK
    return blob_parts(blob)


@pytest.mark.parametrize("T", [80, 600])
def test_route_nan_logits_rank_last(T):
    """NaN router rows and NaN token rows (reading R21): a NaN logit ranks below
    every number.  ids bit-exact with the oracle (k distinct ids in [0, E) for
    every token, all written), weights NaN exactly where the oracle's are,
    the others within the weight tolerance.  T = 600 runs the warp-per-token
    select kernel."""
    cfg = MoEConfig(f"nan{T}", T=T, D=256, E=40, I=64, Is=64, k=4)
    host = make_inputs(cfg, device="cpu")
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
    host.w_router[7, 11] = nan
    host.w_router[30, 0] = nan
    host.x[5, 3] = nan
    host.x[T - 17, 200] = nan
    dev = host.to("cuda")
    ids, w = _route_poisoned(cfg, dev)
    ids_ref, w_ref = oracle_route(host)
    assert np.array_equal(ids, ids_ref)
    assert ((ids >= 0) & (ids < cfg.E)).all() and (np.diff(ids, axis=1) > 0).all()
    assert np.array_equal(np.isnan(w), np.isnan(w_ref))
    np.testing.assert_allclose(w, w_ref, rtol=0, atol=WEIGHT_ABS)
    assert ids[5].tolist() == [0, 1, 2, 3] and np.isnan(w[5]).all()
    assert not np.isin(ids[[t for t in range(T) if t not in (5, T - 17)]], [7, 30]).any()


def test_route_fewer_finite_logits_than_k():
    """A NaN bias on all but three of twelve experts with k = 5: each token gets
    the three finite experts and the two lowest-index NaN experts (reading R21),
    NaN weights, as the oracle."""
    cfg = MoEConfig("nan_bias", T=70, D=256, E=12, I=64, Is=64, k=5)
    host = make_inputs(cfg, device="cpu")
    bias = torch.full((cfg.E,), float("nan"), dtype=torch.float32)
    bias[[2, 6, 11]] = torch.tensor([0.5, -0.25, 0.0])
    host.bias = bias
    dev = host.to("cuda")
    ids, w = _route_poisoned(cfg, dev)
    ids_ref, w_ref = oracle_route(host)
    assert np.array_equal(ids, ids_ref)
    assert (ids == np.array([0, 1, 2, 6, 11], np.int32)).all()
    assert np.isnan(w).all() and np.isnan(w_ref).all()


def test_forward_nan_token_row_stays_in_its_row():
    """A NaN in one token row: that token's output row is NaN, every other row
    matches the oracle (the NaN travels in its own GEMM column only)."""
    cfg = SMALL["ragged"]
    host = make_inputs(cfg, device="cpu")
    host.x[3, 17] = torch.tensor(float("nan"), dtype=torch.bfloat16)
    dev = host.to("cuda")
    ws = B.workspace(cfg, B.MOE_ENTRY_FORWARD)
    y = B.forward(cfg, dev.x, dev, ws=ws)
    torch.cuda.synchronize()
    assert B.get_status(ws) == B.MOE_OK
    yh = y_host(y)
    assert np.isnan(yh[3]).all()
    ids, w = oracle_route(host)
    rows = np.array([t for t in range(cfg.T) if t != 3])
    tol_check(yh[rows], oracle_layer_rows(host, rows, ids, w), what="rows without the NaN")


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)


def test_router_logits_tensor_core_error_bound():
    """The level-1 logits come from tensor-core MMAs whose fp32 accumulation is not
    documented; routing certification assumes an error of at most 2^-15 sum|x w| per
    64-wide K chunk.  Check the measured error against a bound twice as tight, on
    plain inputs, on inputs whose magnitudes span 2^-12..2^12 within a row, and on
    rows built to cancel (large equal-and-opposite products next to small ones)."""
    T, D, E = 192, 1024, 256
    cfg = MoEConfig("rl", T=T, D=D, E=E, I=64, Is=64, k=4)
    rng = np.random.default_rng(7)
    cases = []
    x = rng.standard_normal((T, D)); w = rng.standard_normal((E, D)) * 0.02
    cases.append((x, w))
    xs = rng.standard_normal((T, D)) * 2.0 ** rng.integers(-12, 13, size=(T, D))
    ws_ = rng.standard_normal((E, D)) * 2.0 ** rng.integers(-12, 13, size=(E, D))
    cases.append((xs, ws_))
    xc = np.repeat(rng.standard_normal((T, D // 2)) * 64.0, 2, axis=1)
    wc = np.empty((E, D))
    big = rng.standard_normal((E, D // 2)) * 64.0
    wc[:, 0::2] = big
    wc[:, 1::2] = -big + rng.standard_normal((E, D // 2)) * 2.0 ** -6
    cases.append((xc, wc))
    worst = 0.0
    for xa, wa in cases:
        xb, wb = _bf16(xa), _bf16(wa)
        z = B.router_logits(cfg, xb.cuda(), wb.cuda()).cpu().double().numpy()
        ref = oracle.router_logits(as_u16(xb), as_u16(wb))
        a = np.abs(xb.double().numpy()) @ np.abs(wb.double().numpy()).T
        bound = (2.0 ** -16 + (D / 64 + 2) * 2.0 ** -24) * a
        err = np.abs(z - ref)
        assert (err <= bound + 1e-30).all(), float((err / np.maximum(a, 1e-300)).max())
        worst = max(worst, float((err / np.maximum(a, 1e-300)).max()))
    print(f"worst |z - exact| / sum|x w| = {worst:.3e} (certification assumes 3.1e-05)")


@pytest.mark.parametrize("T,E,k", [(100, 1000, 8), (2100, 1024, 8), (2100, 33, 3), (70, 64, 32),
                                   (600, 1024, 32)])
def test_route_bit_exact_wide_and_long(T, E, k):
    """Many experts (up to 1024: 32 logits per lane in the select kernels), batches
    of 512 tokens or more (the warp-per-token select), a ragged expert count, and
    the largest k the entry points accept (32)."""
    cfg = MoEConfig(f"r{T}x{E}", T=T, D=256, E=E, I=64, Is=64, k=k)
    host, dev = gpu_inputs(cfg)
    check_route(cfg, host, dev)


def test_route_with_bias():
    cfg = SMALL["hot"]
    host, dev = gpu_inputs(cfg)
    assert host.bias is not None
    check_route(cfg, host, dev)


@pytest.mark.parametrize("name", ["tiny", "ragged", "hot", "wide"])
def test_permute_bit_exact(name):
    cfg = SMALL[name]
    host, _ = gpu_inputs(cfg)
    ids, w = oracle_route(host)
    blob = torch.from_numpy(oracle.pack_blob(ids, w)).cuda()
    counts, offsets, perm, inv = B.permute(cfg, blob)
    c_ref, o_ref, p_ref, i_ref = oracle.permute(ids, cfg.E)
    assert (counts.cpu().numpy() == c_ref).all()
    assert (offsets.cpu().numpy() == o_ref).all()
    assert (perm.cpu().numpy() == p_ref).all()
    assert (inv.cpu().numpy() == i_ref).all()


def test_permute_random_ids_properties_large():
    """Random distinct ids per token at a size spanning many permute chunks."""
    T, E, k = 5000, 300, 7
    rng = np.random.default_rng(11)
    ids = np.sort(np.argsort(rng.random((T, E)), axis=1)[:, :k], axis=1).astype(np.int32)
    cfg = MoEConfig("perm", T=T, D=128, E=E, I=64, Is=64, k=k)
    blob = torch.from_numpy(oracle.pack_blob(ids, np.full((T, k), 1.0 / k))).cuda()
    counts, offsets, perm, inv = B.permute(cfg, blob)
    c_ref, o_ref, p_ref, i_ref = oracle.permute(ids, E)
    assert (counts.cpu().numpy() == c_ref).all()
    assert (offsets.cpu().numpy() == o_ref).all()
    assert (perm.cpu().numpy() == p_ref).all()
    assert (inv.cpu().numpy() == i_ref).all()


def grouped_setup(cfg):
    host, dev = gpu_inputs(cfg)
    ids, w = oracle_route(host)
    counts, offsets, perm, inv = oracle.permute(ids, cfg.E)
    blob = oracle.pack_blob(ids, w)
    return host, dev, ids, w, offsets, perm, inv, blob


@pytest.mark.parametrize("name", ["tiny", "ragged", "hot", "wide", "one_token"])
def test_grouped_gate_up_swiglu(name):
    cfg = SMALL[name]
    host, dev, ids, w, offsets, perm, inv, blob = grouped_setup(cfg)
    P = cfg.T * cfg.k
    tok = perm // cfg.k
    h = torch.empty((P, cfg.I), dtype=torch.bfloat16, device="cuda")
    hs = torch.empty((cfg.T, cfg.Is), dtype=torch.bfloat16, device="cuda")
    B.grouped_gemm(cfg, B.MOE_OP_GATE_UP_SWIGLU, dev.x, torch.from_numpy(offsets).cuda(),
                   dev.w_gate_up, h, a_row_index=torch.from_numpy(tok.astype(np.int32)).cuda(),
                   a_shared=dev.x, w_shared=dev.ws_gate_up, out_shared=hs)
    torch.cuda.synchronize()
    xh = as_u16(host.x)
    ref = np.empty((P, cfg.I))
    for e in range(cfg.E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            ref[r0:r1] = oracle.expert_hidden(xh[tok[r0:r1]], as_u16(host.w_gate_up[e]))
    tol_check(y_host(h), ref, what="h")
    ref_s = oracle.expert_hidden(xh, as_u16(host.ws_gate_up))
    tol_check(y_host(hs), ref_s, what="h_shared")


@pytest.mark.parametrize("name", ["tiny", "ragged", "hot", "wide"])
def test_grouped_down_weighted(name):
    cfg = SMALL[name]
    host, dev, ids, w, offsets, perm, inv, blob = grouped_setup(cfg)
    P = cfg.T * cfg.k
    h = normal_bf16((P, cfg.I), 0.5, 3, 77)
    hs = normal_bf16((cfg.T, cfg.Is), 0.5, 3, 78)
    o = torch.empty((P, cfg.D), dtype=torch.float32, device="cuda")
    os_ = torch.empty((cfg.T, cfg.D), dtype=torch.float32, device="cuda")
    B.grouped_gemm(cfg, B.MOE_OP_DOWN_WEIGHTED, h.cuda(), torch.from_numpy(offsets).cuda(),
                   dev.w_down, o, perm_pair=torch.from_numpy(perm).cuda(),
                   blob=torch.from_numpy(blob).cuda(), a_shared=hs.cuda(), w_shared=dev.ws_down,
                   out_shared=os_)
    torch.cuda.synchronize()
    hf = h.float().numpy().astype(np.float64)
    wrow = blob[:, 1, :].view(np.float32).reshape(-1)[perm].astype(np.float64)
    ref = np.empty((P, cfg.D))
    for e in range(cfg.E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            ref[r0:r1] = oracle.expert_down(hf[r0:r1], as_u16(host.w_down[e])) * wrow[r0:r1, None]
    tol_check(o.cpu().numpy(), ref, max_rel=1e-4, mean_rel=1e-5, what="o")
    ref_s = oracle.expert_down(hs.float().numpy().astype(np.float64), as_u16(host.ws_down))
    tol_check(os_.cpu().numpy(), ref_s, max_rel=1e-4, mean_rel=1e-5, what="o_shared")


def test_combine():
    cfg = SMALL["ragged"]
    host, dev, ids, w, offsets, perm, inv, blob = grouped_setup(cfg)
    P = cfg.T * cfg.k
    g = torch.Generator().manual_seed(5)
    o = torch.randn((P, cfg.D), generator=g)
    osh = torch.randn((cfg.T, cfg.D), generator=g)
    y = B.combine(cfg, o.cuda(), osh.cuda(), torch.from_numpy(inv).cuda())
    ref = oracle.combine(o.numpy().astype(np.float64), osh.numpy().astype(np.float64), inv, cfg.k)
    tol_check(y_host(y), ref, max_rel=4e-3, mean_rel=2e-3, what="y")
    y0 = B.combine(cfg, o.cuda(), None, torch.from_numpy(inv).cuda())
    ref0 = oracle.combine(o.numpy().astype(np.float64), None, inv, cfg.k)
    tol_check(y_host(y0), ref0, max_rel=4e-3, mean_rel=2e-3, what="y (no shared)")


@pytest.mark.parametrize("name", list(SMALL))
def test_forward_parity(name):
    cfg = SMALL[name]
    host, dev = gpu_inputs(cfg)
    ws = B.workspace(cfg, B.MOE_ENTRY_FORWARD)
    y = B.forward(cfg, dev.x, dev, ws=ws)
    assert B.get_status(ws) == B.MOE_OK
    ids, w = oracle_route(host)
    ref = oracle_layer_rows(host, np.arange(cfg.T), ids, w)
    tol_check(y_host(y), ref)


# T >= 4096: moe_forward_host copies and routes x in 2048-token chunks (the
# last one 104 tokens, routed by the block-per-token select kernel).
HOST_CHUNKS = MoEConfig("host_chunks", T=4200, D=256, E=32, I=64, Is=64, k=2)


@pytest.mark.parametrize("name,pinned", [("hot", True), ("wide", True), ("wide", False),
                                         ("split", True), ("host_chunks", True),
                                         ("host_chunks", False), ("w4_ragged", True),
                                         ("w4c_wide", True)])
def test_forward_deterministic_and_host_entry(name, pinned):
    """Two calls give the same bits, and moe_forward_host (host x and y, the
    copies inside the call) gives the device entry's bits, bf16 and W4A16.
    "wide" and "split" (T = 2100) take the chunked combine whose copies to the
    host overlap it (eight chunks, the last one shorter); "host_chunks" also
    routes x chunk by chunk as it arrives; pinned and pageable host buffers."""
    cfg = HOST_CHUNKS if name == "host_chunks" else SMALL[name] if name in SMALL else W4[name]
    host, dev = gpu_inputs(cfg)
    ws = B.workspace(cfg, B.MOE_ENTRY_FORWARD)
    y1 = B.forward(cfg, dev.x, dev, ws=ws).clone()
    y2 = B.forward(cfg, dev.x, dev, ws=ws).clone()
    assert torch.equal(y1, y2)
    wsh = B.workspace(cfg, B.MOE_ENTRY_FORWARD_HOST)
    xh = host.x.clone()
    yh = torch.full((cfg.T, cfg.D), 5.0, dtype=torch.bfloat16)
    if pinned:
        xh, yh = xh.pin_memory(), yh.pin_memory()
    for _ in range(2):
        B.forward_host(cfg, xh, dev, yh, wsh)
        torch.cuda.synchronize()
        assert torch.equal(yh, y1.cpu())
        yh.fill_(5.0)
    assert B.get_status(wsh) == B.MOE_OK


@pytest.mark.parametrize("name", list(W4))
def test_forward_parity_w4a16(name):
    cfg = W4[name]
    host, dev = gpu_inputs(cfg)
    ws = B.workspace(cfg, B.MOE_ENTRY_FORWARD)
    y = B.forward(cfg, dev.x, dev, ws=ws)
    assert B.get_status(ws) == B.MOE_OK
    ids, w = oracle_route(host)
    ref = oracle_layer_rows(host, np.arange(cfg.T), ids, w)
    tol_check(y_host(y), ref)


@pytest.mark.parametrize("name", ["w4_tiny", "w4_ragged", "w4_wide", "w4_table", "w4c_ragged",
                                  "w4c_wide"])
def test_grouped_gate_up_w4a16(name):
    cfg = W4[name]
    host, dev, ids, w, offsets, perm, inv, blob = grouped_setup(cfg)
    P = cfg.T * cfg.k
    tok = perm // cfg.k
    h = torch.empty((P, cfg.I), dtype=torch.bfloat16, device="cuda")
    hs = torch.empty((cfg.T, cfg.Is), dtype=torch.bfloat16, device="cuda")
    B.grouped_gemm(cfg, B.MOE_OP_GATE_UP_SWIGLU, dev.x, torch.from_numpy(offsets).cuda(),
                   dev.w_gate_up, h, a_row_index=torch.from_numpy(tok.astype(np.int32)).cuda(),
                   w_scales=dev.s_gate_up, a_shared=dev.x, w_shared=dev.ws_gate_up,
                   ws_scales=dev.ss_gate_up, out_shared=hs)
    torch.cuda.synchronize()
    xh = as_u16(host.x)
    ref = np.empty((P, cfg.I))
    for e in range(cfg.E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            ref[r0:r1] = oracle.expert_hidden(xh[tok[r0:r1]], host.w_gate_up[e].numpy(),
                                              as_u16(host.s_gate_up[e]), group=cfg.group)
    tol_check(y_host(h), ref, what="h")
    ref_s = oracle.expert_hidden(xh, host.ws_gate_up.numpy(), as_u16(host.ss_gate_up),
                                 group=cfg.group)
    tol_check(y_host(hs), ref_s, what="h_shared")


@pytest.mark.parametrize("name", ["w4_tiny", "w4_ragged", "w4_wide", "w4_table", "w4c_ragged",
                                  "w4c_wide"])
def test_grouped_down_w4a16(name):
    cfg = W4[name]
    host, dev, ids, w, offsets, perm, inv, blob = grouped_setup(cfg)
    P = cfg.T * cfg.k
    h = normal_bf16((P, cfg.I), 0.5, 3, 77)
    hs = normal_bf16((cfg.T, cfg.Is), 0.5, 3, 78)
    o = torch.empty((P, cfg.D), dtype=torch.float32, device="cuda")
    os_ = torch.empty((cfg.T, cfg.D), dtype=torch.float32, device="cuda")
    B.grouped_gemm(cfg, B.MOE_OP_DOWN_WEIGHTED, h.cuda(), torch.from_numpy(offsets).cuda(),
                   dev.w_down, o, w_scales=dev.s_down, perm_pair=torch.from_numpy(perm).cuda(),
                   blob=torch.from_numpy(blob).cuda(), a_shared=hs.cuda(), w_shared=dev.ws_down,
                   ws_scales=dev.ss_down, out_shared=os_)
    torch.cuda.synchronize()
    hf = h.float().numpy().astype(np.float64)
    wrow = blob[:, 1, :].view(np.float32).reshape(-1)[perm].astype(np.float64)
    ref = np.empty((P, cfg.D))
    for e in range(cfg.E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            ref[r0:r1] = oracle.expert_down(hf[r0:r1], host.w_down[e].numpy(),
                                            as_u16(host.s_down[e]), group=cfg.group) * \
                wrow[r0:r1, None]
    # dequantised weights are rounded once to bf16 on the GPU: relative error 2^-9 per weight
    tol_check(o.cpu().numpy(), ref, max_rel=1e-2, mean_rel=2e-3, what="o")
    ref_s = oracle.expert_down(hs.float().numpy().astype(np.float64), host.ws_down.numpy(),
                               as_u16(host.ss_down), group=cfg.group)
    tol_check(os_.cpu().numpy(), ref_s, max_rel=1e-2, mean_rel=2e-3, what="o_shared")


def test_bounded_wait_times_out_and_context_survives():
    """A device wait that nothing completes gives up after its limit, reports
    MOE_ERR_TIMEOUT through the workspace status word, and the context keeps
    working (a forward afterwards still matches the oracle)."""
    import time
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.time()
    status = B.selftest_wait_timeout(ws, limit_ms=200)
    dt = time.time() - t0
    assert status == B.MOE_ERR_TIMEOUT
    assert 0.15 <= dt < 5.0, dt
    assert B.get_status(ws) == B.MOE_OK  # read-and-clear
    test_forward_parity("tiny")


def test_status_is_sticky_until_read():
    """An error recorded on a workspace survives later successful calls that use
    the same workspace, and is cleared only by reading it (moe_get_status)."""
    cfg = CONFIGS["tiny"]
    host, dev = gpu_inputs(cfg)
    ws = B.workspace(cfg, B.MOE_ENTRY_FORWARD)
    assert B.selftest_wait_timeout(ws, limit_ms=50, read_status=False) is None
    y = B.forward(cfg, dev.x, dev, ws=ws)          # a later call on the same workspace
    B.route(cfg, dev.x, dev.w_router, ws=ws)       # and a route call
    torch.cuda.synchronize()
    assert B.get_status(ws) == B.MOE_ERR_TIMEOUT   # still reported
    assert B.get_status(ws) == B.MOE_OK            # cleared by the read
    ids_ref, w_ref = oracle_route(host)
    tol_check(y_host(y), oracle_layer_rows(host, np.arange(cfg.T), ids_ref, w_ref))


@pytest.mark.parametrize("layout", ["sequential", "offset8"])
@pytest.mark.parametrize("in_place", [False, True])
def test_repack_int4_sequential_to_pair_order(layout, in_place):
    """Sequential-order words (value j in bits 4j..4j+3), packed here from that
    definition, come out in the order the oracle reads: its exact dequantisation
    with unit scales returns the original values.  1517 words: a ragged tail."""
    rng = np.random.default_rng(11)
    R, C = 37, 8 * 41
    q = rng.integers(-8, 8, size=(R, C))
    nib = ((q + 8) if layout == "offset8" else q) & 15
    words = np.zeros((R, C // 8), np.uint64)
    for j in range(8):
        words |= nib[:, j::8].astype(np.uint64) << np.uint64(4 * j)
    src = torch.from_numpy(words.astype(np.uint32).view(np.int32)).cuda()
    code = B.MOE_INT4_SEQUENTIAL_OFFSET8 if layout == "offset8" else B.MOE_INT4_SEQUENTIAL
    dst = B.repack_int4(src, dst=src if in_place else None, layout=code)
    torch.cuda.synchronize()
    unit = np.full(R, 0x3F80, np.uint16)  # bf16 1.0, one scale per row
    got = oracle.dequant_w4(dst.cpu().numpy(), unit, 0)
    assert np.array_equal(got, q.astype(np.float64))


@pytest.mark.parametrize("sx,sw", [(-70, -70), (-64, -64), (-70, 0), (0, -130)])
def test_route_bit_exact_at_tiny_magnitudes(sx, sw):
    """Token and router rows scaled by 2^sx and 2^sw, so that the products
    x_d * w_d (about 2^(sx+sw)) fall below the fp32 normal range (2^-126) where
    fp32 products and the tensor core's partial sums are no longer exact or may
    be flushed.  The decision must still be the fp64 definition's, bit for bit."""
    cfg = MoEConfig("tiny_mag", T=64, D=256, E=16, I=64, Is=64, k=2)
    host = make_inputs(cfg, device="cpu")
    host.x = (host.x.float() * 2.0 ** sx).to(torch.bfloat16)
    host.w_router = (host.w_router.float() * 2.0 ** sw).to(torch.bfloat16)
    dev = host.to("cuda")
    check_route(cfg, host, dev)


@pytest.mark.parametrize("name", ["hot", "wide", "split", "w4_table", "w4c_wide"])
def test_forward_replays_from_a_cuda_graph(name):
    """moe_forward captured once into a CUDA graph (its launches chained with
    programmatic dependent launch on the caller's stream) and replayed
    on new token rows copied into the captured input buffer: every replay
    equals an eager call on the same rows bit for bit.  "wide" takes the
    three-kernel dispatch and the 256-row tiles, "split" the two grids on two
    streams (forked from and joined to the captured stream); the W4A16 cases
    the TMEM- and shared-memory-restore kernels."""
    cfg = SMALL[name] if name in SMALL else W4[name]
    host, dev = gpu_inputs(cfg)
    W = B.weights_struct(dev, cfg)
    x_in = dev.x.clone()
    y = torch.empty((cfg.T, cfg.D), dtype=torch.bfloat16, device="cuda")
    ws = B.workspace(cfg, B.MOE_ENTRY_FORWARD)
    B.forward(cfg, x_in, W, y=y, ws=ws)  # first call outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        B.forward(cfg, x_in, W, y=y, ws=ws)
    ws_eager = B.workspace(cfg, B.MOE_ENTRY_FORWARD)
    for seed in (11, 12, 13):
        x_new = normal_bf16((cfg.T, cfg.D), 1.0, seed, 77, "cpu").cuda()
        x_in.copy_(x_new)
        graph.replay()
        y_eager = B.forward(cfg, x_new, W, ws=ws_eager)
        torch.cuda.synchronize()
        assert torch.equal(y, y_eager), seed
    assert B.get_status(ws) == B.MOE_OK and B.get_status(ws_eager) == B.MOE_OK
