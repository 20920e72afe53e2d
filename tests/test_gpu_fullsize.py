"""Parity at the full workload sizes, in the launch configuration bench.py times.

Every token's routing (ids bit-exact, weights within 1e-5) and the whole
dispatch grouping (bit-exact) are compared with the oracle.  Layer outputs are
compared on every token of the T=1024 workloads (prefill, W4A16 with group and
channel scales) and of the decode batch; on the T=8192 workloads, on a seeded
sample of tokens (first and last always included) plus, for the skewed one,
every token of the last (ragged) 256-row tile of the three hottest experts.
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_moe_layer_router_gb300 import binding as B
from sparse_moe_layer_router_gb300.build import build
from sparse_moe_layer_router_gb300.synthetic import CONFIGS, make_inputs

from helpers import WEIGHT_ABS, blob_parts, oracle_layer_rows, oracle_route, tol_check, y_host

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# tokens whose layer output is compared (None: all of them)
SAMPLE = {"decode": None, "prefill": None, "skewed": 24, "w4a16": None, "w4a16_decode": None,
          "dense_e64": 32, "w4a16_channel": None, "w4a16_dense_e64": 32}


def hot_tail_tokens(counts, offsets, perm, k, hottest=3, tile=256):
    """Tokens of the last token tile of each of the ``hottest`` largest experts."""
    rows = []
    for e in np.argsort(-counts, kind="stable")[:hottest]:
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        rows.extend(range(lo + (hi - lo - 1) // tile * tile, hi))
    return np.unique(perm[np.asarray(rows)] // k)


@pytest.fixture(scope="module", autouse=True)
def built(cuda_ok):
    build()
    B.lib()


@pytest.mark.parametrize("name", list(SAMPLE))
def test_full_size(name):
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, device="cuda")
    ws = B.workspace(cfg, B.MOE_ENTRY_FORWARD)
    y = B.forward(cfg, inp.x, inp, ws=ws)
    blob = B.route(cfg, inp.x, inp.w_router, inp.bias)
    counts, offsets, perm, inv = B.permute(cfg, blob)
    torch.cuda.synchronize()
    assert B.get_status(ws) == B.MOE_OK

    ids_ref, w_ref = oracle_route(inp)
    ids, w = blob_parts(blob)
    mism = np.argwhere(ids != ids_ref)
    assert mism.size == 0, f"{len(mism)} routing mismatches, first {mism[:3].tolist()}"
    assert np.abs(w - w_ref).max() <= WEIGHT_ABS
    c_ref, o_ref, p_ref, i_ref = oracle.permute(ids_ref, cfg.E)
    assert (counts.cpu().numpy() == c_ref).all()
    assert (offsets.cpu().numpy() == o_ref).all()
    assert (perm.cpu().numpy() == p_ref).all()
    assert (inv.cpu().numpy() == i_ref).all()
    if name == "skewed":
        empty = (c_ref == 0).mean()
        assert 0.15 <= empty <= 0.25, empty  # the workload's "~20% of experts get no token"

    n = SAMPLE[name]
    if n is None:
        rows = np.arange(cfg.T)
    else:
        rng = np.random.default_rng(2024)
        rows = np.unique(np.concatenate([[0, cfg.T - 1],
                                         rng.choice(cfg.T, size=min(n, cfg.T), replace=False)]))
        if name == "skewed":
            tail = hot_tail_tokens(c_ref, o_ref, p_ref, cfg.k)
            assert tail.size > 0
            rows = np.union1d(rows, tail)
    ref = oracle_layer_rows(inp, rows, ids_ref, w_ref)
    tol_check(y_host(y)[rows], ref, what=f"{name} y[{rows.size} tokens]")
