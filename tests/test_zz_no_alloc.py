"""moe_permute_static: the dispatch grouping for callers that cannot allocate.

Some callers of this library cannot call cudaMalloc or pass a workspace (a
plug-in that only holds the tensors it was handed, an engine whose device memory
belongs to an allocator it cannot reach, a serving loop that must not allocate
while it runs).  moe_permute_static serves them: its scratch is a fixed array
inside the library.  These tests call it through the C ABI and require the same
counts, offsets, permutation and gathered rows as moe_permute (integer and byte
results, so bit for bit) on two calls in a row with different routings, and a
clean refusal of problems larger than the fixed scratch.

This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from sparse_moe_layer_router_gb300 import binding as B
from sparse_moe_layer_router_gb300.build import build
from sparse_moe_layer_router_gb300.synthetic import MoEConfig, normal_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built(cuda_ok):
    build()
    B.lib()


def make_blob(T, E, k, seed):
    rng = np.random.default_rng(seed)
    ids = np.sort(np.argsort(rng.random((T, E)), axis=1)[:, :k], axis=1).astype(np.int32)
    blob = np.empty((T, 2, k), np.int32)
    blob[:, 0, :] = ids
    blob[:, 1, :] = np.full((T, k), 1.0 / k, np.float32).view(np.int32)
    return torch.from_numpy(blob).cuda()


def test_static_permute_matches_workspace_permute_on_two_calls():
    cfg = MoEConfig("static", T=5000, D=256, E=300, I=64, Is=64, k=7)  # 18 chunks of pairs
    x = normal_bf16((cfg.T, cfg.D), 1.0, 0, 91).cuda()
    for call, seed in enumerate((1, 2)):
        blob = make_blob(cfg.T, cfg.E, cfg.k, seed)
        xp_ref = torch.empty((cfg.T * cfg.k, cfg.D), dtype=torch.bfloat16, device="cuda")
        ref = B.permute(cfg, blob, x=x, x_perm=xp_ref)
        xp = torch.full((cfg.T * cfg.k, cfg.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        got = B.permute_static(cfg, blob, x=x, x_perm=xp)
        torch.cuda.synchronize()
        for name, a, b in zip(("counts", "offsets", "perm_pair", "inv_row"), got, ref):
            assert torch.equal(a, b), f"call {call}: {name} differs"
        assert torch.equal(xp.view(torch.int16), xp_ref.view(torch.int16)), f"call {call}: x_perm"


def test_static_permute_without_gather():
    cfg = MoEConfig("static_small", T=37, D=128, E=24, I=64, Is=64, k=3)
    blob = make_blob(cfg.T, cfg.E, cfg.k, 3)
    ref = B.permute(cfg, blob)
    got = B.permute_static(cfg, blob)
    torch.cuda.synchronize()
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


def test_static_permute_refuses_problems_beyond_its_scratch():
    cfg = MoEConfig("too_big", T=16384, D=128, E=1024, I=64, Is=64, k=10)  # 80 chunks x 1024
    d = ctypes.c_void_p(4096)
    rc = B.lib().moe_permute_static(ctypes.byref(B.config(cfg)), d, d, d, d, d, None, None, None)
    assert rc == B.MOE_ERR_SCRATCH_LIMIT
    assert "scratch" in B.strerror(rc)
