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


# Runs in a fresh process: the device memory comes from the driver API (no
# torch), first in the device's primary context, then in a second context
# created on the same device, then in the primary context again.  The fixed
# array has another address in each context; every call must use the one of
# the context current at the call.
_CONTEXTS_SCRIPT = r"""
import ctypes, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
from sparse_moe_layer_router_gb300 import binding as B

cu = ctypes.CDLL("libcuda.so.1")
def ck(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what} failed: {rc}")
V = ctypes.c_void_p
ck(cu.cuInit(0), "cuInit")
dev = ctypes.c_int()
ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
L = B.lib()
T, E, k, D = 2000, 40, 3, 128   # 6000 pairs: the chunked path that uses the fixed array
cfg = B.MoeConfig(T, D, E, 64, 64, k, 0, 128)
rng = np.random.default_rng(5)
ids = np.sort(np.argsort(rng.random((T, E)), axis=1)[:, :k], axis=1).astype(np.int32)
blob = np.empty((T, 2, k), np.int32)
blob[:, 0, :] = ids
blob[:, 1, :] = np.full((T, k), 1.0 / k, np.float32).view(np.int32)

def dalloc(nbytes):
    p = ctypes.c_uint64()
    ck(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(nbytes)), "cuMemAlloc")
    return p.value

def run():
    P = T * k
    d_blob = dalloc(blob.nbytes)
    ck(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(d_blob), blob.ctypes.data_as(V), ctypes.c_size_t(blob.nbytes)), "HtoD")
    sizes = [E, E + 1, P, P]
    outs = [[dalloc(4 * n) for n in sizes] for _ in range(2)]
    ws_n = L.moe_workspace_size(ctypes.byref(cfg), B.MOE_ENTRY_PERMUTE)
    ws = dalloc(ws_n)
    ck(cu.cuMemsetD8_v2(ctypes.c_uint64(ws), 0, ctypes.c_size_t(256)), "memset")
    a, b = outs
    ck(L.moe_permute(ctypes.byref(cfg), V(d_blob), V(a[0]), V(a[1]), V(a[2]), V(a[3]), None, None,
                     V(ws), ws_n, None), "moe_permute")
    ck(L.moe_permute_static(ctypes.byref(cfg), V(d_blob), V(b[0]), V(b[1]), V(b[2]), V(b[3]),
                            None, None, None), "moe_permute_static")
    ck(cu.cuCtxSynchronize(), "sync")
    res = []
    for bufs in outs:
        host = []
        for p, n in zip(bufs, sizes):
            h = np.empty(n, np.int32)
            ck(cu.cuMemcpyDtoH_v2(h.ctypes.data_as(V), ctypes.c_uint64(p), ctypes.c_size_t(4 * n)), "DtoH")
            host.append(h)
        res.append(host)
    for p in [d_blob, ws] + outs[0] + outs[1]:
        ck(cu.cuMemFree_v2(ctypes.c_uint64(p)), "cuMemFree")
    for x, y in zip(*res):
        assert np.array_equal(x, y)
    return res[1]

primary = V()
ck(cu.cuDevicePrimaryCtxRetain(ctypes.byref(primary), dev), "retain")
ck(cu.cuCtxSetCurrent(primary), "set primary")
r1 = run()
other = V()
ck(cu.cuCtxCreate_v2(ctypes.byref(other), 0, dev), "cuCtxCreate")   # now current
r2 = run()
ck(cu.cuCtxDestroy_v2(other), "cuCtxDestroy")
ck(cu.cuCtxSetCurrent(primary), "set primary again")
r3 = run()
for x, y, z in zip(r1, r2, r3):
    assert np.array_equal(x, y) and np.array_equal(x, z)
print("contexts ok")
"""


def test_static_permute_in_a_second_context_on_the_same_device():
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = subprocess.run([sys.executable, "-c", _CONTEXTS_SCRIPT, root], capture_output=True,
                         text=True, timeout=300)
    assert res.returncode == 0 and "contexts ok" in res.stdout, res.stdout + res.stderr
