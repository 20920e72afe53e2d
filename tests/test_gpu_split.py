"""The hot/cold split of a bf16 grouped GEMM with 256-row token tiles (taken
below 512 rows per expert on average): groups of at least 64 rows run in one
grid, the smaller ones in a second grid on a second stream.  Row counts on
both sides of the 64-row boundary, every group on one side (one grid then
has no work), with and without the shared group, and a first split call made
by a fresh host thread inside a stream capture.  Outputs are checked against
the oracle's expert functions row by row."""
import threading

import numpy as np
import pytest
import torch

import oracle
from sparse_moe_layer_router_gb300 import binding as B
from sparse_moe_layer_router_gb300.build import build
from sparse_moe_layer_router_gb300.synthetic import MoEConfig, as_u16, make_inputs

from helpers import tol_check, y_host

pytestmark = pytest.mark.gpu

# T >= 2048 (256-row tiles) and T*k = 8400 < 512*E: the split is taken.
CFG = MoEConfig("split_abi", T=2100, D=256, E=64, I=64, Is=64, k=4)
P = CFG.T * CFG.k
LAYOUTS = ["boundary", "all_cold", "all_hot", "one_hot"]


@pytest.fixture(scope="module", autouse=True)
def built(cuda_ok):
    build()
    B.lib()


@pytest.fixture(scope="module")
def inputs():
    host = make_inputs(CFG, device="cpu")
    return host, host.to("cuda")


def row_counts(layout, rng):
    """Rows per expert (sum <= T*k) for one layout of the 64-row boundary."""
    E = CFG.E
    if layout == "boundary":
        c = np.zeros(E, np.int64)
        edge = [63, 64, 65, 1, 0, 127, 128, 129, 255, 256, 257, 16, 17, 48, 62, 66]
        c[: len(edge)] = edge
        c[len(edge):] = rng.integers(0, 140, E - len(edge))
    elif layout == "all_cold":
        c = rng.integers(0, 64, E)
    elif layout == "all_hot":
        c = rng.integers(64, 131, E)
    elif layout == "one_hot":
        c = rng.integers(0, 64, E)
        c[17] = 5000
    else:
        raise ValueError(layout)
    assert c.sum() <= P
    return c


def offsets_of(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


@pytest.mark.parametrize("shared", [True, False])
@pytest.mark.parametrize("layout", LAYOUTS)
def test_split_gate_up_row_counts(inputs, layout, shared):
    host, dev = inputs
    rng = np.random.default_rng(2 * LAYOUTS.index(layout) + int(shared))
    counts = row_counts(layout, rng)
    off = offsets_of(counts)
    n = int(off[-1])
    tok = rng.integers(0, CFG.T, P).astype(np.int32)
    h = torch.full((P, CFG.I), 3.0, dtype=torch.bfloat16, device="cuda")
    hs = torch.empty((CFG.T, CFG.Is), dtype=torch.bfloat16, device="cuda")
    kw = dict(a_shared=dev.x, w_shared=dev.ws_gate_up, out_shared=hs) if shared else {}
    ws = B.workspace(CFG, B.MOE_ENTRY_GROUPED_GEMM)
    B.grouped_gemm(CFG, B.MOE_OP_GATE_UP_SWIGLU, dev.x, torch.from_numpy(off).cuda(),
                   dev.w_gate_up, h, a_row_index=torch.from_numpy(tok).cuda(), ws=ws, **kw)
    torch.cuda.synchronize()
    assert B.get_status(ws) == B.MOE_OK
    xh = as_u16(host.x)
    ref = np.empty((n, CFG.I))
    for e in range(CFG.E):
        r0, r1 = off[e], off[e + 1]
        if r1 > r0:
            ref[r0:r1] = oracle.expert_hidden(xh[tok[r0:r1]], as_u16(host.w_gate_up[e]))
    got = y_host(h)
    tol_check(got[:n], ref, what=f"h ({layout})")
    assert (got[n:] == 3.0).all()  # rows past the last group are not written
    if shared:
        tol_check(y_host(hs), oracle.expert_hidden(xh, as_u16(host.ws_gate_up)), what="h_shared")


@pytest.mark.parametrize("layout", ["boundary", "one_hot"])
def test_split_down_row_counts(inputs, layout):
    host, dev = inputs
    rng = np.random.default_rng(7 if layout == "boundary" else 8)
    counts = row_counts(layout, rng)
    off = offsets_of(counts)
    n = int(off[-1])
    perm = rng.permutation(P).astype(np.int32)
    ids = rng.integers(0, CFG.E, (CFG.T, CFG.k)).astype(np.int32)
    wts = rng.random((CFG.T, CFG.k)).astype(np.float32)
    blob = oracle.pack_blob(ids, wts)
    g = torch.Generator().manual_seed(5)
    h = (torch.randn((P, CFG.I), generator=g) * 0.5).to(torch.bfloat16)
    o = torch.full((P, CFG.D), 9.0, dtype=torch.float32, device="cuda")
    ws = B.workspace(CFG, B.MOE_ENTRY_GROUPED_GEMM)
    B.grouped_gemm(CFG, B.MOE_OP_DOWN_WEIGHTED, h.cuda(), torch.from_numpy(off).cuda(),
                   dev.w_down, o, perm_pair=torch.from_numpy(perm).cuda(),
                   blob=torch.from_numpy(blob).cuda(), ws=ws)
    torch.cuda.synchronize()
    assert B.get_status(ws) == B.MOE_OK
    hf = h.float().numpy().astype(np.float64)
    wrow = wts.reshape(-1)[perm].astype(np.float64)
    ref = np.empty((n, CFG.D))
    for e in range(CFG.E):
        r0, r1 = off[e], off[e + 1]
        if r1 > r0:
            ref[r0:r1] = oracle.expert_down(hf[r0:r1], as_u16(host.w_down[e])) * wrow[r0:r1, None]
    got = o.cpu().numpy()
    tol_check(got[:n], ref, max_rel=1e-4, mean_rel=1e-5, what=f"o ({layout})")
    assert (got[n:] == 9.0).all()


def test_first_split_call_inside_a_capture(inputs):
    """A host thread that has never made a split call captures moe_forward:
    the library's second stream is created inside the capture, and replays
    equal an eager call bit for bit."""
    host, dev = inputs
    W = B.weights_struct(dev, CFG)
    y_eager = B.forward(CFG, dev.x, W, ws=B.workspace(CFG, B.MOE_ENTRY_FORWARD))
    torch.cuda.synchronize()
    out = {}

    def worker():
        try:
            torch.cuda.set_device(0)
            y = torch.empty((CFG.T, CFG.D), dtype=torch.bfloat16, device="cuda")
            ws = B.workspace(CFG, B.MOE_ENTRY_FORWARD)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                B.forward(CFG, dev.x, W, y=y, ws=ws)
            for _ in range(2):
                y.zero_()
                graph.replay()
                torch.cuda.synchronize()
                out.setdefault("same", []).append(bool(torch.equal(y, y_eager)))
            out["status"] = B.get_status(ws)
        except Exception as exc:  # reported on the main thread
            out["error"] = repr(exc)

    t = threading.Thread(target=worker)
    t.start()
    t.join(timeout=300)
    assert not t.is_alive()
    assert "error" not in out, out.get("error")
    assert out["same"] == [True, True] and out["status"] == B.MOE_OK


def test_release_cache_between_split_calls(inputs):
    """moe_release_cache drops the calling thread's split stream and events,
    also with a forward still queued; the next forward creates them again and
    gives the same bits."""
    host, dev = inputs
    W = B.weights_struct(dev, CFG)
    ws = B.workspace(CFG, B.MOE_ENTRY_FORWARD)
    y0 = B.forward(CFG, dev.x, W, ws=ws)
    B.release_cache()  # the forward may still be running
    y1 = B.forward(CFG, dev.x, W, ws=ws)
    B.release_cache()
    B.release_cache()  # nothing cached: still fine
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)
    assert B.get_status(ws) == B.MOE_OK
