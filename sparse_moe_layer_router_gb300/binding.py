"""ctypes binding of the libmoe_gb300 C ABI (``include/moe.h``).

Argument marshalling only: torch tensors become device pointers, the current
torch CUDA stream becomes the ``stream`` argument, and a negative return code
becomes ``MoeError``.  Every step of the layer runs in the library's kernels.
There is no fallback: a missing library or a missing GPU raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_WORKSPACE = -3
MOE_ERR_CUDA = -4
MOE_ERR_TIMEOUT = -5
MOE_ERR_ALIGN = -6
MOE_ERR_SCRATCH_LIMIT = -7

MOE_QUANT_BF16 = 0
MOE_QUANT_W4A16 = 1
MOE_OP_GATE_UP_SWIGLU = 0
MOE_OP_DOWN_WEIGHTED = 1
MOE_ENTRY_ROUTE = 0
MOE_ENTRY_PERMUTE = 1
MOE_ENTRY_GROUPED_GEMM = 2
MOE_ENTRY_FORWARD = 3
MOE_ENTRY_FORWARD_HOST = 4
MOE_ENTRY_FORWARD_EXPERTS = 5
MOE_INT4_SEQUENTIAL = 0
MOE_INT4_SEQUENTIAL_OFFSET8 = 1

# Every function declared in include/moe.h.
EXPORTS = ("moe_workspace_size", "moe_route", "moe_router_logits", "moe_permute", "moe_permute_static",
           "moe_grouped_gemm", "moe_combine", "moe_forward", "moe_forward_host",
           "moe_forward_experts", "moe_repack_int4", "moe_get_status",
           "moe_selftest_wait_timeout", "moe_release_cache", "moe_strerror")


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("D", ctypes.c_int), ("E", ctypes.c_int), ("I", ctypes.c_int),
                ("I_shared", ctypes.c_int), ("k", ctypes.c_int), ("quant", ctypes.c_int),
                ("group", ctypes.c_int)]


class MoeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w_router", "router_bias", "w_gate_up", "w_down", "s_gate_up", "s_down", "ws_gate_up",
        "ws_down", "ss_gate_up", "ss_down")]


class MoeGemmArgs(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int)] + [(n, ctypes.c_void_p) for n in (
        "a", "a_row_index", "offsets", "w", "w_scales", "perm_pair", "blob", "out", "a_shared",
        "w_shared", "ws_scales", "out_shared")]


_lock = threading.Lock()
_lib = None


def lib():
    """Load libmoe_gb300.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m sparse_moe_layer_router_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            cfgp = ctypes.POINTER(MoeConfig)
            L.moe_workspace_size.argtypes = [cfgp, I]
            L.moe_workspace_size.restype = S
            L.moe_route.argtypes = [cfgp, P, P, P, P, P, S, P]
            L.moe_router_logits.argtypes = [cfgp, P, P, P, P, S, P]
            L.moe_permute.argtypes = [cfgp, P, P, P, P, P, P, P, P, S, P]
            L.moe_permute_static.argtypes = [cfgp, P, P, P, P, P, P, P, P]
            L.moe_grouped_gemm.argtypes = [cfgp, ctypes.POINTER(MoeGemmArgs), P, S, P]
            L.moe_combine.argtypes = [cfgp, P, P, P, P, P]
            L.moe_forward.argtypes = [cfgp, P, ctypes.POINTER(MoeWeights), P, P, S, P]
            L.moe_forward_host.argtypes = [cfgp, P, ctypes.POINTER(MoeWeights), P, P, S, P]
            L.moe_forward_experts.argtypes = [cfgp, P, P, ctypes.POINTER(MoeWeights), I, I, I, I,
                                              P, P, S, P]
            L.moe_repack_int4.argtypes = [P, P, S, I, P]
            L.moe_get_status.argtypes = [P, P]
            L.moe_selftest_wait_timeout.argtypes = [P, S, ctypes.c_uint, P]
            L.moe_release_cache.argtypes = []
            L.moe_strerror.argtypes = [I]
            L.moe_strerror.restype = ctypes.c_char_p
            for n in ("moe_route", "moe_router_logits", "moe_permute", "moe_permute_static",
                      "moe_grouped_gemm", "moe_combine", "moe_forward", "moe_forward_host",
                      "moe_forward_experts", "moe_repack_int4", "moe_get_status",
                      "moe_selftest_wait_timeout", "moe_release_cache"):
                getattr(L, n).restype = I
            _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().moe_strerror(int(code)).decode()


def config(cfg) -> MoeConfig:
    """MoeConfig from any object with T, D, E, I, Is, k, quant, group attributes."""
    return MoeConfig(cfg.T, cfg.D, cfg.E, cfg.I, cfg.Is, cfg.k, cfg.quant, cfg.group)


def _p(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        return ctypes.c_void_p(int(t))
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _need(t, name, dtype, numel):
    """Reject a tensor of the wrong type, or one the kernels would read or write
    past the end of (``numel`` elements at least).  Raw integer pointers pass
    unchecked: their extent is the caller's responsibility."""
    if not isinstance(t, torch.Tensor):
        return
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.numel() < numel:
        raise ValueError(f"{name}: needs {numel} elements, has {t.numel()}")


def _weight_spec(cfg, gate_up, shared, n_experts=None):
    """(dtype, weight elements, scale elements) of one projection in the
    format of moe_weights: bf16 rows, or int32 words of 8 int4 values plus bf16
    scales (per group of ``group`` inputs, or one per row when group == 0)."""
    i = cfg.Is if shared else cfg.I
    rows, K = (2 * i, cfg.D) if gate_up else (cfg.D, i)
    n = 1 if shared else (cfg.E if n_experts is None else n_experts)
    if cfg.quant == MOE_QUANT_W4A16:
        per_row = K // cfg.group if cfg.group > 0 else 1
        return torch.int32, n * rows * K // 8, n * rows * per_row
    return torch.bfloat16, n * rows * K, 0


def _need_weights(cfg, inp, n_experts=None):
    """Check the tensors of a MoEInputs-like object against cfg."""
    bf = torch.bfloat16
    _need(getattr(inp, "w_router", None), "w_router", bf, cfg.E * cfg.D)
    _need(getattr(inp, "bias", None), "router_bias", torch.float32, cfg.E)
    for gate_up, shared, w, s in ((True, False, "w_gate_up", "s_gate_up"),
                                  (False, False, "w_down", "s_down"),
                                  (True, True, "ws_gate_up", "ss_gate_up"),
                                  (False, True, "ws_down", "ss_down")):
        dt, nw, ns = _weight_spec(cfg, gate_up, shared, n_experts)
        _need(getattr(inp, w, None), w, dt, nw)
        _need(getattr(inp, s, None), s, bf, ns)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, what: str):
    if rc != MOE_OK:
        raise MoeError(rc, what)


def workspace_size(cfg, entry: int) -> int:
    return int(lib().moe_workspace_size(ctypes.byref(config(cfg)), entry))


def workspace(cfg, entry: int, device=None) -> torch.Tensor:
    n = workspace_size(cfg, entry)
    if n == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "workspace_size")
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    ws[:256].zero_()
    return ws


def route(cfg, x, w_router, bias=None, blob=None, ws=None, stream=None):
    """int32 blob [T, 2, k] (ids ascending, then fp32 weight bits)."""
    if blob is None:
        blob = torch.empty((cfg.T, 2, cfg.k), dtype=torch.int32, device=x.device)
    _need(x, "x", torch.bfloat16, cfg.T * cfg.D)
    _need(w_router, "w_router", torch.bfloat16, cfg.E * cfg.D)
    _need(bias, "bias", torch.float32, cfg.E)
    _need(blob, "blob", torch.int32, cfg.T * 2 * cfg.k)
    if ws is None:
        ws = workspace(cfg, MOE_ENTRY_ROUTE, x.device)
    _check(lib().moe_route(ctypes.byref(config(cfg)), _p(x), _p(w_router), _p(bias), _p(blob),
                           _p(ws), ws.numel(), _stream(stream)), "moe_route")
    return blob


def router_logits(cfg, x, w_router, z=None, ws=None, stream=None):
    """fp32 [T, E] level-1 router logits x . Wr^T (tensor cores, no bias)."""
    if z is None:
        z = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device=x.device)
    _need(x, "x", torch.bfloat16, cfg.T * cfg.D)
    _need(w_router, "w_router", torch.bfloat16, cfg.E * cfg.D)
    _need(z, "z", torch.float32, cfg.T * cfg.E)
    if ws is None:
        ws = workspace(cfg, MOE_ENTRY_ROUTE, x.device)
    _check(lib().moe_router_logits(ctypes.byref(config(cfg)), _p(x), _p(w_router), _p(z), _p(ws),
                                   ws.numel(), _stream(stream)), "moe_router_logits")
    return z


def permute(cfg, blob, ws=None, stream=None, x=None, x_perm=None, out=None):
    """(counts [E], offsets [E+1], perm_pair [T*k], inv_row [T*k]) int32; with ``x``
    and ``x_perm`` also gathers token rows in grouped order.  ``out`` may hold
    preallocated (counts, offsets, perm_pair, inv_row)."""
    dev = blob.device
    if out is None:
        out = (torch.empty(cfg.E, dtype=torch.int32, device=dev),
               torch.empty(cfg.E + 1, dtype=torch.int32, device=dev),
               torch.empty(cfg.T * cfg.k, dtype=torch.int32, device=dev),
               torch.empty(cfg.T * cfg.k, dtype=torch.int32, device=dev))
    counts, offsets, perm, inv = out
    _need_permute(cfg, blob, counts, offsets, perm, inv, x, x_perm)
    if ws is None:
        ws = workspace(cfg, MOE_ENTRY_PERMUTE, dev)
    _check(lib().moe_permute(ctypes.byref(config(cfg)), _p(blob), _p(counts), _p(offsets), _p(perm),
                             _p(inv), _p(x), _p(x_perm), _p(ws), ws.numel(), _stream(stream)),
           "moe_permute")
    return counts, offsets, perm, inv


def _need_permute(cfg, blob, counts, offsets, perm, inv, x, x_perm):
    P = cfg.T * cfg.k
    _need(blob, "blob", torch.int32, cfg.T * 2 * cfg.k)
    _need(counts, "counts", torch.int32, cfg.E)
    _need(offsets, "offsets", torch.int32, cfg.E + 1)
    _need(perm, "perm_pair", torch.int32, P)
    _need(inv, "inv_row", torch.int32, P)
    _need(x, "x", torch.bfloat16, cfg.T * cfg.D)
    _need(x_perm, "x_perm", torch.bfloat16, P * cfg.D)


def permute_static(cfg, blob, stream=None, x=None, x_perm=None):
    """moe_permute without a workspace (fixed scratch inside the library)."""
    dev = blob.device
    counts = torch.empty(cfg.E, dtype=torch.int32, device=dev)
    offsets = torch.empty(cfg.E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(cfg.T * cfg.k, dtype=torch.int32, device=dev)
    inv = torch.empty(cfg.T * cfg.k, dtype=torch.int32, device=dev)
    _need_permute(cfg, blob, counts, offsets, perm, inv, x, x_perm)
    _check(lib().moe_permute_static(ctypes.byref(config(cfg)), _p(blob), _p(counts), _p(offsets),
                                    _p(perm), _p(inv), _p(x), _p(x_perm), _stream(stream)),
           "moe_permute_static")
    return counts, offsets, perm, inv


def grouped_gemm(cfg, op, a, offsets, w, out, *, a_row_index=None, w_scales=None, perm_pair=None,
                 blob=None, a_shared=None, w_shared=None, ws_scales=None, out_shared=None,
                 ws=None, stream=None):
    """One grouped GEMM launch (see moe_gemm_args in include/moe.h)."""
    P, bf, f32 = cfg.T * cfg.k, torch.bfloat16, torch.float32
    gate_up = op == MOE_OP_GATE_UP_SWIGLU
    K, K_s = (cfg.D, cfg.D) if gate_up else (cfg.I, cfg.Is)
    _need(a, "a", bf, (cfg.T if a_row_index is not None else P) * K)
    _need(a_row_index, "a_row_index", torch.int32, P)
    _need(offsets, "offsets", torch.int32, cfg.E + 1)
    dt, nw, ns = _weight_spec(cfg, gate_up, False)
    _need(w, "w", dt, nw)
    _need(w_scales, "w_scales", bf, ns)
    _need(out, "out", bf if gate_up else f32, P * (cfg.I if gate_up else cfg.D))
    _need(perm_pair, "perm_pair", torch.int32, P)
    _need(blob, "blob", torch.int32, cfg.T * 2 * cfg.k)
    _need(a_shared, "a_shared", bf, cfg.T * K_s)
    dt, nw, ns = _weight_spec(cfg, gate_up, True)
    _need(w_shared, "w_shared", dt, nw)
    _need(ws_scales, "ws_scales", bf, ns)
    _need(out_shared, "out_shared", bf if gate_up else f32,
          cfg.T * (cfg.Is if gate_up else cfg.D))
    args = MoeGemmArgs(op, _p(a), _p(a_row_index), _p(offsets), _p(w), _p(w_scales),
                       _p(perm_pair), _p(blob), _p(out), _p(a_shared), _p(w_shared),
                       _p(ws_scales), _p(out_shared))
    if ws is None:
        ws = workspace(cfg, MOE_ENTRY_GROUPED_GEMM, a.device)
    _check(lib().moe_grouped_gemm(ctypes.byref(config(cfg)), ctypes.byref(args), _p(ws), ws.numel(),
                                  _stream(stream)), "moe_grouped_gemm")
    return out, out_shared


def combine(cfg, o, o_shared, inv_row, y=None, stream=None):
    if y is None:
        y = torch.empty((cfg.T, cfg.D), dtype=torch.bfloat16, device=o.device)
    P = cfg.T * cfg.k
    _need(o, "o", torch.float32, P * cfg.D)
    _need(o_shared, "o_shared", torch.float32, cfg.T * cfg.D)
    _need(inv_row, "inv_row", torch.int32, P)
    _need(y, "y", torch.bfloat16, cfg.T * cfg.D)
    _check(lib().moe_combine(ctypes.byref(config(cfg)), _p(o), _p(o_shared), _p(inv_row), _p(y),
                             _stream(stream)), "moe_combine")
    return y


def weights_struct(inp, cfg=None) -> MoeWeights:
    """MoeWeights from a MoEInputs (all tensors on the GPU); with ``cfg`` the
    tensors are first checked against the shapes the layer reads."""
    if cfg is not None:
        _need_weights(cfg, inp)
    return MoeWeights(_p(inp.w_router), _p(inp.bias), _p(inp.w_gate_up), _p(inp.w_down),
                      _p(inp.s_gate_up), _p(inp.s_down), _p(inp.ws_gate_up), _p(inp.ws_down),
                      _p(inp.ss_gate_up), _p(inp.ss_down))


def forward(cfg, x, weights, y=None, ws=None, stream=None):
    """Whole layer; ``weights`` is a MoeWeights or a MoEInputs on the GPU."""
    if not isinstance(weights, MoeWeights):
        weights = weights_struct(weights, cfg)
    if y is None:
        y = torch.empty((cfg.T, cfg.D), dtype=torch.bfloat16, device=x.device)
    _need(x, "x", torch.bfloat16, cfg.T * cfg.D)
    _need(y, "y", torch.bfloat16, cfg.T * cfg.D)
    if ws is None:
        ws = workspace(cfg, MOE_ENTRY_FORWARD, x.device)
    _check(lib().moe_forward(ctypes.byref(config(cfg)), _p(x), ctypes.byref(weights), _p(y), _p(ws),
                             ws.numel(), _stream(stream)), "moe_forward")
    return y


def forward_host(cfg, x_host, weights, y_host, ws, stream=None):
    """Whole layer with host x / y (pinned CPU tensors); caller synchronises."""
    if not isinstance(weights, MoeWeights):
        weights = weights_struct(weights, cfg)
    for t in (x_host, y_host):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("forward_host takes contiguous CPU tensors")
    _need(x_host, "x_host", torch.bfloat16, cfg.T * cfg.D)
    _need(y_host, "y_host", torch.bfloat16, cfg.T * cfg.D)
    _check(lib().moe_forward_host(ctypes.byref(config(cfg)), ctypes.c_void_p(x_host.data_ptr()),
                                  ctypes.byref(weights), ctypes.c_void_p(y_host.data_ptr()),
                                  _p(ws), ws.numel(), _stream(stream)), "moe_forward_host")
    return y_host


def forward_experts(cfg, x, blob, weights, e_begin, e_end, shared_begin=0, shared_end=0,
                    y_partial=None, ws=None, stream=None):
    """fp32 [T, D] partial output of the routed experts [e_begin, e_end) (``weights``
    holds those experts only) plus the shared expert on tokens [shared_begin, shared_end)."""
    if not isinstance(weights, MoeWeights):
        _need_weights(cfg, weights, n_experts=max(int(e_end) - int(e_begin), 0))
        weights = weights_struct(weights)
    if y_partial is None:
        y_partial = torch.empty((cfg.T, cfg.D), dtype=torch.float32, device=x.device)
    _need(x, "x", torch.bfloat16, cfg.T * cfg.D)
    _need(blob, "blob", torch.int32, cfg.T * 2 * cfg.k)
    _need(y_partial, "y_partial", torch.float32, cfg.T * cfg.D)
    if ws is None:
        ws = workspace(cfg, MOE_ENTRY_FORWARD_EXPERTS, x.device)
    _check(lib().moe_forward_experts(ctypes.byref(config(cfg)), _p(x), _p(blob),
                                     ctypes.byref(weights), int(e_begin), int(e_end),
                                     int(shared_begin), int(shared_end), _p(y_partial), _p(ws),
                                     ws.numel(), _stream(stream)), "moe_forward_experts")
    return y_partial


def repack_int4(src, dst=None, layout=MOE_INT4_SEQUENTIAL, stream=None):
    """Sequential-order packed int4 words (int32 tensor) -> this library's pair order."""
    if src.dtype != torch.int32:
        raise ValueError("packed int4 words are int32")
    if dst is None:
        dst = torch.empty_like(src)
    _need(dst, "dst", torch.int32, src.numel())
    _check(lib().moe_repack_int4(_p(src), _p(dst), src.numel(), int(layout), _stream(stream)),
           "moe_repack_int4")
    return dst


def get_status(ws, stream=None) -> int:
    return int(lib().moe_get_status(_p(ws), _stream(stream)))


def release_cache() -> None:
    """moe_release_cache: drop this thread's cached split stream and events."""
    _check(lib().moe_release_cache(), "moe_release_cache")


def selftest_wait_timeout(ws, limit_ms=200, stream=None, read_status=True):
    """Run the bounded-wait self-test; returns the device status it leaves
    (MOE_ERR_TIMEOUT), or None with ``read_status=False`` (status left unread)."""
    _check(lib().moe_selftest_wait_timeout(_p(ws), ws.numel(), int(limit_ms), _stream(stream)),
           "moe_selftest_wait_timeout")
    return get_status(ws, stream) if read_status else None
