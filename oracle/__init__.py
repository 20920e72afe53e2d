"""fp64 CPU oracle for the routed sparse-MoE FFN layer -- TEST INFRASTRUCTURE.

This package is the checker, not the product.  Only ``tests/``, the smoke check
in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.
It shares no code with the CUDA library and never imports it.

The arithmetic lives in ``moe_oracle.c`` (plain loops, fp64); this module only
compiles it with gcc and marshals numpy arrays through ctypes.  bf16 tensors
travel as ``uint16`` bit patterns.

Citations (page title, section):
  * router softmax + top-k, always-on shared expert: "Systems engineering
    playbook: optimizing Qwen 3.5-397B MoE on Ironwood (TPU7x)", section 1,
    "Sparse Mixture-of-Experts (MoE)".
  * packed int32 routing blob: same page, section 3, "3-to-2 All-Gather".
  * dispatch grouping: same page, section 3, "Option B".
  * int4 pack-quantized weights with group scales: "vLLM TPU Inference
    v0.31.0: hierarchical MoE dispatch and W4A16", 4-bit weight section.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FP contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_router_logits.argtypes = [I, I, I, P, P, P, P]
            lib.oracle_route.argtypes = [I, I, I, I, P, P, P, P, P, P]
            lib.oracle_pack_blob.argtypes = [I, I, P, P, P]
            lib.oracle_unpack_blob.argtypes = [I, I, P, P, P]
            lib.oracle_permute.argtypes = [I, I, I, P, P, P, P, P]
            lib.oracle_dequant_w4.argtypes = [I, I, I, P, P, P]
            lib.oracle_forward.argtypes = [I, I, I, I, I, I, I, I, P, P, P, P, P, P, P, P]
            lib.oracle_num_threads.argtypes = []
            lib.oracle_expert_hidden.argtypes = [I, I, I, I, I, P, P, P, P]
            lib.oracle_expert_down.argtypes = [I, I, I, I, I, P, P, P, P]
            lib.oracle_expert_hidden.restype = ctypes.c_int
            lib.oracle_combine.argtypes = [I, I, I, P, P, P, P]
            lib.oracle_combine.restype = ctypes.c_int
            lib.oracle_expert_down.restype = ctypes.c_int
            for f in (lib.oracle_router_logits, lib.oracle_route, lib.oracle_pack_blob,
                      lib.oracle_unpack_blob, lib.oracle_permute, lib.oracle_dequant_w4,
                      lib.oracle_forward, lib.oracle_num_threads):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def router_logits(x, wr, bias=None):
    """fp64 logits z[t, e] = sum_d x[t,d] Wr[e,d] (index order) + bias[e]."""
    x = _c(x, np.uint16)
    wr = _c(wr, np.uint16)
    T, D = x.shape
    E = wr.shape[0]
    assert wr.shape[1] == D
    b = None if bias is None else _c(bias, np.float32)
    z = np.empty((T, E), np.float64)
    _check(_load().oracle_router_logits(T, D, E, _ptr(x), _ptr(wr), _ptr(b), _ptr(z)),
           "router_logits")
    return z


def route(x, wr, k, bias=None, return_logits=False):
    """Top-k routing of every token: ids [T,k] int32 (ascending), w [T,k] fp64."""
    x = _c(x, np.uint16)
    wr = _c(wr, np.uint16)
    T, D = x.shape
    E = wr.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    z = np.empty((T, E), np.float64) if return_logits else None
    _check(_load().oracle_route(T, D, E, k, _ptr(x), _ptr(wr), _ptr(b), _ptr(ids), _ptr(w),
                                _ptr(z)), "route")
    return (ids, w, z) if return_logits else (ids, w)


def pack_blob(ids, w):
    """int32 blob [T][2][k]: ids, then the fp32 bit patterns of the weights."""
    ids = _c(ids, np.int32)
    w = _c(w, np.float64)
    T, k = ids.shape
    blob = np.empty((T, 2, k), np.int32)
    _check(_load().oracle_pack_blob(T, k, _ptr(ids), _ptr(w), _ptr(blob)), "pack_blob")
    return blob


def unpack_blob(blob):
    blob = _c(blob, np.int32)
    T, two, k = blob.shape
    assert two == 2
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    _check(_load().oracle_unpack_blob(T, k, _ptr(blob), _ptr(ids), _ptr(w)), "unpack_blob")
    return ids, w


def permute(ids, E):
    """Stable grouping of pairs by expert: counts, offsets, perm_pair, inv_row."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    _check(_load().oracle_permute(T, E, k, _ptr(ids), _ptr(counts), _ptr(offsets), _ptr(perm),
                                  _ptr(inv)), "permute")
    return counts, offsets, perm, inv


def dequant_w4(q, s, group):
    """Exact fp64 value of a packed int4 matrix: q [R, C/8] int32, s [R, C/group] bf16
    (group 0: channel-wise, s [R] or [R, 1])."""
    q = _c(q, np.int32)
    s = _c(s, np.uint16)
    R = q.shape[0]
    C = q.shape[1] * 8
    out = np.empty((R, C), np.float64)
    _check(_load().oracle_dequant_w4(R, C, group, _ptr(q), _ptr(s), _ptr(out)), "dequant_w4")
    return out


def expert_hidden(x_rows, w_gate_up, s_gate_up=None, *, group=128):
    """SwiGLU hidden (fp64) of one expert for each row: [n, Ie]."""
    x_rows = _c(x_rows, np.uint16)
    n, D = x_rows.shape
    quant = 0 if s_gate_up is None else 1
    wg = _c(w_gate_up, np.uint16 if quant == 0 else np.int32)
    sg = None if quant == 0 else _c(s_gate_up, np.uint16)
    Ie = wg.shape[0] // 2
    h = np.empty((n, Ie), np.float64)
    _check(_load().oracle_expert_hidden(n, D, Ie, quant, group, _ptr(x_rows), _ptr(wg), _ptr(sg),
                                        _ptr(h)), "expert_hidden")
    return h


def expert_down(h, w_down, s_down=None, *, group=128):
    """Down projection (fp64) of one expert for each row of h [n, Ie]: [n, D]."""
    h = _c(h, np.float64)
    n, Ie = h.shape
    quant = 0 if s_down is None else 1
    wd = _c(w_down, np.uint16 if quant == 0 else np.int32)
    sd = None if quant == 0 else _c(s_down, np.uint16)
    D = wd.shape[0]
    o = np.empty((n, D), np.float64)
    _check(_load().oracle_expert_down(n, D, Ie, quant, group, _ptr(h), _ptr(wd), _ptr(sd), _ptr(o)),
           "expert_down")
    return o


def combine(o, o_shared, inv_row, k):
    """y [T, D] (fp64) = o_shared[t] + sum_j o[inv_row[t*k+j]]."""
    o = _c(o, np.float64)
    inv_row = _c(inv_row, np.int32).reshape(-1)
    T = inv_row.size // k
    D = o.shape[1]
    osh = None if o_shared is None else _c(o_shared, np.float64)
    y = np.empty((T, D), np.float64)
    _check(_load().oracle_combine(T, D, k, _ptr(o), _ptr(osh), _ptr(inv_row), _ptr(y)), "combine")
    return y


def forward(x_rows, ids, w, experts, shared, *, E, I, Is, quant=0, group=128):
    """Layer output (fp64) for the tokens in ``x_rows`` given their routing.

    ``experts`` maps expert index -> weights of that expert; only the experts
    the given tokens use need to be present.  Weights of one expert are
    ``(w_gate_up, w_down)`` (bf16 as uint16) when quant == 0, and
    ``(q_gate_up, s_gate_up, q_down, s_down)`` when quant == 1.  ``shared`` has
    the same form.
    """
    x_rows = _c(x_rows, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float64)
    nt, D = x_rows.shape
    k = ids.shape[1]
    keep = []
    a_gu = np.zeros(E + 1, np.uint64)
    a_dn = np.zeros(E + 1, np.uint64)
    s_gu = np.zeros(E + 1, np.uint64)
    s_dn = np.zeros(E + 1, np.uint64)

    def put(idx, tensors):
        if quant == 0:
            gu, dn = (_c(tensors[0], np.uint16), _c(tensors[1], np.uint16))
            keep.extend([gu, dn])
            a_gu[idx], a_dn[idx] = gu.ctypes.data, dn.ctypes.data
        else:
            qgu, sgu, qdn, sdn = (_c(tensors[0], np.int32), _c(tensors[1], np.uint16),
                                  _c(tensors[2], np.int32), _c(tensors[3], np.uint16))
            keep.extend([qgu, sgu, qdn, sdn])
            a_gu[idx], s_gu[idx] = qgu.ctypes.data, sgu.ctypes.data
            a_dn[idx], s_dn[idx] = qdn.ctypes.data, sdn.ctypes.data

    for e, t in experts.items():
        if not 0 <= e < E:
            raise ValueError(f"expert index {e} outside [0, {E})")
        put(e, t)
    put(E, shared)
    y = np.empty((nt, D), np.float64)
    _check(_load().oracle_forward(nt, D, E, I, Is, k, quant, group, _ptr(x_rows), _ptr(ids),
                                  _ptr(w), _ptr(a_gu), _ptr(s_gu) if quant else None, _ptr(a_dn),
                                  _ptr(s_dn) if quant else None, _ptr(y)), "forward")
    return y


def layer(x, wr, k, experts, shared, *, I, Is, bias=None, quant=0, group=128):
    """Whole layer: route every token, then the fp64 forward.  Returns (y, ids, w)."""
    ids, w = route(x, wr, k, bias)
    E = int(np.asarray(wr).shape[0])
    y = forward(x, ids, w, experts, shared, E=E, I=I, Is=Is, quant=quant, group=group)
    return y, ids, w
