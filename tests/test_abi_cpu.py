"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/moe.h declares, sizes workspaces, and rejects invalid
arguments on the host (before any CUDA call)."""
import ctypes
import dataclasses
import os
import re

import pytest

from sparse_moe_layer_router_gb300 import binding as B
from sparse_moe_layer_router_gb300.build import build
from sparse_moe_layer_router_gb300.synthetic import CONFIGS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return B.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert set(names) == set(B.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_sizes(lib):
    for name, cfg in CONFIGS.items():
        for entry in range(6):
            n = B.workspace_size(cfg, entry)
            assert n >= 256 and n % 256 == 0, (name, entry, n)
        fwd = B.workspace_size(cfg, B.MOE_ENTRY_FORWARD)
        host = B.workspace_size(cfg, B.MOE_ENTRY_FORWARD_HOST)
        assert host >= fwd + 2 * 2 * cfg.T * cfg.D
    assert B.workspace_size(CONFIGS["tiny"], 99) == 0


@pytest.mark.parametrize("field,value,code", [
    ("k", 0, B.MOE_ERR_INVALID_ARG),
    ("k", 17, B.MOE_ERR_INVALID_ARG),     # k > E
    ("T", 0, B.MOE_ERR_INVALID_ARG),
    ("D", 200, B.MOE_ERR_UNSUPPORTED),    # not a multiple of 128
    ("I", 100, B.MOE_ERR_UNSUPPORTED),    # not a multiple of 64
    ("E", 2000, B.MOE_ERR_UNSUPPORTED),
    ("quant", 7, B.MOE_ERR_UNSUPPORTED),
])
def test_invalid_config_rejected_on_host(lib, field, value, code):
    cfg = B.config(CONFIGS["tiny"])
    setattr(cfg, field, value)
    assert lib.moe_workspace_size(ctypes.byref(cfg), B.MOE_ENTRY_FORWARD) == 0
    dummy = ctypes.c_void_p(4096)
    rc = lib.moe_route(ctypes.byref(cfg), dummy, dummy, None, dummy, dummy, 1 << 30, None)
    assert rc == code


@pytest.mark.parametrize("group,ok", [(128, True), (0, True), (64, False), (256, False),
                                      (-1, False)])
def test_w4a16_group_is_128_or_channel(lib, group, ok):
    """Group scales of 128 along K, or channel-wise (group 0); nothing else."""
    cfg = B.config(CONFIGS["w4a16"])
    cfg.group = group
    assert (lib.moe_workspace_size(ctypes.byref(cfg), B.MOE_ENTRY_FORWARD) > 0) == ok


def test_w4a16_needs_whole_packed_k_tiles(lib):
    cfg = B.config(CONFIGS["w4a16"])
    cfg.I = 1024 + 128  # not a multiple of 256
    assert lib.moe_workspace_size(ctypes.byref(cfg), B.MOE_ENTRY_FORWARD) == 0


def test_null_and_misaligned_pointers_rejected(lib):
    cfg = B.config(CONFIGS["tiny"])
    d = ctypes.c_void_p(4096)
    assert lib.moe_route(ctypes.byref(cfg), None, d, None, d, d, 1 << 30, None) == B.MOE_ERR_INVALID_ARG
    odd = ctypes.c_void_p(4096 + 2)
    assert lib.moe_route(ctypes.byref(cfg), odd, d, None, d, d, 1 << 30, None) == B.MOE_ERR_ALIGN
    assert lib.moe_permute(ctypes.byref(cfg), None, d, d, d, d, None, None, d, 1 << 30, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_permute(ctypes.byref(cfg), d, d, d, d, d, d, None, d, 1 << 30, None) == B.MOE_ERR_INVALID_ARG
    w = B.MoeWeights()
    assert lib.moe_forward(ctypes.byref(cfg), d, ctypes.byref(w), d, d, 1 << 30, None) == B.MOE_ERR_INVALID_ARG
    args = B.MoeGemmArgs()
    assert lib.moe_grouped_gemm(ctypes.byref(cfg), ctypes.byref(args), d, 1 << 30, None) == B.MOE_ERR_INVALID_ARG


def test_router_logits_host_validation(lib):
    cfg = B.config(CONFIGS["tiny"])
    d = ctypes.c_void_p(4096)
    odd = ctypes.c_void_p(4096 + 4)
    assert lib.moe_router_logits(ctypes.byref(cfg), d, d, None, d, 1 << 30, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_router_logits(ctypes.byref(cfg), d, d, odd, d, 1 << 30, None) == B.MOE_ERR_ALIGN
    need = lib.moe_workspace_size(ctypes.byref(cfg), B.MOE_ENTRY_ROUTE)
    assert lib.moe_router_logits(ctypes.byref(cfg), d, d, d, d, need - 1, None) == B.MOE_ERR_WORKSPACE
    bad = B.config(CONFIGS["tiny"])
    bad.k = 0
    assert lib.moe_router_logits(ctypes.byref(bad), d, d, d, d, 1 << 30, None) == B.MOE_ERR_INVALID_ARG


def test_small_workspace_rejected(lib):
    cfg = B.config(CONFIGS["tiny"])
    d = ctypes.c_void_p(4096)
    need = lib.moe_workspace_size(ctypes.byref(cfg), B.MOE_ENTRY_ROUTE)
    assert lib.moe_route(ctypes.byref(cfg), d, d, None, d, d, need - 1, None) == B.MOE_ERR_WORKSPACE


def test_bf16_weights_with_scales_rejected(lib):
    cfg = B.config(CONFIGS["tiny"])
    d = ctypes.c_void_p(4096)
    w = B.MoeWeights(d, None, d, d, d, None, d, d, None, None)
    assert lib.moe_forward(ctypes.byref(cfg), d, ctypes.byref(w), d, d, 1 << 30, None) == B.MOE_ERR_INVALID_ARG


def test_strerror(lib):
    for c in (0, -1, -2, -3, -4, -5, -6):
        assert B.strerror(c) and B.strerror(c) != "unknown error"
    assert B.strerror(-99) == "unknown error"


def test_repack_and_expert_slice_host_validation(lib):
    d = ctypes.c_void_p(4096)
    assert lib.moe_repack_int4(None, d, 8, B.MOE_INT4_SEQUENTIAL, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_repack_int4(d, d, 8, 5, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_repack_int4(ctypes.c_void_p(4100), d, 8, 0, None) == B.MOE_ERR_ALIGN
    assert lib.moe_repack_int4(d, d, 0, 0, None) == B.MOE_OK  # nothing to do
    cfg = B.config(CONFIGS["tiny"])
    w = B.MoeWeights(None, None, d, d, None, None, d, d, None, None)
    ws_n = B.workspace_size(CONFIGS["tiny"], B.MOE_ENTRY_FORWARD_EXPERTS)
    assert ws_n >= 256

    def call(e0, e1, s0, s1, ws_bytes=ws_n, weights=w):
        return lib.moe_forward_experts(ctypes.byref(cfg), d, d, ctypes.byref(weights), e0, e1,
                                       s0, s1, d, d, ws_bytes, None)
    assert call(2, 2, 0, 0) == B.MOE_ERR_INVALID_ARG        # empty expert range
    assert call(0, 17, 0, 0) == B.MOE_ERR_INVALID_ARG       # past E
    assert call(0, 4, 3, 2) == B.MOE_ERR_INVALID_ARG        # reversed shared range
    assert call(0, 4, 0, 65) == B.MOE_ERR_INVALID_ARG       # past T
    assert call(0, 4, 0, 8, ws_bytes=255) == B.MOE_ERR_WORKSPACE
    no_shared = B.MoeWeights(None, None, d, d, None, None, None, None, None, None)
    assert call(0, 4, 0, 8, weights=no_shared) == B.MOE_ERR_INVALID_ARG


def test_binding_rejects_tensors_the_kernels_would_overrun(lib):
    """The binding checks dtype and extent of every tensor against cfg before
    the call: an fp32 output given as bf16 (half the bytes), a short buffer or
    int4 words given as bf16 raise ValueError on the host."""
    import torch
    cfg = CONFIGS["tiny"]
    P = cfg.T * cfg.k
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    h = torch.empty((P, cfg.I), dtype=bf)
    off = torch.empty(cfg.E + 1, dtype=i32)
    wd = torch.empty((cfg.E, cfg.D, cfg.I), dtype=bf)
    perm = torch.empty(P, dtype=i32)
    blob = torch.empty((cfg.T, 2, cfg.k), dtype=i32)
    o_half = torch.empty((P, cfg.D), dtype=bf)       # down output is fp32
    with pytest.raises(ValueError, match="out: expected torch.float32"):
        B.grouped_gemm(cfg, B.MOE_OP_DOWN_WEIGHTED, h, off, wd, o_half, perm_pair=perm, blob=blob)
    o_short = torch.empty((P - 1, cfg.D), dtype=f32)
    with pytest.raises(ValueError, match="out: needs"):
        B.grouped_gemm(cfg, B.MOE_OP_DOWN_WEIGHTED, h, off, wd, o_short, perm_pair=perm, blob=blob)
    with pytest.raises(ValueError, match="o: expected torch.float32"):
        B.combine(cfg, o_half, None, perm, y=torch.empty((cfg.T, cfg.D), dtype=bf))
    with pytest.raises(ValueError, match="y_partial: needs"):
        B.forward_experts(cfg, torch.empty((cfg.T, cfg.D), dtype=bf), blob,
                          B.MoeWeights(), 0, 1, y_partial=torch.empty(cfg.T, dtype=f32))
    with pytest.raises(ValueError, match="blob: needs"):
        B.permute(cfg, torch.empty(cfg.T, dtype=i32))
    with pytest.raises(ValueError, match="dst: needs"):
        B.repack_int4(torch.empty(64, dtype=i32), torch.empty(63, dtype=i32))
    # W4A16: packed int32 words, bf16 scales per group of inputs
    w4 = dataclasses.replace(cfg, quant=B.MOE_QUANT_W4A16, group=128)
    with pytest.raises(ValueError, match="w: expected torch.int32"):
        B.grouped_gemm(w4, B.MOE_OP_DOWN_WEIGHTED, h, off, wd, torch.empty((P, cfg.D), dtype=f32),
                       perm_pair=perm, blob=blob)
    # right dtypes and extents get as far as the device check
    with pytest.raises(ValueError, match="CUDA"):
        B.grouped_gemm(cfg, B.MOE_OP_DOWN_WEIGHTED, h, off, wd, torch.empty((P, cfg.D), dtype=f32),
                       perm_pair=perm, blob=blob)


def test_header_is_plain_c(tmp_path):
    """include/moe.h compiles as C99 (no C++ or CUDA types in the ABI), and a
    caller written as the README shows type-checks against it."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "caller.c"
    src.write_text('''
#include <stddef.h>
#include <stdio.h>
#include "moe.h"
int call(const void *x, void *y, const void *wr, const void *w_gu, const void *w_dn,
         const void *ws_gu, const void *ws_dn, void *ws, void *stream) {
  moe_config cfg = {.T = 64, .D = 4096, .E = 512, .I = 1024, .I_shared = 1024, .k = 10,
                    .quant = MOE_QUANT_BF16, .group = 128};
  moe_weights w = {.w_router = wr, .router_bias = NULL, .w_gate_up = w_gu, .w_down = w_dn,
                   .ws_gate_up = ws_gu, .ws_down = ws_dn};
  size_t ws_bytes = moe_workspace_size(&cfg, MOE_ENTRY_FORWARD);
  int rc = moe_forward(&cfg, x, &w, y, ws, ws_bytes, stream);
  if (rc != MOE_OK) fprintf(stderr, "%s\\n", moe_strerror(rc));
  return rc != MOE_OK ? rc : moe_get_status(ws, stream);
}
''')
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-pedantic", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
