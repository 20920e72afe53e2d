"""Seeded synthetic inputs for the MoE layer (both the CUDA path and the oracle use these).

This module draws random numbers and lays tensors out; it holds none of the
layer's arithmetic.  Every tensor is reproducible from (config, seed): each
tensor, and each expert's weights, has its own sub-seed, so a single expert can
be regenerated without the others.

Distributions (the layer configurations): x ~ N(0, 1); router weight ~ N(0, 0.02);
expert and shared-expert weights ~ N(0, 1/sqrt(fan_in)) with fan_in = D for
gate/up and I for down.  Values are drawn in fp32 and rounded to bf16
(round-to-nearest-even).

The skewed-load configuration adds a router bias from log Zipf(s=1.2)
probabilities of a seeded random ranking of the experts, scaled by ``alpha``
so that about a fifth of the experts receive no token.

The W4A16 configuration quantises the same bf16 weights to symmetric int4
(range -8..7, no zero point), group 128 along K, bf16 scale per group, packed
8 values per int32 in pair order (value 2i at bit 4i, value 2i+1 at bit 16+4i).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class MoEConfig:
    """Shapes of one MoE layer call (names follow the pages' notation)."""

    name: str
    T: int          # tokens in the batch
    D: int          # hidden size
    E: int          # routed experts
    I: int          # expert intermediate size
    Is: int         # shared-expert intermediate size
    k: int          # experts per token
    quant: int = 0  # 0 = bf16 weights, 1 = W4A16 (int4 group-quantised)
    group: int = 128  # W4A16 scale group along K; 0 = channel-wise (one scale per row)
    zipf_s: float = 0.0     # > 0: add a log-Zipf router bias
    zipf_alpha: float = 0.0  # scale of that bias
    seed: int = 0
    extra: dict = field(default_factory=dict, compare=False)

    @property
    def P(self) -> int:
        return self.T * self.k

    def with_(self, **kw) -> "MoEConfig":
        return replace(self, **kw)


# The five synthetic workloads.  The skewed bias scale was calibrated with
# oracle/calibrate_zipf.py on the seed-0 inputs (19.7% of experts empty).
CONFIGS = {
    "tiny": MoEConfig("tiny", T=64, D=256, E=16, I=128, Is=128, k=2),
    "decode": MoEConfig("decode", T=64, D=4096, E=512, I=1024, Is=1024, k=10),
    "prefill": MoEConfig("prefill", T=1024, D=4096, E=512, I=1024, Is=1024, k=10),
    "skewed": MoEConfig("skewed", T=8192, D=4096, E=512, I=1024, Is=1024, k=10,
                        zipf_s=1.2, zipf_alpha=0.9492),
    "w4a16": MoEConfig("w4a16", T=1024, D=4096, E=512, I=1024, Is=1024, k=10, quant=1,
                       group=128),
    # Same per-expert shapes as "decode" with 64 experts (1.6 GB of weights): the
    # case the detailed hardware-counter captures run on.
    "decode_e64": MoEConfig("decode_e64", T=64, D=4096, E=64, I=1024, Is=1024, k=10),
    # bf16 with ~20 token rows per expert (as in the T=1024 prefill) on 64 experts
    # (1.6 GB of weights): the hardware-counter capture case of the prefill shape.
    "prefill_e64": MoEConfig("prefill_e64", T=128, D=4096, E=64, I=1024, Is=1024, k=10),
    # W4A16 with ~20 token rows per expert (as in the T=1024 prefill) on 64 experts
    # (0.42 GB of packed weights): the W4A16 hardware-counter capture case.
    "w4a16_e64": MoEConfig("w4a16_e64", T=128, D=4096, E=64, I=1024, Is=1024, k=10, quant=1),
    # W4A16 at the decode batch (T=64): ~370 touched experts, 1-6 rows each.
    "w4a16_decode": MoEConfig("w4a16_decode", T=64, D=4096, E=512, I=1024, Is=1024, k=10,
                              quant=1, group=128),
    # W4A16 with channel-wise scales (one bf16 scale per output row), the release
    # note's other supported scale strategy, at the prefill batch.
    "w4a16_channel": MoEConfig("w4a16_channel", T=1024, D=4096, E=512, I=1024, Is=1024, k=10,
                               quant=1, group=0),
    # Compute-bound grouped GEMM: T=8192 on 64 experts, ~1280 rows per expert
    # (256-row token tiles), where the tensor pipe rather than HBM bounds the GEMMs.
    "dense_e64": MoEConfig("dense_e64", T=8192, D=4096, E=64, I=1024, Is=1024, k=10),
    # W4A16 on the compute-bound shape (T=8192 on 64 experts, 256-row token
    # tiles): the case of the W4A16 kernel that restores into shared memory.
    "w4a16_dense_e64": MoEConfig("w4a16_dense_e64", T=8192, D=4096, E=64, I=1024, Is=1024,
                                 k=10, quant=1, group=128),
    # Zipf-biased routing at T=2048 (256-row token tiles) on 64 experts (1.6 GB of
    # weights): the hardware-counter capture case of the skewed kernel shape.
    "skewed_e64": MoEConfig("skewed_e64", T=2048, D=4096, E=64, I=1024, Is=1024, k=10,
                            zipf_s=1.2, zipf_alpha=0.9492),
}

_TAG_X, _TAG_WR, _TAG_RANK = 1, 2, 3
_TAG_EXPERT = 1000
_TAG_SHARED = 900_000


def _gen(seed: int, tag: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + tag) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def normal_bf16(shape, std: float, seed: int, tag: int, device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in fp32 on ``device`` and rounded to bf16."""
    g = _gen(seed, tag, device)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return (v * std).to(torch.bfloat16)


def zipf_bias(E: int, s: float, alpha: float, seed: int) -> torch.Tensor:
    """fp32 [E]: alpha * log Zipf_s(rank_e) with ranks a seeded permutation of 1..E."""
    g = _gen(seed, _TAG_RANK, "cpu")
    ranks = torch.randperm(E, generator=g).to(torch.float64) + 1.0
    h = sum(r ** (-s) for r in range(1, E + 1))
    logp = -s * torch.log(ranks) - math.log(h)
    return (alpha * logp).to(torch.float32)


# Bit position of value j (0..7) of a packed int32: pairs (2i, 2i+1) at bits 4i and 16+4i.
PACK_SHIFTS = (0, 16, 4, 20, 8, 24, 12, 28)


def quantize_w4(w: torch.Tensor, group: int = 128):
    """Symmetric int4, one bf16 scale per ``group`` consecutive K values
    (group 0: channel-wise, one scale per row).

    w: [..., R, C] bf16.  Returns (q [..., R, C/8] int32, s [..., R, C/group] bf16,
    or s [..., R] when group is 0) with s = bf16(absmax / 7),
    q = clamp(round_half_even(w / s), -8, 7) (q = 0 where s = 0).  Pair order
    within each int32: value 2i of the group of 8 in bits [4i, 4i+4), value 2i+1
    in bits [16+4i, 20+4i).
    """
    *lead, R, C = w.shape
    g = C if group == 0 else group
    assert C % g == 0 and C % 8 == 0
    wf = w.to(torch.float32).reshape(*lead, R, C // g, g)
    s = (wf.abs().amax(dim=-1) / 7.0).to(torch.bfloat16)
    sf = s.to(torch.float32).unsqueeze(-1)
    safe = torch.where(sf == 0, torch.ones_like(sf), sf)
    q = torch.round(wf / safe).clamp_(-8, 7)
    q = torch.where(sf == 0, torch.zeros_like(q), q).to(torch.int32)
    q = q.reshape(*lead, R, C // 8, 8) & 0xF
    shifts = torch.tensor(PACK_SHIFTS, device=w.device, dtype=torch.int32)
    packed = torch.zeros((*lead, R, C // 8), dtype=torch.int64, device=w.device)
    packed = (q.to(torch.int64) << shifts.to(torch.int64)).sum(dim=-1)
    packed = torch.where(packed >= 2**31, packed - 2**32, packed).to(torch.int32)
    return packed, (s.squeeze(-1) if group == 0 else s)


@dataclass
class MoEInputs:
    cfg: MoEConfig
    x: torch.Tensor             # bf16 [T, D]
    w_router: torch.Tensor      # bf16 [E, D]
    bias: torch.Tensor | None   # fp32 [E] or None
    w_gate_up: torch.Tensor     # bf16 [E, 2I, D] or int32 [E, 2I, D/8]
    w_down: torch.Tensor        # bf16 [E, D, I] or int32 [E, D, I/8]
    s_gate_up: torch.Tensor | None   # bf16 [E, 2I, D/group]
    s_down: torch.Tensor | None      # bf16 [E, D, I/group]
    ws_gate_up: torch.Tensor    # shared expert, same formats with Is
    ws_down: torch.Tensor
    ss_gate_up: torch.Tensor | None
    ss_down: torch.Tensor | None

    def to(self, device) -> "MoEInputs":
        def mv(t):
            return None if t is None else t.to(device)
        return MoEInputs(self.cfg, *(mv(getattr(self, f)) for f in (
            "x", "w_router", "bias", "w_gate_up", "w_down", "s_gate_up", "s_down",
            "ws_gate_up", "ws_down", "ss_gate_up", "ss_down")))


def expert_weights_bf16(cfg: MoEConfig, e: int, device="cpu"):
    """bf16 (gate_up [2I, D], down [D, I]) of routed expert e (e == E: the shared one)."""
    Ie = cfg.Is if e == cfg.E else cfg.I
    tag = _TAG_SHARED if e == cfg.E else _TAG_EXPERT + 2 * e
    gu = normal_bf16((2 * Ie, cfg.D), 1.0 / math.sqrt(cfg.D), cfg.seed, tag, device)
    dn = normal_bf16((cfg.D, Ie), 1.0 / math.sqrt(Ie), cfg.seed, tag + 1, device)
    return gu, dn


def tokens(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    """The batch's token rows x: bf16 [T, D] ~ N(0, 1), drawn on the CPU."""
    return normal_bf16((cfg.T, cfg.D), 1.0, cfg.seed, _TAG_X, "cpu").to(device)


def with_tokens(inp: MoEInputs, cfg: MoEConfig) -> MoEInputs:
    """Inputs of ``cfg``, a configuration that differs from ``inp.cfg`` only in
    the token count T and the router bias: the same router and expert weights
    (the expert weights depend on (seed, E, D, I, Is, quant, group) only), fresh
    token rows and the bias of ``cfg`` (as make_inputs draws them)."""
    same = ("D", "E", "I", "Is", "k", "quant", "group", "seed")
    if any(getattr(cfg, f) != getattr(inp.cfg, f) for f in same):
        raise ValueError(f"{cfg.name} differs from {inp.cfg.name} in more than T and the bias")
    dev = inp.x.device
    bias = zipf_bias(cfg.E, cfg.zipf_s, cfg.zipf_alpha, cfg.seed).to(dev) if cfg.zipf_s > 0 else None
    return replace(inp, cfg=cfg, x=tokens(cfg, dev), bias=bias)


def make_inputs(cfg: MoEConfig, device="cpu", weight_device=None) -> MoEInputs:
    """All inputs of one layer call.

    ``x``, the router weight and the bias are drawn on the CPU (so they do not
    depend on the device); expert weights are drawn on ``weight_device``
    (default: ``device``), one expert at a time.
    """
    wdev = torch.device(weight_device if weight_device is not None else device)
    x = tokens(cfg)
    wr = normal_bf16((cfg.E, cfg.D), 0.02, cfg.seed, _TAG_WR, "cpu")
    bias = zipf_bias(cfg.E, cfg.zipf_s, cfg.zipf_alpha, cfg.seed) if cfg.zipf_s > 0 else None

    def alloc(shape, dtype):
        return torch.empty(shape, dtype=dtype, device=wdev)

    E, D, I, Is, G = cfg.E, cfg.D, cfg.I, cfg.Is, cfg.group
    if cfg.quant == 0:
        w_gu, w_dn = alloc((E, 2 * I, D), torch.bfloat16), alloc((E, D, I), torch.bfloat16)
        s_gu = s_dn = None
    else:
        w_gu, w_dn = alloc((E, 2 * I, D // 8), torch.int32), alloc((E, D, I // 8), torch.int32)
        if G == 0:  # channel-wise: one scale per output row
            s_gu, s_dn = alloc((E, 2 * I), torch.bfloat16), alloc((E, D), torch.bfloat16)
        else:
            s_gu = alloc((E, 2 * I, D // G), torch.bfloat16)
            s_dn = alloc((E, D, I // G), torch.bfloat16)
    for e in range(E):
        gu, dn = expert_weights_bf16(cfg, e, wdev)
        if cfg.quant == 0:
            w_gu[e].copy_(gu)
            w_dn[e].copy_(dn)
        else:
            q, s = quantize_w4(gu, G)
            w_gu[e].copy_(q)
            s_gu[e].copy_(s)
            q, s = quantize_w4(dn, G)
            w_dn[e].copy_(q)
            s_dn[e].copy_(s)
    gu, dn = expert_weights_bf16(cfg, E, wdev)
    if cfg.quant == 0:
        ws_gu, ws_dn, ss_gu, ss_dn = gu, dn, None, None
    else:
        ws_gu, ss_gu = quantize_w4(gu, G)
        ws_dn, ss_dn = quantize_w4(dn, G)
    dev = torch.device(device)
    return MoEInputs(cfg, x.to(dev), wr.to(dev), None if bias is None else bias.to(dev),
                     w_gu, w_dn, s_gu, s_dn, ws_gu, ws_dn, ss_gu, ss_dn)


def as_u16(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")
