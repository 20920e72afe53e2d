"""Benchmark of the MoE layer forward: decode step (T=64, D=4096, E=512, I=1024,
top-10) as the headline, and every other synthetic workload beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Prints ONE JSON line (rank 0).  A step is one pass of the whole hot path
(router -> dispatch -> grouped gate/up -> grouped down -> combine, shared
expert included) over one batch of synthetic input, through the C ABI.

  value     tokens/s of moe_forward with every input resident in HBM (K steps
            timed with CUDA events between a barrier + synchronize on both sides;
            the touched expert weights, ~9.3 GB per step, exceed L2, so no flush).
  e2e       the same metric through moe_forward_host: pinned host x copied in and
            y copied out inside every timed step.
  roofline  the dominant kernel (grouped gate/up GEMM): algorithmic bytes per
            launch / its mean CUDA-event duration inside a timed pass of the
            path split into its ABI calls, against the measured HBM copy peak.
  cpu_baseline  the fp64 oracle on this host's cores over the same batch (at
            most its first 1024 tokens).
  graph_ms_per_step  the same step captured once into a CUDA graph and
            replayed (no host launch cost).
  configs   the same measurements for the other workloads: the T=1024 prefill
            chunk (the metric's second configuration) and the skewed T=8192
            batch on the same expert weights, the tiny layer, W4A16 at T=1024
            (group and channel-wise scales) and T=64, and the compute-bound
            T=8192 batch on 64 experts.  A workload whose kernels record a
            device error carries "error" instead of numbers.

After warm-up, after the timed steps, after the split pass and after the e2e
steps the workspace status words are read: a kernel that recorded a device
error (a bounded wait that gave up) fails the run instead of being timed.

With --gpus N > 1 (launched by torch.distributed.run) every rank runs an
independent replica of the layer on its own GPU (the path has no exchange step
on one device); value = all ranks' tokens / the slowest rank's time.
``--impl reference`` times the fp64 oracle (the CPU reference) on the same
workload and metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (T=64 decode, T=1024 prefill) and % of HBM/BF16 roofline"
# ncu DRAM counters of the decode gate/up launch with the hash of the kernel
# sources they were taken with (machine-readable; the .md beside it explains them)
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "grouped_gemm_gate_up_decode.json")
NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e nominal (context for the measured-copy fraction)
GEMM_SOURCES = [os.path.join(ROOT, "sparse_moe_layer_router_gb300", "csrc", f)
                for f in ("grouped_gemm.cu", "common.cuh")]
L2_BYTES = 129 * 2**20
# Measured beside the decode headline, in this order (the first two reuse the
# decode expert weights; the W4A16 decode batch reuses the W4A16 weights).
EXTRA_WORKLOADS = ("prefill", "skewed", "tiny", "w4a16", "w4a16_decode", "w4a16_channel",
                   "dense_e64", "w4a16_dense_e64")
ORACLE_SAMPLE_TOKENS = 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", default="decode")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--decode-only", action="store_true",
                    help="with the default decode workload, skip the other workloads")
    ap.add_argument("--extra", default=",".join(EXTRA_WORKLOADS),
                    help="comma-separated workloads measured beside the decode headline")
    return ap.parse_args()


def workload_desc(cfg):
    d = (f"{cfg.name}: T={cfg.T}, D={cfg.D}, E={cfg.E}, I={cfg.I}, Is={cfg.Is}, top-{cfg.k}, "
         f"{('W4A16 int4 ' + ('channel-wise' if cfg.group == 0 else f'g{cfg.group}')) if cfg.quant else 'bf16'} weights")
    if cfg.zipf_s:
        d += f", log-Zipf(s={cfg.zipf_s}) router bias x{cfg.zipf_alpha}"
    return d


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, enabled=True):
        self.proc = None
        self.path = None
        self.gpu = gpu_index
        if not enabled:
            return
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5], f[6], f[7], f[8], f[4]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        sm = [r[0] for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------ helpers
def slowest_rank(x, world, device):
    """The largest of every rank's ``x`` (a duration): the job runs as long as its
    slowest replica.  One rank: ``x`` itself."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, tokens_per_rank_step, steps, seconds):
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank_step * steps / seconds


def scales_per_row(cfg, K):
    """bf16 scales per weight row of length K: K / group, or 1 (channel-wise, group 0)."""
    return 1 if cfg.group == 0 else K // cfg.group


def touched_gate_up_bytes(cfg, counts):
    """Algorithmic HBM bytes of one grouped gate/up launch: every touched expert's
    gate/up weights (and scales) once, the shared expert's, the token rows read
    and the hidden rows written."""
    import torch
    touched = int((counts > 0).sum().item())
    P = cfg.T * cfg.k
    if cfg.quant == 0:
        w_exp = 2 * cfg.I * cfg.D * 2
        w_sh = 2 * cfg.Is * cfg.D * 2
    else:
        w_exp = 2 * cfg.I * cfg.D // 2 + 2 * cfg.I * scales_per_row(cfg, cfg.D) * 2
        w_sh = 2 * cfg.Is * cfg.D // 2 + 2 * cfg.Is * scales_per_row(cfg, cfg.D) * 2
    act = P * cfg.D * 2 + cfg.T * cfg.D * 2 + P * cfg.I * 2 + cfg.T * cfg.Is * 2
    del torch
    return touched * w_exp + w_sh + act, touched


def layer_bytes_flops(cfg, touched):
    """Algorithmic bytes / flops of one layer forward (touched weights + router + x + y)."""
    if cfg.quant == 0:
        per_exp = 3 * cfg.I * cfg.D * 2
        sh = 3 * cfg.Is * cfg.D * 2
    else:
        # gate/up rows of length D and down rows of length I (or Is)
        per_exp = (3 * cfg.I * cfg.D // 2 + 2 * cfg.I * scales_per_row(cfg, cfg.D) * 2
                   + cfg.D * scales_per_row(cfg, cfg.I) * 2)
        sh = (3 * cfg.Is * cfg.D // 2 + 2 * cfg.Is * scales_per_row(cfg, cfg.D) * 2
              + cfg.D * scales_per_row(cfg, cfg.Is) * 2)
    byts = touched * per_exp + sh + cfg.E * cfg.D * 2 + 2 * cfg.T * cfg.D * 2
    flops = (2 * cfg.T * cfg.D * cfg.E + 6 * cfg.T * cfg.k * cfg.D * cfg.I
             + 6 * cfg.T * cfg.D * cfg.Is)
    return byts, flops


def gate_up_flops(cfg):
    """Tensor-core flops of one grouped gate/up launch (routed pairs + shared rows)."""
    return 2 * cfg.T * cfg.k * cfg.D * 2 * cfg.I + 2 * cfg.T * cfg.D * 2 * cfg.Is


def profile_traffic():
    """(traffic bytes per decode gate/up launch, source) from the committed ncu
    counters, or (None, why) when the kernel sources changed since they were taken."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None, "no committed ncu counters"
    d = json.load(open(PROFILE_TRAFFIC))
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        h.update(open(f, "rb").read())
    if h.hexdigest() != d.get("source_sha256"):
        return None, "kernel changed since the ncu capture"
    return int(d["traffic_bytes_per_launch"]), "ncu"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------ oracle leg
def oracle_pass(cfg, rows, host_x, host_wr, host_bias, experts, shared):
    """The oracle's layer over the token rows ``rows``: routing, then the forward."""
    import oracle
    x = host_x[rows]
    ids, w = oracle.route(x, host_wr, cfg.k, host_bias)
    return oracle.forward(x, ids, w, experts, shared, E=cfg.E, I=cfg.I, Is=cfg.Is,
                          quant=cfg.quant, group=cfg.group)


def oracle_host_inputs(inp, n_tokens=None):
    """Host copies of the inputs (the first ``n_tokens`` token rows, default all)
    and of every expert those rows touch."""
    import numpy as np
    import oracle
    from sparse_moe_layer_router_gb300.synthetic import as_u16
    cfg = inp.cfg
    x = as_u16(inp.x if n_tokens is None else inp.x[:n_tokens])
    wr = as_u16(inp.w_router)
    bias = None if inp.bias is None else inp.bias.cpu().numpy()
    ids, _ = oracle.route(x, wr, cfg.k, bias)

    def one(e):
        if e == cfg.E:
            t = (inp.ws_gate_up, inp.ws_down, inp.ss_gate_up, inp.ss_down)
        else:
            t = (inp.w_gate_up[e], inp.w_down[e],
                 None if inp.s_gate_up is None else inp.s_gate_up[e],
                 None if inp.s_down is None else inp.s_down[e])
        if cfg.quant == 0:
            return as_u16(t[0]), as_u16(t[1])
        return t[0].cpu().numpy(), as_u16(t[2]), t[1].cpu().numpy(), as_u16(t[3])

    experts = {int(e): one(int(e)) for e in np.unique(ids)}
    return x, wr, bias, experts, one(cfg.E)


def cpu_baseline(cfg, inputs, min_seconds=10.0, max_passes=20):
    """Oracle passes over the sampled token rows (all rows of ``inputs``) until
    ``min_seconds`` of CPU work: (tokens/s, cores, passes, rows per pass)."""
    import numpy as np
    import oracle
    rows = np.arange(inputs[0].shape[0])
    done, t0 = 0, time.perf_counter()
    while True:
        oracle_pass(cfg, rows, *inputs)
        done += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or done >= max_passes:
            return len(rows) * done / dt, oracle.num_threads(), done, len(rows)


def run_reference(args, cfg, base_config, local):
    """The reference arm: the fp64 oracle on the host cores, K timed steps of a
    bounded token sample each (rotating through the batch)."""
    import numpy as np
    import torch
    import oracle
    from sparse_moe_layer_router_gb300.synthetic import make_inputs
    oracle.build()
    wdev = f"cuda:{local}" if torch.cuda.is_available() else "cpu"
    inp = make_inputs(cfg, device="cpu", weight_device=wdev)
    inputs = oracle_host_inputs(inp)
    del inp
    if torch.cuda.is_available():
        torch.cuda.empty_cache()
    cores = oracle.num_threads()
    # size the per-step sample so that K + W steps take about two minutes
    n0 = min(cfg.T, cores)
    t1 = time.perf_counter()
    oracle_pass(cfg, np.arange(n0), *inputs)
    per_tok = (time.perf_counter() - t1) / n0
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(cfg.T, budget / max(per_tok, 1e-9))))
    W = max(3, args.warmup)

    def rows(i):
        return (np.arange(n) + i * n) % cfg.T

    for i in range(W):
        oracle_pass(cfg, rows(i), *inputs)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_pass(cfg, rows(W + i), *inputs)
    dt = time.perf_counter() - t0
    val = n * args.steps / dt
    return {"metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": W, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; random-init weights of the stated shapes)",
            "config": base_config, "impl": "reference",
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{n} of the batch's {cfg.T} tokens per step (routing + "
                                       f"layer, fp64), rotating through the batch"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ GPU leg
class DeviceError(RuntimeError):
    pass


def check_status(B, ws, what):
    """Fail the run if a kernel recorded a device-side error (a wait that gave
    up stops issuing work, so its step would be timed as if it had run)."""
    st = B.get_status(ws)
    if st != B.MOE_OK:
        raise DeviceError(f"device status {st} ({B.strerror(st)}) after {what}")


def measure(cfg, inp, args, world, rank, dev, clocks_on, hbm_peak, bf16_peak, peak_src,
            with_traffic):
    """One workload: K timed moe_forward steps, the path split into its ABI calls
    (per-call CUDA events), e2e through moe_forward_host, and the oracle baseline."""
    import torch
    from sparse_moe_layer_router_gb300 import binding as B

    stream = torch.cuda.current_stream()
    ws = B.workspace(cfg, B.MOE_ENTRY_FORWARD, dev)
    y = torch.empty((cfg.T, cfg.D), dtype=torch.bfloat16, device=dev)
    W = B.weights_struct(inp, cfg)

    def step():
        B.forward(cfg, inp.x, W, y=y, ws=ws)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    check_status(B, ws, "warm-up")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    # ---------------- timed region: K steps of moe_forward
    clocks = ClockSampler(dev.index, enabled=clocks_on)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    barrier()
    ms_total = e0.elapsed_time(e1)
    clk = clocks.stop()
    check_status(B, ws, "the timed steps")
    ms_total = slowest_rank(ms_total, world, dev)
    ms_step = ms_total / args.steps
    value = job_tokens_per_s(world, cfg.T, args.steps, ms_total / 1e3)

    # ---------------- the same step replayed from a CUDA graph (captured once):
    # no host launch cost, which is what bounds the tiny layer
    graph_ms = None
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    barrier()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    kg = max(10, args.steps // 3)
    g0.record()
    for _ in range(kg):
        graph.replay()
    g1.record()
    barrier()
    check_status(B, ws, "the graph replays")
    graph_ms = slowest_rank(g0.elapsed_time(g1), world, dev) / kg
    del graph
    launches_per_step = step_launches(cfg)

    # ---------------- the path split into its ABI calls, events around each call
    blob = torch.empty((cfg.T, 2, cfg.k), dtype=torch.int32, device=dev)
    ws_r = B.workspace(cfg, B.MOE_ENTRY_ROUTE, dev)
    ws_p = B.workspace(cfg, B.MOE_ENTRY_PERMUTE, dev)
    ws_g = B.workspace(cfg, B.MOE_ENTRY_GROUPED_GEMM, dev)
    P = cfg.T * cfg.k
    perm_out = (torch.empty(cfg.E, dtype=torch.int32, device=dev),
                torch.empty(cfg.E + 1, dtype=torch.int32, device=dev),
                torch.empty(P, dtype=torch.int32, device=dev),
                torch.empty(P, dtype=torch.int32, device=dev))
    xp = torch.empty((P, cfg.D), dtype=torch.bfloat16, device=dev)
    h = torch.empty((P, cfg.I), dtype=torch.bfloat16, device=dev)
    hs = torch.empty((cfg.T, cfg.Is), dtype=torch.bfloat16, device=dev)
    o = torch.empty((P, cfg.D), dtype=torch.float32, device=dev)
    os_ = torch.empty((cfg.T, cfg.D), dtype=torch.float32, device=dev)
    y2 = torch.empty_like(y)
    names = ["route", "permute", "gate_up", "down", "combine"]

    def split_step(ev):
        ev[0].record(stream)
        B.route(cfg, inp.x, inp.w_router, inp.bias, blob=blob, ws=ws_r)
        ev[1].record(stream)
        counts, offsets, perm, inv = B.permute(cfg, blob, ws=ws_p, x=inp.x, x_perm=xp, out=perm_out)
        ev[2].record(stream)
        B.grouped_gemm(cfg, B.MOE_OP_GATE_UP_SWIGLU, xp, offsets, inp.w_gate_up, h,
                       w_scales=inp.s_gate_up, a_shared=inp.x, w_shared=inp.ws_gate_up,
                       ws_scales=inp.ss_gate_up, out_shared=hs, ws=ws_g)
        ev[3].record(stream)
        B.grouped_gemm(cfg, B.MOE_OP_DOWN_WEIGHTED, h, offsets, inp.w_down, o,
                       w_scales=inp.s_down, perm_pair=perm, blob=blob, a_shared=hs,
                       w_shared=inp.ws_down, ws_scales=inp.ss_down, out_shared=os_, ws=ws_g)
        ev[4].record(stream)
        B.combine(cfg, o, os_, inv, y=y2)
        ev[5].record(stream)

    ksplit = max(10, min(args.steps, 100))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(ksplit)]
    for _ in range(3):
        split_step(evs[0])
    barrier()
    for i in range(ksplit):
        split_step(evs[i])
    barrier()
    for w_, what in ((ws_r, "route"), (ws_p, "permute"), (ws_g, "the grouped GEMMs")):
        check_status(B, w_, f"the split pass ({what})")
    per = {n: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(ksplit)) / ksplit
           for j, n in enumerate(names)}
    split_total = sum(evs[i][0].elapsed_time(evs[i][5]) for i in range(ksplit)) / ksplit
    same = bool(torch.equal(y, y2))
    refined = int(ws_r[4:8].view(torch.int32).item())
    exact = int(ws_r[8:12].view(torch.int32).item())

    counts = perm_out[0]
    gu_bytes, touched = touched_gate_up_bytes(cfg, counts)
    gu_ms = per["gate_up"]
    achieved = gu_bytes / (gu_ms / 1e3) / 1e9
    gu_tflops = gate_up_flops(cfg) / (gu_ms / 1e3) / 1e12
    traffic, traffic_src = profile_traffic() if with_traffic else (None, "not captured")
    roofline = {"bound": "hbm", "kernel": "grouped_gemm gate/up + SwiGLU (tcgen05)",
                "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "peak_source": f"{peak_src} (HBM copy, burst)",
                "frac_of_nominal_hbm": achieved / NOMINAL_HBM_GBS,
                "tensor_tflops": gu_tflops, "tensor_frac": gu_tflops / bf16_peak,
                "traffic": traffic, "traffic_source": traffic_src,
                "algorithmic_bytes_per_launch": gu_bytes, "touched_experts": touched,
                "mean_launch_ms": gu_ms}
    lay_bytes, lay_flops = layer_bytes_flops(cfg, touched)
    layer = {"algorithmic_bytes": lay_bytes, "algorithmic_flops": lay_flops,
             "hbm_frac": lay_bytes / (ms_step / 1e3) / 1e9 / hbm_peak,
             "tensor_frac": lay_flops / (ms_step / 1e3) / 1e12 / bf16_peak,
             "binding_frac": max(lay_bytes / (hbm_peak * 1e9), lay_flops / (bf16_peak * 1e12))
             / (ms_step / 1e3),
             "per_call_ms": per, "split_step_ms": split_total, "split_matches_forward": same,
             "router_refined_tokens": refined, "router_exact_fallback_tokens": exact}
    del xp, h, hs, o, os_, ws_r, ws_p, ws_g

    # ---------------- e2e: host buffers through moe_forward_host
    e2e = None
    if not args.no_e2e:
        ws_h = B.workspace(cfg, B.MOE_ENTRY_FORWARD_HOST, dev)
        xh = inp.x.cpu().pin_memory()
        yh = torch.empty((cfg.T, cfg.D), dtype=torch.bfloat16).pin_memory()
        for _ in range(3):
            B.forward_host(cfg, xh, W, yh, ws_h)
        torch.cuda.synchronize()
        ke = max(10, args.steps // 3)
        barrier()
        t0 = time.perf_counter()
        for _ in range(ke):
            B.forward_host(cfg, xh, W, yh, ws_h)
            stream.synchronize()  # the step's result is on the host
        barrier()
        dt = time.perf_counter() - t0
        check_status(B, ws_h, "the e2e steps")
        dt = slowest_rank(dt, world, dev)
        e2e = {"value": job_tokens_per_s(world, cfg.T, ke, dt), "unit": "tokens/s",
               "h2d_bytes_per_step": cfg.T * cfg.D * 2, "d2h_bytes_per_step": cfg.T * cfg.D * 2,
               "ms_per_step": 1e3 * dt / ke, "steps": ke,
               "same_output_as_device_path": bool(torch.equal(yh, y.cpu()))}
        del ws_h

    # ---------------- CPU baseline: the oracle on this host's cores (rank 0 only, N = 1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        inputs = oracle_host_inputs(inp, min(cfg.T, ORACLE_SAMPLE_TOKENS))
        val, cores, passes, n = cpu_baseline(cfg, inputs)
        what = (f"the full {cfg.name} batch ({cfg.T} tokens" if n == cfg.T
                else f"the first {n} of the {cfg.name} batch's {cfg.T} tokens (")
        cpu = {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{what}{'; ' if n == cfg.T else ''}fp64 routing + layer) "
                         f"x{passes} passes"}
        del inputs
    del ws, y
    return {"value": value, "ms_per_step": ms_step, "graph_ms_per_step": graph_ms,
            "roofline": roofline, "layer": layer,
            "e2e": e2e, "cpu_baseline": cpu, "clocks": clk,
            "gpu_launches": launches_per_step * args.steps, "workload": workload_desc(cfg)}


def step_launches(cfg):
    """Kernel launches of one moe_forward: sums of squares, logits, select,
    dispatch (one block up to 4096 pairs, else count + scan + scatter), gather,
    two GEMMs, combine.  A bf16 GEMM with 256-row token tiles and under 512 rows
    per expert on average adds a plan kernel and a second grid (the hot/cold
    split)."""
    n = 8 if cfg.T * cfg.k <= 4096 else 10
    tiles256 = cfg.T >= 2048 or cfg.T * cfg.k >= 48 * cfg.E
    if cfg.quant == 0 and tiles256 and cfg.T * cfg.k < 512 * cfg.E:
        n += 4
    return n


def measure_extra(names, inp, args, world, rank, dev, hbm_peak, bf16_peak, peak_src):
    """The workloads beside the headline, one after the other.  Inputs that share
    expert weights with the previous ones (same D, E, I, Is, k, quant, group) reuse
    them with fresh token rows and router bias; others are drawn anew."""
    import torch
    from sparse_moe_layer_router_gb300.synthetic import CONFIGS, make_inputs, with_tokens
    same = ("D", "E", "I", "Is", "k", "quant", "group", "seed")
    out = {}
    cur = inp
    for name in names:
        cfg = CONFIGS[name]
        if all(getattr(cfg, f) == getattr(cur.cfg, f) for f in same):
            w = with_tokens(cur, cfg)
        else:
            cur = w = None
            torch.cuda.empty_cache()
            cur = w = make_inputs(cfg, device=dev)
        try:
            r = measure(cfg, w, args, world, rank, dev, not args.no_clocks, hbm_peak, bf16_peak,
                        peak_src, with_traffic=False)
        except DeviceError as e:
            out[name] = {"config": {"workload": workload_desc(cfg)}, "error": str(e)}
            continue
        lay = r["layer"]["algorithmic_bytes"]
        l2 = ("no flush: the touched expert weights streamed each step exceed L2 (129 MB)"
              if lay > L2_BYTES else
              f"no flush: the whole layer's {lay / 2**20:.1f} MiB fit in L2 (launch-bound)")
        out[name] = {"metric": METRIC, "unit": "tokens/s", "steps": args.steps,
                     "config": {"workload": r.pop("workload"), "T": cfg.T, "l2": l2}, **r}
    return out


# ------------------------------------------------------------------ main
def main():
    args = parse()
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if args.impl == "gb300" else "gloo")

    from sparse_moe_layer_router_gb300.build import build
    from sparse_moe_layer_router_gb300.synthetic import CONFIGS, make_inputs, with_tokens

    cfg = CONFIGS[args.config]
    hbm_peak, bf16_peak, peak_src = peaks()
    base_config = {"workload": workload_desc(cfg), "T": cfg.T, "D": cfg.D, "E": cfg.E,
                   "I": cfg.I, "Is": cfg.Is, "k": cfg.k, "quant": cfg.quant,
                   "parallelism": f"replicas x{args.gpus}",
                   "l2": "no flush: the touched expert weights streamed each step exceed L2 (129 MB)",
                   "seed": cfg.seed}

    if args.impl == "reference":
        if rank == 0:
            line = run_reference(args, cfg, base_config, local)
            print(json.dumps(line), flush=True)
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    torch.cuda.set_device(local)
    build()
    dev = torch.device("cuda", local)
    inp = make_inputs(cfg, device=dev)
    head = measure(cfg, inp, args, world, rank, dev, not args.no_clocks, hbm_peak, bf16_peak,
                   peak_src, with_traffic=args.config == "decode")
    extra = {}
    if args.config == "decode" and not args.decode_only:
        names = [n for n in args.extra.split(",") if n]
        extra = measure_extra(names, inp, args, world, rank, dev, hbm_peak, bf16_peak, peak_src)

    if rank == 0:
        line = {"metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": max(3, args.warmup),
                "ms_per_step": head["ms_per_step"], "graph_ms_per_step": head["graph_ms_per_step"],
                "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic (seeded; random-init weights of the stated shapes)",
                "config": base_config, "roofline": head["roofline"],
                "cpu_baseline": head["cpu_baseline"], "e2e": head["e2e"],
                "gpu_launches": head["gpu_launches"], "clocks": head["clocks"],
                "layer": head["layer"], "impl": "gb300"}
        if extra:
            line["configs"] = extra
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
