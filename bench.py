"""Benchmark of the per-layer MoE expert hot path (libspx) on one GB300.

One step = one 26-layer DeepSeek-V2-Lite-shaped draft-then-verify cycle (the
largest single-GPU workload): K = 16 draft steps at T = 1 through all 26 layers
(fused INT4 experts, the lookahead counters on), then one verify pass at
T = K+1 = 17 through all 26 layers (expert-reordered FP16 experts); every
layer is the full chain route -> top-k -> counters -> gather -> experts ->
shared expert -> combine through spx_moe_layer.  Independent seeded weights per
layer (37 GB) are generated on the device, so no layer finds its weights in the
126 MB L2.

value = algorithmic HBM bytes of a cycle / device time of a cycle (GB/s): the
unique routed experts of every call (INT4 for the draft, FP16 for the verify,
from the library's own routing), the FP16 shared expert of every call,
activations, logits and outputs.  The same line carries per-layer figures of
the three single-layer shapes (DeepSeek-V2-Lite, Qwen1.5-MoE, Phi-3.5-MoE;
draft T = 1 and verify T = K+1), each timed as a chain of back-to-back calls.

``--impl reference`` times the CPU oracle (test infrastructure, single core)
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import spx_workloads as W  # noqa: E402

METRIC = "MoE layer µs & achieved HBM GB/s vs GB300 peak, draft T=1 / verify T=K+1"
CYCLE = "deepseek_v2_lite_x26"
GATE_CONFIGS = ("deepseek_v2_lite", "qwen15_moe", "phi35_moe")
# DRAM bytes (read + write) of one launch from an ncu capture of
# `bench.py --loop draft|verify --sets 2` (DeepSeek-V2-Lite-shaped, input set
# 0), with that launch's algorithmic bytes and the hash of the kernel sources
# the capture ran.  traffic_of() returns the bytes only while the sources still
# hash the same; a changed kernel reports null until it is captured again.
KERNEL_SOURCES = {
    "draft": ["spx_draft.cu", "spx_draft_gguf.cuh", "spx_routing.cuh", "spx_internal.cuh"],
    "verify": ["spx_tc.cu", "spx_route.cu", "spx_routing.cuh", "spx_internal.cuh"],
}
PROFILED_TRAFFIC = {
    "verify": {"kernel": "tc_mlp_kernel", "dram_bytes": 677_542_912 + 3_924_480,
               "algorithmic_bytes": 674_897_920, "source_sha": "09a4a987efe1e0e7"},
    "draft": {"kernel": "draft_kernel<2,0>", "dram_bytes": 61_500_160 + 238_848, "algorithmic_bytes": 61_374_720,
              "source_sha": "b75136a8eb199793"},
}
NSETS = 8  # default; --sets overrides (profiling captures use fewer)
NINPUTS = 16


def source_sha(which):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[which]:
        with open(os.path.join(ROOT, "quantized_expert_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_of(which):
    """DRAM bytes per launch from the last capture, or None when the kernel's
    sources changed since (or no capture was recorded for them)."""
    t = PROFILED_TRAFFIC.get(which)
    if t is None or t["source_sha"] != source_sha(which):
        return None
    return t["dram_bytes"]


def traffic_note(which):
    t = PROFILED_TRAFFIC[which]
    if traffic_of(which) is None:
        return f"no ncu capture of the current {t['kernel']} sources"
    return (f"ncu dram__bytes_read.sum + dram__bytes_write.sum of one {t['kernel']} launch "
            f"(algorithmic {t['algorithmic_bytes']} B), sources {t['source_sha']}")


def spread_us(ms_list):
    """p10 / median / p90 of per-call times given in ms, in us (nearest rank)."""
    v = sorted(ms_list)
    if not v:
        return {"p10": None, "median": None, "p90": None}

    def rank(q):
        return v[min(len(v) - 1, max(0, int(round(q * (len(v) - 1)))))] * 1e3

    return {"p10": round(rank(0.1), 2), "median": round(statistics.median(v) * 1e3, 2), "p90": round(rank(0.9), 2)}


def job_throughput(tot_bytes, ms_total, device=None):
    """Whole-job GB/s: the bytes every rank processed over the slowest rank's
    device time (max over ranks), and that time in ms.  One process when
    torch.distributed is not initialised; otherwise all ranks must call it
    (tensors on `device`: the GPU under NCCL, the CPU under gloo)."""
    import torch
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        t_max = torch.tensor([float(ms_total)], dtype=torch.float64, device=device)
        b_sum = torch.tensor([float(tot_bytes)], dtype=torch.float64, device=device)
        dist.all_reduce(t_max, op=dist.ReduceOp.MAX)
        dist.all_reduce(b_sum, op=dist.ReduceOp.SUM)
        ms_total, tot_bytes = float(t_max.item()), float(b_sum.item())
    return tot_bytes / (ms_total * 1e-3) / 1e9, ms_total


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------------ bytes --
def w4_expert_bytes(s):
    return 3 * s.H * s.I // 2 + 2 * (s.H // 128) * s.I * 2 + (s.I // 128) * s.H * 2


def f16_expert_bytes(s, I=None):
    I = s.I if I is None else I
    return 3 * s.H * I * 2


def layer_bytes(s, mode, T, n_unique, zeros=False, gguf=None):
    if gguf == "q8_0":  # GGUF Q8_0: 34 bytes per 32 weights
        b = n_unique * 3 * s.H * s.I * 34 // 32
    elif gguf in ("q2_k", "q4_k"):  # K-quant gate/up as packed (84 or 148 bytes per 256 weights), Q8_0 down
        b = n_unique * (2 * s.H * s.I * (84 if gguf == "q2_k" else 148) // 256 + s.H * s.I * 34 // 32)
    else:
        b = n_unique * (w4_expert_bytes(s) if mode == "draft" else f16_expert_bytes(s))
    if zeros:  # fp16 zero points: one per group of 128 rows and column, of the three matrices
        b += n_unique * 2 * (3 * s.H * s.I // 128)
    if s.I_s:
        b += f16_expert_bytes(s, s.I_s) + (s.H * 2 if s.shared_gate else 0)
    if s.logits == "router":
        b += s.E * s.H * 2
    b += T * s.H * 2 * 2 + T * s.E * 4  # x in, out, logits
    return b


# ----------------------------------------------------------------- clocks --
class ClockSampler:
    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- workload ----
def make_weight_set(s, idx, torch, spx, tc_pack=False):
    """Random canonical weights on the device (seeded), repacked for the kernels
    (tc_pack: the FP16 verify weights also in the tile pack of the
    tensor-memory verify launches)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(1_000_003 * (s.seed + 1) + idx)
    E, H, I = s.E, s.H, s.I
    dev = "cuda"

    def codes(*shape):
        return torch.randint(-2 ** 31, 2 ** 31, shape, dtype=torch.int32, device=dev, generator=g)

    def scales(*shape):
        return (torch.rand(shape, device=dev, generator=g) * 0.015 + 0.005).half()

    def normal(*shape):
        return (torch.randn(shape, device=dev, generator=g) * 0.02).half()

    w4 = spx.spx_w4_repack(codes(E, H // 8, I), scales(E, H // 128, I), codes(E, H // 8, I),
                           scales(E, H // 128, I), codes(E, I // 8, H), scales(E, I // 128, H), slice_cols=32)
    f16 = spx.spx_f16_repack(normal(E, I, H), normal(E, I, H), normal(E, H, I), tc=tc_pack)
    sh = None
    if s.I_s:
        sh = spx.pack_shared(normal(s.I_s, H), normal(s.I_s, H), normal(H, s.I_s),
                             normal(H) if s.shared_gate else None, tc=tc_pack)
    wr = normal(E, H) if s.logits == "router" else None
    torch.cuda.synchronize()
    return dict(w4=w4, f16=f16, shared=sh, w_router=wr)


def make_inputs(s, i):
    Td, Tv = s.T_draft, s.T_verify
    d = dict(x_d=W.gen_x(s, Td, step=i, which=0), x_v=W.gen_x(s, Tv, step=i, which=1))
    if s.logits != "router":
        d["lg_d"] = W.gen_logits(s, Td, step=i, which=0)
        d["lg_v"] = W.gen_logits(s, Tv, step=i, which=1)
    return d


def run_mine(args):
    """The headline step: one 26-layer draft-then-verify cycle (K = 16 draft
    steps at T = 1 through every layer with the lookahead counters on, then one
    verify pass at T = 17), plus per-layer figures of the three single-layer
    shapes, all through spx_moe_layer."""
    import torch
    from quantized_expert_gb300 import build as spx_build
    from quantized_expert_gb300 import spx

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    if rank == 0 or world == 1:
        spx_build.build()
    if world > 1:
        dist.barrier()
    spx.load()
    peak, peak_src = measured_peaks()
    s = W.CONFIGS[CYCLE]
    L, K, E, k, H, Tv = s.layers, s.K, s.E, s.k, s.H, s.T_verify
    lays = [make_weight_set(s, l, torch, spx, tc_pack=True) for l in range(L)]
    stream = torch.cuda.Stream()

    def sync_all():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
            torch.cuda.synchronize()

    def ev():
        return torch.cuda.Event(enable_timing=True)

    # one cycle's inputs: host (pinned) and two device copies (e2e double buffer)
    host = {"xd": np.stack([[W.gen_x(s, 1, layer=l, step=st) for l in range(L)] for st in range(1, K + 1)]),
            "lgd": np.stack([[W.draft_logits(s, l, st) for l in range(L)] for st in range(1, K + 1)]),
            "xv": np.stack([W.gen_x(s, Tv, layer=l, step=K + 1, which=1) for l in range(L)]),
            "lgv": np.stack([W.verify_logits(s, l) for l in range(L)])}
    host_t = {n: torch.from_numpy(np.ascontiguousarray(a.view(np.float16) if a.dtype == np.uint16 else a)).pin_memory()
              for n, a in host.items()}
    dev_in = [{n: t.cuda() for n, t in host_t.items()} for _ in range(2)]
    dev_out = [{"od": torch.zeros(L, 1, H, dtype=torch.float16, device="cuda"),
                "ov": torch.zeros(L, Tv, H, dtype=torch.float16, device="cuda"),
                "elb": torch.zeros(L, E, dtype=torch.int32, device="cuda")} for _ in range(2)]
    ws_d, ws_v = spx.new_workspace(1, H, s.I, E, k, s.I_s), spx.new_workspace(Tv, H, s.I, E, k, s.I_s)
    r_d, r_v = spx.Routing.empty(1, E, k), spx.Routing.empty(Tv, E, k)

    def cycle_args(b):
        di, do = dev_in[b], dev_out[b]
        d = [[spx.layer_args(0, di["xd"][st, l], E, k, s.renorm, di["lgd"][st, l], r_d, do["od"][l], ws_d,
                             w4=lays[l]["w4"], shared=lays[l]["shared"], elb=do["elb"], layer=l)
              for l in range(L)] for st in range(K)]
        v = [spx.layer_args(1, di["xv"][l], E, k, s.renorm, di["lgv"][l], r_v, do["ov"][l], ws_v,
                            f16=lays[l]["f16"], shared=lays[l]["shared"]) for l in range(L)]
        return d, v

    cargs = [cycle_args(0), cycle_args(1)]

    def cycle(b, evs=None):
        d, v = cargs[b]
        if evs:
            evs[0].record(stream)
        spx.spx_elb_reset(dev_out[b]["elb"], stream)
        for st in range(K):
            for l in range(L):
                spx.spx_moe_layer(d[st][l][0], stream)
        if evs:
            evs[1].record(stream)
        for l in range(L):
            spx.spx_moe_layer(v[l][0], stream)
        if evs:
            evs[2].record(stream)

    # algorithmic bytes of a cycle, from the library's own routing (untimed pass)
    draft_bytes = verify_bytes = 0
    nv_list = []
    d0, v0 = cargs[0]
    spx.spx_elb_reset(dev_out[0]["elb"])
    for st in range(K):
        for l in range(L):
            spx.spx_moe_layer(d0[st][l][0])
            draft_bytes += layer_bytes(s, "draft", 1, int(r_d.n_active.item()))
    for l in range(L):
        spx.spx_moe_layer(v0[l][0])
        nv_list.append(int(r_v.n_active.item()))
        verify_bytes += layer_bytes(s, "verify", Tv, nv_list[-1])
    elb = dev_out[0]["elb"].cpu().numpy()
    distinct = (elb > 0).sum(1)
    cycle_bytes = draft_bytes + verify_bytes
    n_draft = K * L

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            cycle(i % 2)
    sync_all()
    evs = [(ev(), ev(), ev()) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        e0, e1 = ev(), ev()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for i in range(args.steps):
                cycle(i % 2, evs[i])
            e1.record(stream)
        sync_all()
        ms_total = e0.elapsed_time(e1)
        time.sleep(0.05)
    clocks = clk.summary()
    dph = [a.elapsed_time(b) for a, b, c in evs]
    vph = [b.elapsed_time(c) for a, b, c in evs]
    value, _ = job_throughput(cycle_bytes * args.steps, ms_total, device="cuda")
    ms_step = ms_total / args.steps
    d_us = statistics.median(dph) * 1e3 / n_draft  # per chained draft launch
    v_us = statistics.median(vph) * 1e3 / L         # per verify layer (routing + expert launch)

    # e2e: each step's inputs copied in from pinned host memory and its outputs
    # (verify outputs, last draft outputs, lookahead counters) copied back, on a
    # copy stream that overlaps the neighbouring steps (double buffers).
    host_out = [{n: torch.empty_like(t, device="cpu").pin_memory() for n, t in dev_out[0].items()} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_t.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    cstream = torch.cuda.Stream()
    n_all = args.warmup + args.steps
    ev_in = [torch.cuda.Event() for _ in range(n_all)]
    ev_done = [torch.cuda.Event() for _ in range(n_all)]
    ev_out = [torch.cuda.Event() for _ in range(n_all)]

    def h2d_step(i):
        with torch.cuda.stream(cstream):
            if i >= 2:
                cstream.wait_event(ev_done[i - 2])  # the buffer's previous step has finished
            for n, t in host_t.items():
                dev_in[i % 2][n].copy_(t, non_blocking=True)
            ev_in[i].record(cstream)

    sync_all()
    t0 = time.perf_counter()
    for i in range(n_all):
        if i == args.warmup:
            cstream.synchronize()
            stream.synchronize()
            t0 = time.perf_counter()
        if i == 0 or i == args.warmup:
            h2d_step(i)
        if i + 1 < n_all and i + 1 != args.warmup:
            h2d_step(i + 1)
        with torch.cuda.stream(stream):
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])  # this output buffer has been read back
            cycle(i % 2)
            ev_done[i].record(stream)
        with torch.cuda.stream(cstream):
            cstream.wait_event(ev_done[i])
            for n, t in host_out[i % 2].items():
                t.copy_(dev_out[i % 2][n], non_blocking=True)
            ev_out[i].record(cstream)
    cstream.synchronize()
    stream.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_gbs, _ = job_throughput(cycle_bytes * args.steps, e2e_s * 1e3, device="cuda")
    assert spx.spx_workspace_status(ws_d) == 0 and spx.spx_workspace_status(ws_v) == 0

    # per-layer figures of the three single-layer shapes
    per_cfg = {}
    for name in GATE_CONFIGS:
        c = W.CONFIGS[name]
        sets = lays if name == "deepseek_v2_lite" else [make_weight_set(c, i, torch, spx, tc_pack=True)
                                                        for i in range(NSETS)]
        per_cfg[name] = layer_figures(c, sets, torch, spx, stream, peak)
        if sets is not lays:
            del sets
            torch.cuda.empty_cache()

    pt_d, pt_v = traffic_of("draft"), traffic_of("verify")
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 (int4 draft weights, fp32 accumulate)",
        "data": "synthetic (seeded random weights and activations per layer; drawn Zipf(1.1) router logits)",
        "config": {"workload": f"{s.name}: 26-layer DeepSeek-V2-Lite-shaped draft-then-verify cycle, {K} draft steps "
                               f"(T=1) x {L} layers + one verify pass (T={Tv}) x {L} layers",
                   "layers": L, "K": K, "H": H, "I": s.I, "E": E, "k": k, "I_shared": s.I_s,
                   "l2": f"{L} layer weight sets ({L * 1.43:.0f} GB) > L2; no flush",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "cycle": {"us_per_cycle": round(ms_step * 1e3, 1), "draft_phase_us": round(statistics.median(dph) * 1e3, 1),
                  "verify_phase_us": round(statistics.median(vph) * 1e3, 1),
                  "draft_layer_us": round(d_us, 2), "verify_layer_us": round(v_us, 2),
                  "bytes_per_cycle": int(cycle_bytes), "draft_bytes": int(draft_bytes),
                  "verify_bytes": int(verify_bytes), "frac_of_peak": round(value / peak, 3),
                  "verify_unique_experts_mean": round(statistics.mean(nv_list), 2),
                  "elb_distinct_experts_per_layer": {"mean": round(float(distinct.mean()), 2),
                                                     "min": int(distinct.min()), "max": int(distinct.max())}},
        "roofline": {"bound": "hbm", "kernel": "draft_kernel<2, 0> (draft launch: routing + INT4 experts + shared "
                                               "expert + combine), the cycle's dominant kernel",
                     "achieved": round(draft_bytes / n_draft / (d_us * 1e-6) / 1e9, 1), "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s",
                     "frac": round(draft_bytes / n_draft / (d_us * 1e-6) / 1e9 / peak, 3),
                     "traffic": pt_d, "traffic_source": traffic_note("draft"),
                     "launch_us": round(d_us, 2), "bytes_per_launch": int(draft_bytes / n_draft),
                     "timing": f"CUDA events around the draft phase of every timed cycle ({n_draft} launches back "
                               f"to back on the launching stream), median over cycles / {n_draft}"},
        "verify_roofline": {"bound": "hbm", "kernel": "route_kernel + tc_gather_kernel + tc_mlp_kernel (tcgen05 "
                                                      "gate/up and down) + tc_out_kernel (verify layer)",
                            "achieved": round(verify_bytes / L / (v_us * 1e-6) / 1e9, 1), "peak": peak,
                            "unit": "GB/s", "frac": round(verify_bytes / L / (v_us * 1e-6) / 1e9 / peak, 3),
                            "layer_us": round(v_us, 2), "bytes_per_layer": int(verify_bytes / L),
                            "traffic": pt_v, "traffic_source": traffic_note("verify")},
        "configs": per_cfg,
        "clocks": clocks,
        "e2e": {"value": round(e2e_gbs, 1), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        # per cycle: K*L draft launches; per verify layer a routing launch and the three tensor-memory
        # launches (gather, gate/up + down, output)
        "gpu_launches": (n_draft + 4 * L) * args.steps,
    }
    if rank == 0 and args.cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(s)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def layer_figures(s, sets, torch, spx, stream, peak, n_batches=10):
    """Per-layer figures of one shape: draft (T = 1) and verify (T = K+1) layers
    timed back to back (batches of chained calls over rotated weight sets and
    inputs; events around each batch only, so the launch chain is kept), and the
    expert launch alone (events around it)."""
    out = {}
    for mode, T, chain in (("draft", s.T_draft, 64), ("verify", s.T_verify, 16)):
        which = 0 if mode == "draft" else 1
        xs = [torch.from_numpy(np.ascontiguousarray(W.gen_x(s, T, step=i, which=which)).view(np.float16)).cuda()
              for i in range(NINPUTS)]
        lgs = [torch.from_numpy(W.gen_logits(s, T, step=i, which=which)).cuda() if s.logits != "router"
               else torch.empty(T, s.E, device="cuda") for i in range(NINPUTS)]
        ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s)
        r = spx.Routing.empty(T, s.E, s.k)
        o = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
        n = len(sets) * NINPUTS // int(np.gcd(len(sets), NINPUTS))

        def call_args(i, events=None):
            st = sets[i % len(sets)]
            return spx.layer_args(which, xs[i % NINPUTS], s.E, s.k, s.renorm, lgs[i % NINPUTS], r, o, ws,
                                  w4=st["w4"] if mode == "draft" else None,
                                  f16=st["f16"] if mode == "verify" else None, shared=st["shared"],
                                  w_router=st["w_router"], events=events)

        keep = [call_args(i) for i in range(n)]
        nb = []
        for i in range(NINPUTS):  # unique experts per input, from the library's routing
            spx.spx_moe_layer(keep[i][0])
            nb.append(layer_bytes(s, mode, T, int(r.n_active.item())))
        byt = float(np.mean(nb))
        with torch.cuda.stream(stream):
            for i in range(2 * chain):
                spx.spx_moe_layer(keep[i % n][0], stream)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n_batches)]
            j = 0
            for a, b in evs:
                a.record(stream)
                for _ in range(chain):
                    spx.spx_moe_layer(keep[j % n][0], stream)
                    j += 1
                b.record(stream)
        torch.cuda.synchronize()
        per = [a.elapsed_time(b) / chain for a, b in evs]  # ms per layer, per batch
        # the expert launch alone (events recorded around it; no overlap with neighbours)
        kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(16)]
        kkeep = []
        with torch.cuda.stream(stream):
            for i, e_ in enumerate(kev):
                for x in e_:
                    x.record(stream)
                ka = call_args(i, events=e_)
                kkeep.append(ka)
                spx.spx_moe_layer(ka[0], stream)
        torch.cuda.synchronize()
        k_us = statistics.mean(a.elapsed_time(b) for a, b in kev) * 1e3
        k_bytes = byt - (T * s.E * 4 if mode == "verify" else 0) - (s.E * s.H * 2 if s.logits == "router" else 0)
        assert spx.spx_workspace_status(ws) == 0
        us = statistics.median(per) * 1e3
        out[mode] = {"T": T, "layer_us": spread_us(per), "gbs": round(byt / (us * 1e-6) / 1e9, 1),
                     "frac": round(byt / (us * 1e-6) / 1e9 / peak, 3), "tokens_per_s": round(T / (us * 1e-6), 1),
                     "bytes": int(byt),
                     "expert_launch_alone": {"us": round(k_us, 2), "bytes": int(k_bytes),
                                             "gbs": round(k_bytes / (k_us * 1e-6) / 1e9, 1),
                                             "frac": round(k_bytes / (k_us * 1e-6) / 1e9 / peak, 3)},
                     "timing": f"{n_batches} batches of {chain} layer calls back to back; spread over batches"}
        if mode == "verify":
            # the library's automatic choice (every shape here has its tile packs)
            tc = sets[0]["f16"].tc is not None and T >= 9
            out[mode]["launches"] = ("routing + tensor-memory launches (gather, tcgen05 gate/up + down, output)"
                                     if tc else "routing + expert launch")
    return out


# ---------------------------------------------------------------- oracle --
def cpu_baseline(s, reps=1):
    """The CPU oracle (single thread) on one draft + one verify layer."""
    import oracle
    oracle.build()
    d = make_inputs(s, 0)
    ids_d, _ = oracle.route_topk(d["lg_d"].astype(np.float64), s.k, s.renorm)
    ids_v, _ = oracle.route_topk(d["lg_v"].astype(np.float64), s.k, s.renorm)
    need_d = sorted(set(ids_d.reshape(-1).tolist()))
    need_v = sorted(set(ids_v.reshape(-1).tolist()))
    w4 = {e: W.gen_w4_expert(s, 0, e) for e in need_d}
    f16 = {e: W.gen_f16_expert(s, 0, e) for e in need_v}
    sh = W.gen_shared(s, 0)
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.moe_layer("draft", d["x_d"], s.k, s.renorm, w4.__getitem__, s.E, logits=d["lg_d"], shared=sh)
        oracle.moe_layer("verify", d["x_v"], s.k, s.renorm, f16.__getitem__, s.E, logits=d["lg_v"], shared=sh)
    dt = (time.perf_counter() - t0) / reps
    b = layer_bytes(s, "draft", s.T_draft, len(need_d)) + layer_bytes(s, "verify", s.T_verify, len(need_v))
    return {"value": round(b / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"1 draft (T={s.T_draft}) + 1 verify (T={s.T_verify}) layer of {s.name} (one of the cycle's "
                      f"{s.layers * (s.K + 1)} layer calls), input set 0, {reps} rep(s), {dt:.2f} s per sample; "
                      f"GB/s = the sample's algorithmic bytes / its time"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    s = W.CONFIGS[CYCLE]
    times = []
    cb = None
    for i in range(args.warmup + args.steps):
        cb = cpu_baseline(s)
        if i >= args.warmup:
            times.append(cb)
    vals = [c["value"] for c in times]
    v = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{s.name}: 26-layer DeepSeek-V2-Lite-shaped draft-then-verify cycle, {s.K} draft "
                                   f"steps (T=1) x {s.layers} layers + one verify pass (T={s.T_verify}) x {s.layers} "
                                   f"layers"},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": cb["sample"]},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def apply_formats(s, sets, args, torch, spx):
    """Replace each weight set's INT4 draft experts by the format the flags ask
    for: --zeros (INT4 with seeded per-group zero points) or --gguf (GGUF
    super-blocks with random codes and scales of the INT4 weights' magnitude)."""
    if args.zeros:  # asymmetric INT4: seeded per-group zero points on every set
        E, H, I = s.E, s.H, s.I
        for i, st in enumerate(sets):
            g = torch.Generator(device="cuda")
            g.manual_seed(2_000_003 * (s.seed + 1) + i)

            def words(*shape):
                return torch.randint(-2 ** 31, 2 ** 31, shape, dtype=torch.int32, device="cuda", generator=g)

            st["w4"] = spx.spx_w4_zeros_repack(st["w4"], words(E, H // 128, I // 8), words(E, H // 128, I // 8),
                                               words(E, I // 128, H // 8))
        torch.cuda.synchronize()
    if args.gguf:  # GGUF experts instead of INT4: random codes, scales of the INT4 weights' magnitude
        E, H, I = s.E, s.H, s.I
        for i, st in enumerate(sets):
            g = torch.Generator(device="cuda")
            g.manual_seed(3_000_017 * (s.seed + 1) + i)

            def scales(shape, lo, hi):
                return (torch.rand(shape, device="cuda", generator=g) * (hi - lo) + lo).half().view(torch.uint8)

            def q8(N, K):  # Q8_0 blocks, d U(0.0003, 0.00125)
                b = torch.randint(0, 256, (E, N, K // 32, 34), dtype=torch.uint8, device="cuda", generator=g)
                b[..., :2] = scales((E, N, K // 32), 0.0003, 0.00125).view(E, N, K // 32, 2)
                return b

            def q2k(N, K):  # Q2_K super-blocks, d U(0.001, 0.003), dmin U(0.001, 0.004)
                b = torch.randint(0, 256, (E, N, K // 256, 84), dtype=torch.uint8, device="cuda", generator=g)
                b[..., 80:82] = scales((E, N, K // 256), 0.001, 0.003).view(E, N, K // 256, 2)
                b[..., 82:84] = scales((E, N, K // 256), 0.001, 0.004).view(E, N, K // 256, 2)
                return b

            def q4k(N, K):  # Q4_K super-blocks, d U(0.00015, 0.0004), dmin U(0.0003, 0.001)
                b = torch.randint(0, 256, (E, N, K // 256, 144), dtype=torch.uint8, device="cuda", generator=g)
                b[..., 0:2] = scales((E, N, K // 256), 0.00015, 0.0004).view(E, N, K // 256, 2)
                b[..., 2:4] = scales((E, N, K // 256), 0.0003, 0.001).view(E, N, K // 256, 2)
                return b

            gu, ty = {"q8_0": (q8, spx.SPX_GGUF_Q8_0), "q2_k": (q2k, spx.SPX_GGUF_Q2_K),
                      "q4_k": (q4k, spx.SPX_GGUF_Q4_K)}[args.gguf]
            st["w4"] = None
            st["gguf"] = spx.spx_gguf_repack(gu(I, H), gu(I, H), q8(H, I), ty)
            torch.cuda.synchronize()


def run_loop(args):
    """Profiling driver: --loop-n layer calls of one mode on --sets weight sets,
    no timing (the command that ncu captures wrap)."""
    import torch
    from quantized_expert_gb300 import build as B, spx
    B.build()
    spx.load()
    s = W.CONFIGS[args.config]
    draft = args.loop == "draft"
    launch = 0 if draft else args.verify_launch
    sets = [make_weight_set(s, i, torch, spx, tc_pack=launch != 1) for i in range(NSETS)]
    if draft:
        apply_formats(s, sets, args, torch, spx)
    if args.tokens:  # another token count than the shape's draft / verify one
        T = args.tokens
        x = torch.from_numpy(np.ascontiguousarray(W.gen_x(s, T, step=1)).view(np.float16)).cuda()
        lg = (torch.from_numpy(W.gen_logits(s, T, step=1)).cuda() if s.logits != "router"
              else torch.empty(T, s.E, device="cuda"))
    else:
        inp = make_inputs(s, 0)
        T = s.T_draft if draft else s.T_verify
        xk, lk = ("x_d", "lg_d") if draft else ("x_v", "lg_v")
        x = torch.from_numpy(np.ascontiguousarray(inp[xk]).view(np.float16)).cuda()
        lg = torch.from_numpy(inp[lk]).cuda() if lk in inp else torch.empty(T, s.E, device="cuda")
    ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s, tc=launch == 2)
    r = spx.Routing.empty(T, s.E, s.k)
    out = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
    keep = [spx.layer_args(0 if draft else 1, x, s.E, s.k, s.renorm, lg, r, out, ws,
                           w4=st["w4"] if draft else None, f16=None if draft else st["f16"], shared=st["shared"],
                           w_router=st["w_router"], gguf=st.get("gguf") if draft else None, verify_launch=launch)
            for st in sets]
    for i in range(args.loop_n):
        spx.spx_moe_layer(keep[i % len(keep)][0])
    torch.cuda.synchronize()
    assert spx.spx_workspace_status(ws) == 0
    print(json.dumps({"loop": args.loop, "config": s.name, "calls": args.loop_n}), flush=True)


def run_cached(args):
    """Cache-aware verify execution: the verify layer with its routed experts
    queued resident first (resident = the experts the K draft steps before it
    selected, i.e. the lookahead counters' nonzero entries) and a ready flag
    per expert (all set), against the plain verify layer on the same inputs.
    Prints one JSON line: device us per layer of both, and the share of the
    verify's routed experts that were resident."""
    import torch
    from quantized_expert_gb300 import build as B, spx
    B.build()
    spx.load()
    s = W.CONFIGS[args.config]
    Tv = s.T_verify
    sets = [make_weight_set(s, i, torch, spx) for i in range(NSETS)]
    inputs = [make_inputs(s, i) for i in range(NINPUTS)]
    if "lg_d" not in inputs[0]:
        print(json.dumps({"metric": "cache-aware verify", "unavailable": "shape computes its logits on the device"}))
        return
    # resident experts: union of the draft top-k of K = T_verify - 1 draft steps
    K = Tv - 1
    ids = [oracle_free_topk(inputs[i]["lg_d"], s.k) for i in range(K)]
    res = np.zeros(s.E, np.uint8)
    for x in ids:
        res[x.reshape(-1)] = 1
    resident = torch.from_numpy(res).cuda()
    ready = torch.ones(s.E, dtype=torch.int32, device="cuda")
    ws = spx.new_workspace(Tv, s.H, s.I, s.E, s.k, s.I_s)
    r = spx.Routing.empty(Tv, s.E, s.k)
    out = torch.empty(Tv, s.H, dtype=torch.float16, device="cuda")
    dev = []
    for d in inputs:
        dev.append((torch.from_numpy(np.ascontiguousarray(d["x_v"]).view(np.float16)).cuda(),
                    torch.from_numpy(d["lg_v"]).cuda()))
    hits = []
    for i in range(NINPUTS):
        top = oracle_free_topk(inputs[i]["lg_v"], s.k)
        u = np.unique(top)
        hits.append(float(res[u].mean()))

    def calls(cached):
        return [spx.layer_args(1, dev[i % NINPUTS][0], s.E, s.k, s.renorm, dev[i % NINPUTS][1], r, out, ws,
                               f16=sets[i % NSETS]["f16"], shared=sets[i % NSETS]["shared"],
                               resident=resident if cached else None, ready=ready if cached else None)
                for i in range(NSETS * NINPUTS)]

    res_us = {}
    stream = torch.cuda.Stream()
    for name, cached in (("plain", False), ("cached", True)):
        keep = calls(cached)
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                spx.spx_moe_layer(keep[i % len(keep)][0], stream)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(args.steps):
                spx.spx_moe_layer(keep[i % len(keep)][0], stream)
            e1.record(stream)
        torch.cuda.synchronize()
        res_us[name] = e0.elapsed_time(e1) * 1e3 / args.steps
    assert spx.spx_workspace_status(ws) == 0
    line = {"metric": "cache-aware verify layer (resident first + ready flags) vs plain, device us per layer",
            "config": {"workload": f"{s.name} verify T={Tv}", "resident": f"draft top-{s.k} of {K} steps",
                       "resident_experts": int(res.sum())},
            "plain_us": round(res_us["plain"], 2), "cached_us": round(res_us["cached"], 2),
            "overhead_pct": round(100 * (res_us["cached"] / res_us["plain"] - 1), 2),
            "verify_expert_hit_share": round(float(np.mean(hits)), 3), "steps": args.steps, "warmup": args.warmup}
    print(json.dumps(line), flush=True)


def run_draft_batch(args):
    """Draft layers carrying T = 1, 2, 4, 8, 16 tokens (one per request) in one
    call, or with --verify-batch verify layers of T = 9, 17, 33 tokens (more
    tokens per expert): device us per layer, unique experts, algorithmic GB/s
    and tokens/s.  Prints one JSON line."""
    import torch
    from quantized_expert_gb300 import build as B, spx
    B.build()
    spx.load()
    s = W.CONFIGS[args.config]
    verify = args.verify_batch
    launch = args.verify_launch if verify else 0
    sets = [make_weight_set(s, i, torch, spx, tc_pack=verify and launch != 1) for i in range(NSETS)]
    if not verify:
        apply_formats(s, sets, args, torch, spx)
    peak, peak_src = measured_peaks()
    rows = []
    stream = torch.cuda.Stream()
    mode = 1 if verify else 0
    for T in ((9, 17, 33, 64) if verify else (1, 2, 4, 8, 16)):
        xs = [torch.from_numpy(np.ascontiguousarray(W.gen_x(s, T, step=i)).view(np.float16)).cuda()
              for i in range(NINPUTS)]
        lgs = [torch.from_numpy(W.gen_logits(s, T, step=i)).cuda() if s.logits != "router"
               else torch.empty(T, s.E, device="cuda") for i in range(NINPUTS)]
        ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s, tc=launch == 2)
        r = spx.Routing.empty(T, s.E, s.k)
        out = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
        try:
            keep = [spx.layer_args(mode, xs[i % NINPUTS], s.E, s.k, s.renorm, lgs[i % NINPUTS], r, out, ws,
                                   w4=None if verify else sets[i % NSETS]["w4"],
                                   f16=sets[i % NSETS]["f16"] if verify else None, shared=sets[i % NSETS]["shared"],
                                   w_router=sets[i % NSETS]["w_router"],
                                   gguf=None if verify else sets[i % NSETS].get("gguf"), verify_launch=launch)
                    for i in range(NSETS * NINPUTS)]
            nb = []
            for i in range(NINPUTS):
                spx.spx_moe_layer(keep[i][0])
                torch.cuda.synchronize()
                nb.append((int(r.n_active.item()), layer_bytes(s, "verify" if verify else "draft", T,
                                                               int(r.n_active.item()), args.zeros, args.gguf)))
        except spx.SpxError as err:  # a shape the launch does not take (activation rows beyond shared memory)
            rows.append({"T": T, "unsupported": str(err)})
            continue
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                spx.spx_moe_layer(keep[i % len(keep)][0], stream)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(args.steps):
                spx.spx_moe_layer(keep[i % len(keep)][0], stream)
            e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / args.steps
        ua = float(np.mean([a for a, _ in nb]))
        byt = float(np.mean([b for _, b in nb]))
        rows.append({"T": T, "layer_us": round(us, 2), "unique_experts": round(ua, 2),
                     "gbs": round(byt / (us * 1e-6) / 1e9, 1), "frac": round(byt / (us * 1e-6) / 1e9 / peak, 3),
                     "tokens_per_s": round(T / (us * 1e-6), 1)})
        assert spx.spx_workspace_status(ws) == 0
    zp = (", per-group zero points" if args.zeros else ", GGUF Q8_0 experts" if args.gguf == "q8_0"
          else f", GGUF {args.gguf.upper()} gate/up + Q8_0 down experts" if args.gguf else "")
    line = {"metric": ("verify layer with T tokens per call" if verify else
                       "draft layer with T requests' tokens per call") + ", device us per layer",
            "config": {"workload": f"{s.name} verify, T = 9, 17, 33, 64, " + {
                0: "automatic launch choice (tensor-memory launches from 25 tokens)", 1: "expert launch",
                2: "tensor-memory launches"}[launch] if verify else
                       f"{s.name} draft{zp}, T = 1, 2, 4, 8, 16 (one token per request; 8 and 16 on the "
                       f"routing launch + expert launch)"},
            "peak": peak, "peak_source": peak_src, "rows": rows, "steps": args.steps, "warmup": args.warmup}
    print(json.dumps(line), flush=True)


def run_prefetch(args):
    """The Layer-Aware Prefetch Planner on GB300: L DeepSeek-V2-Lite-shaped
    layers whose routed FP16 verify experts live in page-locked host (Grace)
    memory and reach HBM over NVLink-C2C, one speculation cycle of K draft
    steps then the verify pass.  Three arms on the same inputs: every expert
    resident (no copy); on demand (each layer's verify experts copied when the
    verify pass starts, the verify launches waiting on their ready flags); and
    planned (the planner's copies issued at the draft-chunk boundaries from the
    lookahead counters, the rest loaded behind the verify launches).  Prints
    one JSON line: cycle and verify-pass us of each arm, and the share of the
    on-demand copy wait that the plan hides."""
    import ctypes as C  # noqa: F401
    import torch
    from quantized_expert_gb300 import build as B, spx
    B.build()
    lib = spx.load()
    s = W.CONFIGS[CYCLE]
    L, K, E, k, H, Tv = min(args.prefetch_layers, s.layers), s.K, s.E, s.k, s.H, s.T_verify
    lays = [make_weight_set(s, l, torch, spx) for l in range(L)]
    eb = lib.spx_f16_packed_bytes(1, H, s.I)
    host = [ly["f16"].buf.cpu().pin_memory() for ly in lays]
    dev = [ly["f16"].buf for ly in lays]
    f16 = [spx.PackedF16(d, E, H, s.I) for d in dev]
    stream = torch.cuda.Stream()
    sides = [torch.cuda.Stream() for _ in range(max(1, args.prefetch_streams))]  # copy streams
    f16dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.float16)).cuda()  # noqa: E731
    xd = [[f16dev(W.gen_x(s, 1, layer=l, step=st)) for l in range(L)] for st in range(1, K + 1)]
    lgd = [[torch.from_numpy(W.draft_logits(s, l, st)).cuda() for l in range(L)] for st in range(1, K + 1)]
    xv = [f16dev(W.gen_x(s, Tv, layer=l, step=K + 1, which=1)) for l in range(L)]
    lgv_host = [W.verify_logits(s, l) for l in range(L)]
    lgv = [torch.from_numpy(a).cuda() for a in lgv_host]
    verify_need = [sorted(set(oracle_free_topk(a, k).reshape(-1).tolist())) for a in lgv_host]
    elb = torch.zeros(L, E, dtype=torch.int32, device="cuda")
    elb_host = torch.zeros(L, E, dtype=torch.int32).pin_memory()
    ready = torch.zeros(L, E, dtype=torch.int32, device="cuda")
    resident = torch.zeros(L, E, dtype=torch.uint8, device="cuda")
    ws_d, ws_v = spx.new_workspace(1, H, s.I, E, k, s.I_s), spx.new_workspace(Tv, H, s.I, E, k, s.I_s)
    r_d, r_v = spx.Routing.empty(1, E, k), spx.Routing.empty(Tv, E, k)
    od = torch.empty(1, H, dtype=torch.float16, device="cuda")
    ov = torch.empty(Tv, H, dtype=torch.float16, device="cuda")
    dargs = [[spx.layer_args(0, xd[st][l], E, k, s.renorm, lgd[st][l], r_d, od, ws_d, w4=lays[l]["w4"],
                             shared=lays[l]["shared"], elb=elb, layer=l) for l in range(L)] for st in range(K)]
    vres = [spx.layer_args(1, xv[l], E, k, s.renorm, lgv[l], r_v, ov, ws_v, f16=f16[l], shared=lays[l]["shared"])
            for l in range(L)]
    vflag = [spx.layer_args(1, xv[l], E, k, s.renorm, lgv[l], r_v, ov, ws_v, f16=f16[l], shared=lays[l]["shared"],
                            resident=resident[l], ready=ready[l]) for l in range(L)]

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def draft_steps(a, b):
        with torch.cuda.stream(stream):
            for st in range(a, b):
                for l in range(L):
                    spx.spx_moe_layer(dargs[st][l][0], stream)

    # measured inputs of the plan: one draft step through the L layers, one expert's copy
    draft_steps(0, K)
    torch.cuda.synchronize()
    e0, e1 = ev(), ev()
    e0.record(stream)
    draft_steps(0, K)
    e1.record(stream)
    torch.cuda.synchronize()
    step_us = e0.elapsed_time(e1) * 1e3 / K
    # one expert's copy time with the copies spread over the copy streams
    ncp = 8 * len(sides)
    torch.cuda.synchronize()
    e0.record(stream)
    for sd in sides:
        sd.wait_stream(stream)
    for i in range(ncp):
        with torch.cuda.stream(sides[i % len(sides)]):
            dev[0][(i % E) * eb:(i % E + 1) * eb].copy_(host[0][(i % E) * eb:(i % E + 1) * eb], non_blocking=True)
    for sd in sides:
        stream.wait_stream(sd)
    e1.record(stream)
    torch.cuda.synchronize()
    copy_us = e0.elapsed_time(e1) * 1e3 / ncp
    cfg = spx.PlanCfg(L, E, K, E, 1, step_us, copy_us)

    def offload():
        torch.cuda.synchronize()
        for d in dev:
            d.zero_()
        ready.zero_()
        resident.zero_()
        torch.cuda.synchronize()

    def verify_pass(flags):
        with torch.cuda.stream(stream):
            for l in range(L):
                spx.spx_moe_layer((vflag if flags else vres)[l][0], stream)

    def issue(acts):
        # actions dealt round-robin to the copy streams: each expert's copy and
        # its flags stay in one stream's order
        acts = np.asarray(acts, np.int32).reshape(-1, 3)
        for sd in sides:
            sd.wait_stream(stream)
        for j, sd in enumerate(sides):
            part = acts[j::len(sides)]
            if len(part):
                spx.spx_prefetch_issue(part, host, dev, eb, ready, resident, stream=sd)

    def load_all(need_by_layer, cached):
        acts = [[l, e, spx.SPX_PLAN_LOAD] for l in range(L) for e in need_by_layer[l] if not cached[l, e]]
        for l in range(L):
            cached[l, need_by_layer[l]] = 1
        issue(acts)
        return len(acts)

    res = {}
    for arm in ("resident", "on_demand", "planned"):
        reps = []
        for rep in range(max(1, min(args.steps, 5))):
            if arm == "resident":
                for l in range(L):  # restore the weights once; they stay
                    if rep == 0:
                        dev[l].copy_(host[l], non_blocking=True)
                torch.cuda.synchronize()
            else:
                offload()
            spx.spx_elb_reset(elb, stream)
            cached = np.zeros((L, E), np.uint8)
            c0, c1, c2 = ev(), ev(), ev()
            c0.record(stream)
            nload = 0
            if arm == "planned":
                done, phase = 0, spx.SPX_PLAN_COLD_START
                while True:
                    if done:
                        spx.spx_elb_read(elb, elb_host, stream)
                        stream.synchronize()  # the snapshot at the chunk boundary
                    snap = elb_host.numpy().astype(np.uint32) if done else np.zeros((L, E), np.uint32)
                    phase, acts, chunk = spx.spx_plan_prefetch(cfg, snap, done, cached)
                    issue(acts)
                    nload += int((acts[:, 2] == spx.SPX_PLAN_LOAD).sum()) if len(acts) else 0
                    if phase == spx.SPX_PLAN_FINAL_CLEANUP:
                        break
                    draft_steps(done, done + chunk)
                    done += chunk
            else:
                draft_steps(0, K)
            c1.record(stream)
            if arm != "resident":
                nload += load_all(verify_need, cached)  # the verify's experts not cached yet
            verify_pass(arm != "resident")
            c2.record(stream)
            for sd in sides:
                stream.wait_stream(sd)
            torch.cuda.synchronize()
            reps.append((c0.elapsed_time(c2) * 1e3, c1.elapsed_time(c2) * 1e3, nload))
            assert spx.spx_workspace_status(ws_v) == 0 and spx.spx_workspace_status(ws_d) == 0
        res[arm] = {"cycle_us": round(statistics.median(r[0] for r in reps), 1),
                    "verify_pass_us": round(statistics.median(r[1] for r in reps), 1),
                    "expert_loads": reps[-1][2]}
    wait_od = res["on_demand"]["verify_pass_us"] - res["resident"]["verify_pass_us"]
    wait_pl = res["planned"]["verify_pass_us"] - res["resident"]["verify_pass_us"]
    line = {"metric": "verify-pass copy wait hidden by the Layer-Aware Prefetch Planner",
            "config": {"workload": f"{s.name} shape, {L} layers, K={K} draft steps (T=1) then verify (T={Tv}); routed "
                                   f"FP16 experts in page-locked host memory, copied over NVLink-C2C",
                       "expert_bytes": int(eb), "step_us": round(step_us, 1), "copy_streams": len(sides),
                       "copy_us_per_expert": round(copy_us, 1),
                       "link_gbs": round(eb / (copy_us * 1e-6) / 1e9, 1)},
            "arms": res,
            "hidden_share": round(1.0 - wait_pl / wait_od, 3) if wait_od > 0 else None,
            "reps": max(1, min(args.steps, 5))}
    print(json.dumps(line), flush=True)


TL_EVENTS = ["entry", "prod_static", "prod_griddep", "x_staged", "routed", "first_fill", "gu_last", "dn_w_first",
             "dn_h_first", "dn_last", "prod_last", "cons_done", "out_done", "sg_last", "rg_first", "rg_last",
             "w_full", "w_hfull", "w_empty", "n_sg", "n_rg", "n_sd", "n_rd", "exit", "rd_h_last", "sd_last",
             "w_poll", "bytes", "w_ticket", "n_ticket", "w_route", "issue", "p_sg", "p_rg", "p_dn", "p_fence",
             "p_slot", "c_sg", "c_rg", "c_sd", "c_rd", "c_gu_done", "c_out"]
TL_FIRST_EV = {"entry", "prod_static", "prod_griddep", "x_staged", "routed", "first_fill", "dn_w_first",
               "dn_h_first", "cons_done", "rg_first"}
TL_SUM_EV = {"w_full", "w_hfull", "w_empty", "n_sg", "n_rg", "n_sd", "n_rd", "w_poll", "bytes", "w_ticket",
             "n_ticket", "w_route", "issue", "p_sg", "p_rg", "p_dn", "p_fence", "p_slot", "c_sg", "c_rg", "c_sd",
             "c_rd", "c_gu_done", "c_out"}


def timeline_phases(buf, slots, nblocks):
    """Per-phase table of draft launches from the profiling build's marks
    (buf [slots][blocks][events] uint64): for each mark the earliest, median
    and latest block in us after the launch's first block entered; sums per
    block.  Averaged over the given slots."""
    acc = {}
    for sl in slots:
        b = buf[sl, :nblocks, :].astype(np.uint64)
        t = {}
        for j, nm in enumerate(TL_EVENTS):
            col = b[:, j]
            if nm in TL_SUM_EV:
                t[nm] = col.astype(np.float64)
            elif nm in TL_FIRST_EV:
                t[nm] = np.where(col != 0, (~col).astype(np.float64), np.nan)
            else:
                t[nm] = np.where(col != 0, col.astype(np.float64), np.nan)
        t0 = np.nanmin(t["entry"])
        for nm in TL_EVENTS:
            v = t[nm]
            if nm in TL_SUM_EV:
                row = {"per_block_mean": float(np.mean(v)), "total": float(np.sum(v))}
            else:
                r = (v - t0) / 1e3
                r = r[~np.isnan(r)]
                if r.size == 0:
                    continue
                row = {"min": float(r.min()), "median": float(np.median(r)), "max": float(r.max()), "blocks": int(r.size)}
            for k2, v2 in row.items():
                acc.setdefault(nm, {}).setdefault(k2, []).append(v2)
        acc.setdefault("_t0", []).append(t0)
    out = {nm: {k2: round(float(np.mean(v2)), 3) for k2, v2 in d.items()} for nm, d in acc.items() if nm != "_t0"}
    t0s = acc["_t0"]
    if len(t0s) > 1:
        out["launch_period_us"] = round(float(np.mean(np.diff(t0s))) / 1e3, 3)
    return out


def run_timeline(args):
    """Phase marks of the draft launch at T = 1 (profiling build with
    %globaltimer marks; timings of that build are not bench values): 8 launches
    each alone (synchronised between them), then 8 back to back.  Prints one
    JSON line with the per-phase table of both."""
    import ctypes as C
    import torch
    from quantized_expert_gb300 import build as B, spx
    lib = spx.load(B.build(variant="timeline"))
    lib.spx_timeline_reset.restype = C.c_int
    lib.spx_timeline_read.restype = C.c_int
    lib.spx_timeline_read.argtypes = [C.c_void_p, C.c_size_t]
    s = W.CONFIGS[args.config]
    T = s.T_draft
    sets = [make_weight_set(s, i, torch, spx) for i in range(NSETS)]
    xs = [torch.from_numpy(np.ascontiguousarray(W.gen_x(s, T, step=i)).view(np.float16)).cuda() for i in range(NINPUTS)]
    lgs = [torch.from_numpy(W.gen_logits(s, T, step=i)).cuda() if s.logits != "router"
           else torch.empty(T, s.E, device="cuda") for i in range(NINPUTS)]
    ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s)
    r = spx.Routing.empty(T, s.E, s.k)
    out = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
    keep = [spx.layer_args(0, xs[i % NINPUTS], s.E, s.k, s.renorm, lgs[i % NINPUTS], r, out, ws,
                           w4=sets[i % NSETS]["w4"], shared=sets[i % NSETS]["shared"],
                           w_router=sets[i % NSETS]["w_router"]) for i in range(NSETS * NINPUTS)]
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    stream = torch.cuda.Stream()
    buf = np.zeros((8, 256, 48), np.uint64)

    lib.spx_timeline_trace.restype = C.c_int
    lib.spx_timeline_trace.argtypes = [C.c_void_p, C.c_size_t]
    # per launch slot, 2 traced blocks: fill[48][4], item[64][4], unit[16][4] u32, t0 u64, nitem, pad
    tr_words = 48 * 4 + 64 * 4 + 16 * 4 + 2 + 2 + 8
    trbuf = np.zeros((8, 2, tr_words), np.uint32)
    traces = {}

    def read():
        torch.cuda.synchronize()
        assert lib.spx_timeline_read(buf.ctypes.data, buf.size) == 0
        assert lib.spx_timeline_trace(trbuf.ctypes.data, trbuf.nbytes) == 0
        traces[len(traces)] = trbuf.copy()
        return buf.copy()

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            spx.spx_moe_layer(keep[i % len(keep)][0], stream)
        torch.cuda.synchronize()
        assert lib.spx_timeline_reset() == 0
        for i in range(8):
            spx.spx_moe_layer(keep[i][0], stream)
            torch.cuda.synchronize()
        iso = read()
        assert lib.spx_timeline_reset() == 0
        for i in range(8):
            spx.spx_moe_layer(keep[8 + i][0], stream)
        chained = read()
    assert spx.spx_workspace_status(ws) == 0
    line = {"timeline": "draft launch phase marks (profiling build; us after the launch's first block entered)",
            "config": {"workload": f"{s.name} draft T={T}", "blocks": nsm},
            "isolated": timeline_phases(iso, range(8), nsm),
            "chained": timeline_phases(chained, range(1, 8), nsm),
            "trace": {"words": "per launch slot, blocks 0 and grid/2: fill[48][4] (wait start, stage free, issued, "
                               "kind<<24|bytes), item[64][4] (warp<<8|kind, landed, intermediate landed, done), "
                               "unit[16][4] (start, unit, described, issued), t0 (2 words), nitem, pad, route[8] (routing warp: "
                               "start, selected, outputs, tables, published); ns after block entry",
                      "isolated_slot4": traces[0][4].tolist(), "chained_slot4": traces[1][4].tolist()}}
    print(json.dumps(line), flush=True)


def oracle_free_topk(lg, k):
    """Top-k expert ids of fp32 logits (value descending, index ascending), for
    choosing the resident set; no method arithmetic beyond the ordering."""
    lg = np.asarray(lg, np.float32)
    order = np.lexsort((np.arange(lg.shape[-1])[None, :].repeat(lg.shape[0], 0), -lg), axis=-1)
    return order[:, :k]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--config", default="deepseek_v2_lite", choices=sorted(W.CONFIGS))
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--sets", type=int, default=NSETS, help="rotated weight sets (8 defeat L2)")
    ap.add_argument("--loop", choices=["draft", "verify"], help="profiling driver: layer calls only, no timing")
    ap.add_argument("--loop-n", type=int, default=12)
    ap.add_argument("--tokens", type=int, default=0, help="with --loop: tokens per call (default: the shape's)")
    ap.add_argument("--cached", action="store_true", help="cache-aware verify vs plain (prints its own line)")
    ap.add_argument("--draft-batch", action="store_true", help="draft layers at T = 1, 2, 4, 8, 16 (prints its own line)")
    ap.add_argument("--verify-batch", action="store_true",
                    help="verify layers at T = 9, 17, 33, 64 (prints its own line)")
    ap.add_argument("--verify-launch", type=int, default=0, choices=(0, 1, 2),
                    help="--verify-batch: 0 automatic, 1 the expert launch, 2 the tensor-memory launches")
    ap.add_argument("--zeros", action="store_true",
                    help="with --draft-batch or --loop draft: INT4 experts with per-group zero points")
    ap.add_argument("--gguf", choices=["q8_0", "q2_k", "q4_k"],
                    help="with --draft-batch or --loop draft: GGUF experts instead of INT4")
    ap.add_argument("--prefetch", action="store_true",
                    help="verify copy wait hidden by the prefetch plan (prints its own line)")
    ap.add_argument("--prefetch-layers", type=int, default=4)
    ap.add_argument("--prefetch-streams", type=int, default=4, help="with --prefetch: copy streams of the executor")
    ap.add_argument("--timeline", action="store_true",
                    help="draft launch phase marks from the profiling build (prints its own line)")
    args = ap.parse_args()
    globals()["NSETS"] = max(1, args.sets)
    if args.prefetch:
        run_prefetch(args)
    elif args.timeline:
        run_timeline(args)
    elif args.loop:
        run_loop(args)
    elif args.cached:
        run_cached(args)
    elif args.draft_batch or args.verify_batch:
        run_draft_batch(args)
    elif args.impl == "reference":
        if args.steps > 3:
            args.steps = 3
        if args.warmup > 1:
            args.warmup = 1
        run_reference(args)
    else:
        run_mine(args)


if __name__ == "__main__":
    main()
