"""Benchmark of the per-layer MoE expert hot path (libspx) on one GB300.

One step = one draft layer (T = 1, fused INT4 experts) + one verify layer
(T = K+1 = 17, expert-reordered FP16 experts), each the full chain route ->
top-k -> counters -> gather -> experts -> shared expert -> combine, on the
DeepSeek-V2-Lite-shaped layer (H 2048, I 1408, 64 experts top-6, 2 shared
experts).  Weights are random (seeded, generated on the device); 8 weight sets
(11.4 GB) are rotated so that no step finds its weights in the 126 MB L2.

value = algorithmic HBM bytes of the step / device time of the step (GB/s):
  routed INT4 bytes of the unique experts the draft token selects, routed FP16
  bytes of the unique experts the 17 verify tokens select, the FP16 shared
  expert twice, activations, logits and outputs.

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
# DRAM bytes (read + write) of one launch in the ncu captures summarised in
# profiles/ (bench.py --loop, input set 0), with that launch's algorithmic
# bytes.  They describe the kernels as captured: set them to None when a
# kernel changes until it is captured again.
PROFILED_TRAFFIC = {
    "verify": {"dram_bytes": 675_098_624 + 3_160_320, "algorithmic_bytes": 674_897_920,
               "summary": "profiles/engine_kernel_deepseek_v2_lite_verify.md"},
    "draft": {"dram_bytes": 61_515_008 + 109_568, "algorithmic_bytes": 61_374_720,
              "summary": "profiles/draft_kernel_deepseek_v2_lite_draft.md"},
}
NSETS = 8  # default; --sets overrides (profiling captures use fewer)
NINPUTS = 16


def traffic_of(which):
    t = PROFILED_TRAFFIC.get(which)
    return None if t is None else t["dram_bytes"]


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
                                          "--format=csv,noheader,nounits", "-lms", "100"],
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
def make_weight_set(s, idx, torch, spx):
    """Random canonical weights on the device (seeded), repacked for the kernels."""
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
    f16 = spx.spx_f16_repack(normal(E, I, H), normal(E, I, H), normal(E, H, I))
    sh = None
    if s.I_s:
        sh = spx.pack_shared(normal(s.I_s, H), normal(s.I_s, H), normal(H, s.I_s),
                             normal(H) if s.shared_gate else None)
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
    import torch
    from quantized_expert_gb300 import build as spx_build
    from quantized_expert_gb300 import spx

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    if rank == 0 or world == 1:
        spx_build.build()
    if world > 1:
        dist.barrier()
    spx.load()
    s = W.CONFIGS[args.config]
    Td, Tv = s.T_draft, s.T_verify

    sets = [make_weight_set(s, i, torch, spx) for i in range(NSETS)]
    inputs = [make_inputs(s, i) for i in range(NINPUTS)]

    def f16dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.float16)).cuda()

    dev_in = []
    for d in inputs:
        e = dict(x_d=f16dev(d["x_d"]), x_v=f16dev(d["x_v"]))
        e["lg_d"] = torch.from_numpy(d["lg_d"]).cuda() if "lg_d" in d else torch.empty(Td, s.E, device="cuda")
        e["lg_v"] = torch.from_numpy(d["lg_v"]).cuda() if "lg_v" in d else torch.empty(Tv, s.E, device="cuda")
        dev_in.append(e)
    L = s.layers
    elb = torch.zeros(max(L, NSETS), s.E, dtype=torch.int32, device="cuda")
    ws_d = spx.new_workspace(Td, s.H, s.I, s.E, s.k, s.I_s)
    ws_v = spx.new_workspace(Tv, s.H, s.I, s.E, s.k, s.I_s)
    r_d = spx.Routing.empty(Td, s.E, s.k)
    r_v = spx.Routing.empty(Tv, s.E, s.k)
    out_d = torch.empty(Td, s.H, dtype=torch.float16, device="cuda")
    out_v = torch.empty(Tv, s.H, dtype=torch.float16, device="cuda")

    def step_args(i):
        st_d = sets[i % NSETS]
        st_v = sets[(i + NSETS // 2) % NSETS]
        inp = dev_in[i % NINPUTS]
        ad, kd = spx.layer_args(0, inp["x_d"], s.E, s.k, s.renorm, inp["lg_d"], r_d, out_d, ws_d, w4=st_d["w4"],
                                shared=st_d["shared"], w_router=st_d["w_router"], elb=elb, layer=i % NSETS)
        av, kv = spx.layer_args(1, inp["x_v"], s.E, s.k, s.renorm, inp["lg_v"], r_v, out_v, ws_v, f16=st_v["f16"],
                                shared=st_v["shared"], w_router=st_v["w_router"])
        return ad, av, (kd, kv)

    timed_keep = []

    def step_args_timed(i, evd, evv):
        st_d = sets[i % NSETS]
        st_v = sets[(i + NSETS // 2) % NSETS]
        inp = dev_in[i % NINPUTS]
        ad, kd = spx.layer_args(0, inp["x_d"], s.E, s.k, s.renorm, inp["lg_d"], r_d, out_d, ws_d, w4=st_d["w4"],
                                shared=st_d["shared"], w_router=st_d["w_router"], elb=elb, layer=i % NSETS,
                                events=evd)
        av, kv = spx.layer_args(1, inp["x_v"], s.E, s.k, s.renorm, inp["lg_v"], r_v, out_v, ws_v, f16=st_v["f16"],
                                shared=st_v["shared"], w_router=st_v["w_router"], events=evv)
        timed_keep.append((ad, av, kd, kv))
        return ad, av

    # unique experts per input (from the library's own routing) -> algorithmic bytes
    nbytes = []
    nd_list, nv_list = [], []
    for i in range(NINPUTS):
        ad, av, keep = step_args(i)
        spx.spx_moe_layer(ad)
        spx.spx_moe_layer(av)
        torch.cuda.synchronize()
        nd, nv = int(r_d.n_active.item()), int(r_v.n_active.item())
        nd_list.append(nd)
        nv_list.append(nv)
        nbytes.append((layer_bytes(s, "draft", Td, nd), layer_bytes(s, "verify", Tv, nv)))

    stream = torch.cuda.Stream()
    nrot = NSETS * NINPUTS // int(np.gcd(NSETS, NINPUTS))
    keeps = [step_args(i) for i in range(nrot)]

    def sync_all():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
            torch.cuda.synchronize()

    def ev():
        return torch.cuda.Event(enable_timing=True)

    # pass 1: the timed region proper (eager launches; the host enqueues well
    # ahead of the device, so launch overhead is off the clock)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            ad, av, _ = keeps[i % nrot]
            spx.spx_moe_layer(ad, stream)
            spx.spx_moe_layer(av, stream)
    sync_all()
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            e0, e1 = ev(), ev()
            e0.record(stream)
            for i in range(args.steps):
                ad, av, _ = keeps[i % nrot]
                spx.spx_moe_layer(ad, stream)
                spx.spx_moe_layer(av, stream)
            e1.record(stream)
        sync_all()
        ms_total = e0.elapsed_time(e1)
        time.sleep(0.2)
    clocks = clk.summary()

    # pass 2: same steps with events between the layers and around each
    # expert launch (per-layer and per-kernel durations for the roofline)
    lay_ev, ker_ev = [], []
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            a, b, c = ev(), ev(), ev()
            kd, kv = (ev(), ev()), (ev(), ev())
            for e_ in kd + kv:  # create the event; libspx re-records it around the expert launch
                e_.record(stream)
            ad, ae = step_args_timed(i, kd, kv)
            a.record(stream)
            spx.spx_moe_layer(ad, stream)
            b.record(stream)
            spx.spx_moe_layer(ae, stream)
            c.record(stream)
            lay_ev.append((a, b, c))
            ker_ev.append((kd, kv))
    sync_all()
    d_ms = [a.elapsed_time(b) for a, b, c in lay_ev]
    v_ms = [b.elapsed_time(c) for a, b, c in lay_ev]
    kd_ms = [k[0][0].elapsed_time(k[0][1]) for k in ker_ev]
    kv_ms = [k[1][0].elapsed_time(k[1][1]) for k in ker_ev]

    step_bytes = [nbytes[i % NINPUTS] for i in range(args.steps)]
    tot_bytes = sum(d + v for d, v in step_bytes)
    ms_step = ms_total / args.steps
    value, t_max = job_throughput(tot_bytes, ms_total, device="cuda")

    d_bytes = statistics.mean(b[0] for b in step_bytes)
    v_bytes = statistics.mean(b[1] for b in step_bytes)
    d_us = statistics.median(d_ms) * 1e3
    v_us = statistics.median(v_ms) * 1e3
    kd_us = statistics.mean(kd_ms) * 1e3
    kv_us = statistics.mean(kv_ms) * 1e3
    # expert-launch bytes.  Verify: the layer's bytes minus what the routing
    # launch reads.  Draft: the draft launch routes its token itself, so it
    # reads everything the layer reads (a router product, where there is one,
    # runs in a launch of its own before it).
    kv_bytes = v_bytes - Tv * s.E * 4 - (s.E * s.H * 2 if s.logits == "router" else 0)
    kd_bytes = d_bytes - (s.E * s.H * 2 if s.logits == "router" else 0)
    peak, peak_src = measured_peaks()

    # e2e: host buffers through the public API, copies inside the timed region.
    # A serving loop's pipelining: a copy stream moves step i+1's inputs in and
    # step i's outputs out while the compute stream runs step i (two output
    # buffers, events between the streams).
    host_in = []
    for d in inputs:
        h = {k: torch.from_numpy(np.ascontiguousarray(v.view(np.float16) if v.dtype == np.uint16 else v)).pin_memory()
             for k, v in d.items()}
        host_in.append(h)
    host_out_d = torch.empty(Td, s.H, dtype=torch.float16).pin_memory()
    host_out_v = torch.empty(Tv, s.H, dtype=torch.float16).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host_in[0].values())
    d2h = host_out_d.numel() * 2 + host_out_v.numel() * 2
    outs2 = [(out_d, out_v), (torch.empty_like(out_d), torch.empty_like(out_v))]

    def e2e_args(i):
        st_d = sets[i % NSETS]
        st_v = sets[(i + NSETS // 2) % NSETS]
        inp = dev_in[i % NINPUTS]
        od, ov = outs2[i % 2]
        ad, kd = spx.layer_args(0, inp["x_d"], s.E, s.k, s.renorm, inp["lg_d"], r_d, od, ws_d, w4=st_d["w4"],
                                shared=st_d["shared"], w_router=st_d["w_router"], elb=elb, layer=i % NSETS)
        av, kv = spx.layer_args(1, inp["x_v"], s.E, s.k, s.renorm, inp["lg_v"], r_v, ov, ws_v, f16=st_v["f16"],
                                shared=st_v["shared"], w_router=st_v["w_router"])
        return ad, av, (kd, kv)

    nrot2 = nrot if nrot % 2 == 0 else 2 * nrot
    keeps2 = [e2e_args(i) for i in range(nrot2)]
    cstream = torch.cuda.Stream()
    n_all = args.warmup + args.steps
    ev_in = [torch.cuda.Event() for _ in range(n_all)]
    ev_done = [torch.cuda.Event() for _ in range(n_all)]
    ev_out = [torch.cuda.Event() for _ in range(n_all)]

    def h2d_step(i):
        with torch.cuda.stream(cstream):
            h = host_in[i % NINPUTS]
            inp = dev_in[i % NINPUTS]
            for k, v in h.items():
                inp[k].copy_(v, non_blocking=True)
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
            h2d_step(i + 1)  # the next step's inputs, during this step's layers
        with torch.cuda.stream(stream):
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])  # this output buffer has been read back
            ad, av, _ = keeps2[i % nrot2]
            spx.spx_moe_layer(ad, stream)
            spx.spx_moe_layer(av, stream)
            ev_done[i].record(stream)
        with torch.cuda.stream(cstream):
            cstream.wait_event(ev_done[i])
            od, ov = outs2[i % 2]
            host_out_d.copy_(od, non_blocking=True)
            host_out_v.copy_(ov, non_blocking=True)
            ev_out[i].record(cstream)
    cstream.synchronize()
    stream.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_gbs, _ = job_throughput(tot_bytes, e2e_s * 1e3, device="cuda")  # slowest rank's wall time

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 (int4 draft weights, fp32 accumulate)",
        "data": "synthetic (seeded random weights and activations; drawn Zipf(1.1) router logits)",
        "config": {"workload": f"{s.name} layer: draft T={Td} + verify T={Tv}", "H": s.H, "I": s.I, "E": s.E,
                   "k": s.k, "I_shared": s.I_s, "draft_T": Td, "verify_T": Tv,
                   "l2": f"{NSETS} rotated weight sets ({NSETS * 1.43:.1f} GB) > L2; no flush",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "unique_experts_draft": statistics.mean(nd_list), "unique_experts_verify": statistics.mean(nv_list)},
        "layers": {"draft_us": round(d_us, 2), "draft_gbs": round(d_bytes / (d_us * 1e-6) / 1e9, 1),
                   "draft_frac": round(d_bytes / (d_us * 1e-6) / 1e9 / peak, 3),
                   "draft_tokens_per_s": round(Td / (d_us * 1e-6), 1),
                   "verify_us": round(v_us, 2), "verify_gbs": round(v_bytes / (v_us * 1e-6) / 1e9, 1),
                   "verify_frac": round(v_bytes / (v_us * 1e-6) / 1e9 / peak, 3),
                   "verify_tokens_per_s": round(Tv / (v_us * 1e-6), 1),
                   "draft_bytes": int(d_bytes), "verify_bytes": int(v_bytes),
                   "draft_us_spread": spread_us(d_ms), "verify_us_spread": spread_us(v_ms)},
        "roofline": {"bound": "hbm", "kernel": "engine_kernel<1,1,3> (verify expert launch, FP16 experts)",
                     "achieved": round(kv_bytes / (kv_us * 1e-6) / 1e9, 1), "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s",
                     "frac": round(kv_bytes / (kv_us * 1e-6) / 1e9 / peak, 3),
                     "traffic": traffic_of("verify"), "traffic_capture": PROFILED_TRAFFIC["verify"],
                     "launch_us": round(kv_us, 2), "bytes_per_launch": int(kv_bytes)},
        "draft_roofline": {"bound": "hbm", "kernel": "draft_kernel<2, 0> (draft launch: routing + INT4 experts)",
                           "achieved": round(kd_bytes / (kd_us * 1e-6) / 1e9, 1), "peak": peak, "unit": "GB/s",
                           "frac": round(kd_bytes / (kd_us * 1e-6) / 1e9 / peak, 3), "launch_us": round(kd_us, 2),
                           "bytes_per_launch": int(kd_bytes), "traffic": traffic_of("draft"),
                           "traffic_capture": PROFILED_TRAFFIC["draft"]},
        "clocks": clocks,
        "e2e": {"value": round(e2e_gbs, 1), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        # per step: the draft launch (+ the router product when the layer has a
        # router weight), the verify routing launch, the verify expert launch
        "gpu_launches": (3 + (1 if s.logits == "router" else 0)) * args.steps,
    }
    if rank == 0 and args.cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(s)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


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
            "sample": f"1 draft (T={s.T_draft}) + 1 verify (T={s.T_verify}) layer of {s.name}, input set 0, "
                      f"{reps} rep(s), {dt:.2f} s per step"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    s = W.CONFIGS[args.config]
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
            "config": {"workload": f"{s.name} layer: draft T={s.T_draft} + verify T={s.T_verify}"},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": cb["sample"]},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_cycle(args):
    """The 26-layer draft-then-verify cycle: K draft steps at T = 1 through every
    layer (Expert Lookahead Buffer counters on), then one verify pass at T = K+1;
    independent weights per layer.  Prints one JSON line: device us per cycle,
    achieved GB/s of the cycle's algorithmic bytes, ELB distinct experts per layer."""
    import torch
    from quantized_expert_gb300 import build as B, spx
    import oracle
    B.build()
    spx.load()
    s = W.CONFIGS["deepseek_v2_lite_x26"]
    L, K, E, k, Tv = s.layers, s.K, s.E, s.k, s.T_verify
    lays = [make_weight_set(s, l, torch, spx) for l in range(L)]

    def f16dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.float16)).cuda()
    xd = {(st, l): f16dev(W.gen_x(s, 1, layer=l, step=st)) for st in range(1, K + 1) for l in range(L)}
    lgd = {(st, l): torch.from_numpy(W.draft_logits(s, l, st)).cuda() for st in range(1, K + 1) for l in range(L)}
    xv = [f16dev(W.gen_x(s, Tv, layer=l, step=K + 1, which=1)) for l in range(L)]
    lgv = [torch.from_numpy(W.verify_logits(s, l)).cuda() for l in range(L)]
    # algorithmic bytes of one cycle (unique experts of every call, from the drawn logits)
    cyc_bytes = 0
    for l in range(L):
        for st in range(1, K + 1):
            ids, _ = oracle.route_topk(W.draft_logits(s, l, st).astype(np.float64), k, s.renorm)
            cyc_bytes += layer_bytes(s, "draft", 1, len(set(ids.reshape(-1).tolist())))
        ids, _ = oracle.route_topk(W.verify_logits(s, l).astype(np.float64), k, s.renorm)
        cyc_bytes += layer_bytes(s, "verify", Tv, len(set(ids.reshape(-1).tolist())))
    elb = torch.zeros(L, E, dtype=torch.int32, device="cuda")
    ws_d, ws_v = spx.new_workspace(1, s.H, s.I, E, k, s.I_s), spx.new_workspace(Tv, s.H, s.I, E, k, s.I_s)
    r_d, r_v = spx.Routing.empty(1, E, k), spx.Routing.empty(Tv, E, k)
    out_d = torch.empty(1, s.H, dtype=torch.float16, device="cuda")
    out_v = torch.empty(Tv, s.H, dtype=torch.float16, device="cuda")
    draft_args = [[spx.layer_args(0, xd[(st, l)], E, k, s.renorm, lgd[(st, l)], r_d, out_d, ws_d,
                                  w4=lays[l]["w4"], shared=lays[l]["shared"], elb=elb, layer=l)
                   for l in range(L)] for st in range(1, K + 1)]
    verify_args = [spx.layer_args(1, xv[l], E, k, s.renorm, lgv[l], r_v, out_v, ws_v, f16=lays[l]["f16"],
                                  shared=lays[l]["shared"]) for l in range(L)]
    stream = torch.cuda.Stream()

    def cycle():
        spx.spx_elb_reset(elb, stream)
        for st in range(K):
            for l in range(L):
                spx.spx_moe_layer(draft_args[st][l][0], stream)
        for l in range(L):
            spx.spx_moe_layer(verify_args[l][0], stream)

    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup)):
            cycle()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = max(1, args.steps)
        e0.record(stream)
        for _ in range(n):
            cycle()
        e1.record(stream)
        torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / n
    got = elb.cpu().numpy()
    distinct = (got > 0).sum(1)
    peak, peak_src = measured_peaks()
    gbs = cyc_bytes / (us * 1e-6) / 1e9
    line = {"metric": "26-layer draft-then-verify cycle, device us per cycle", "value": round(us, 1), "unit": "us",
            "higher_is_better": False, "n_gpus": 1, "steps": n, "warmup": max(1, args.warmup),
            "data": "synthetic (independent seeded weights per layer; drawn Zipf(1.1) router logits)",
            "config": {"workload": f"{s.name}: {K} draft steps (T=1) x {L} layers + verify (T={Tv}) x {L} layers",
                       "layer_calls_per_cycle": (K + 1) * L},
            "achieved_gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 3), "peak": peak,
            "peak_source": peak_src, "bytes_per_cycle": int(cyc_bytes),
            "elb_distinct_experts_per_layer": {"mean": round(float(distinct.mean()), 2), "min": int(distinct.min()),
                                               "max": int(distinct.max())},
            "elb_calls_per_layer": int(got.sum(1)[0]) // k}
    print(json.dumps(line), flush=True)


def run_loop(args):
    """Profiling driver: --loop-n layer calls of one mode on --sets weight sets,
    no timing (the command that ncu captures wrap)."""
    import torch
    from quantized_expert_gb300 import build as B, spx
    B.build()
    spx.load()
    s = W.CONFIGS[args.config]
    sets = [make_weight_set(s, i, torch, spx) for i in range(NSETS)]
    inp = make_inputs(s, 0)
    draft = args.loop == "draft"
    T = s.T_draft if draft else s.T_verify
    xk, lk = ("x_d", "lg_d") if draft else ("x_v", "lg_v")
    x = torch.from_numpy(np.ascontiguousarray(inp[xk]).view(np.float16)).cuda()
    lg = torch.from_numpy(inp[lk]).cuda() if lk in inp else torch.empty(T, s.E, device="cuda")
    ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s)
    r = spx.Routing.empty(T, s.E, s.k)
    out = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
    keep = [spx.layer_args(0 if draft else 1, x, s.E, s.k, s.renorm, lg, r, out, ws,
                           w4=st["w4"] if draft else None, f16=None if draft else st["f16"], shared=st["shared"],
                           w_router=st["w_router"]) for st in sets]
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
    """Draft layers carrying T = 1, 2, 4, 8 tokens (one per request) in one
    call: device us per layer, unique experts, algorithmic GB/s and draft
    tokens/s.  Prints one JSON line."""
    import torch
    from quantized_expert_gb300 import build as B, spx
    B.build()
    spx.load()
    s = W.CONFIGS[args.config]
    sets = [make_weight_set(s, i, torch, spx) for i in range(NSETS)]
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
    peak, peak_src = measured_peaks()
    rows = []
    stream = torch.cuda.Stream()
    for T in (1, 2, 4, 8):
        xs = [torch.from_numpy(np.ascontiguousarray(W.gen_x(s, T, step=i)).view(np.float16)).cuda()
              for i in range(NINPUTS)]
        lgs = [torch.from_numpy(W.gen_logits(s, T, step=i)).cuda() if s.logits != "router"
               else torch.empty(T, s.E, device="cuda") for i in range(NINPUTS)]
        ws = spx.new_workspace(T, s.H, s.I, s.E, s.k, s.I_s)
        r = spx.Routing.empty(T, s.E, s.k)
        out = torch.empty(T, s.H, dtype=torch.float16, device="cuda")
        keep = [spx.layer_args(0, xs[i % NINPUTS], s.E, s.k, s.renorm, lgs[i % NINPUTS], r, out, ws,
                               w4=sets[i % NSETS]["w4"], shared=sets[i % NSETS]["shared"],
                               w_router=sets[i % NSETS]["w_router"], gguf=sets[i % NSETS].get("gguf"))
                for i in range(NSETS * NINPUTS)]
        nb = []
        for i in range(NINPUTS):
            spx.spx_moe_layer(keep[i][0])
            torch.cuda.synchronize()
            nb.append((int(r.n_active.item()),
                       layer_bytes(s, "draft", T, int(r.n_active.item()), args.zeros, args.gguf)))
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
    line = {"metric": "draft layer with T requests' tokens per call, device us per layer",
            "config": {"workload": f"{s.name} draft{zp}, T = 1, 2, 4, 8 (one token per request)"},
            "peak": peak, "peak_source": peak_src, "rows": rows, "steps": args.steps, "warmup": args.warmup}
    print(json.dumps(line), flush=True)


TL_EVENTS = ["entry", "prod_static", "prod_griddep", "x_staged", "routed", "first_fill", "gu_last", "dn_w_first",
             "dn_h_first", "dn_last", "prod_last", "cons_done", "out_done", "sg_last", "rg_first", "rg_last",
             "w_full", "w_hfull", "w_empty", "n_sg", "n_rg", "n_sd", "n_rd", "exit", "rd_h_last", "sd_last",
             "w_poll", "bytes"]
TL_FIRST_EV = {"entry", "prod_static", "prod_griddep", "x_staged", "routed", "first_fill", "dn_w_first",
               "dn_h_first", "cons_done", "rg_first"}
TL_SUM_EV = {"w_full", "w_hfull", "w_empty", "n_sg", "n_rg", "n_sd", "n_rd", "w_poll", "bytes"}


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
    buf = np.zeros((8, 256, 32), np.uint64)

    def read():
        torch.cuda.synchronize()
        assert lib.spx_timeline_read(buf.ctypes.data, buf.size) == 0
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
            "chained": timeline_phases(chained, range(1, 8), nsm)}
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
    ap.add_argument("--cycle", action="store_true", help="the 26-layer draft-then-verify cycle (prints its own line)")
    ap.add_argument("--loop-n", type=int, default=12)
    ap.add_argument("--cached", action="store_true", help="cache-aware verify vs plain (prints its own line)")
    ap.add_argument("--draft-batch", action="store_true", help="draft layers at T = 1, 2, 4, 8 (prints its own line)")
    ap.add_argument("--zeros", action="store_true", help="with --draft-batch: INT4 experts with per-group zero points")
    ap.add_argument("--gguf", choices=["q8_0", "q2_k", "q4_k"], help="with --draft-batch: GGUF experts instead of INT4")
    ap.add_argument("--timeline", action="store_true",
                    help="draft launch phase marks from the profiling build (prints its own line)")
    args = ap.parse_args()
    globals()["NSETS"] = max(1, args.sets)
    if args.timeline:
        run_timeline(args)
    elif args.loop:
        run_loop(args)
    elif args.cached:
        run_cached(args)
    elif args.draft_batch:
        run_draft_batch(args)
    elif args.cycle:
        run_cycle(args)
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
