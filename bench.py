#!/usr/bin/env python3
"""Benchmark of the batch-1 fine-grained MoE verify step on GB300.

Workload (one "step"): the full verify step at M = 5 tokens (gamma = 4):
30 MoE layers of the Gemma-4-26B-A4B shape (128 routed + 1 shared expert,
2816 x 704, E4M3 weights with per-row fp32 scales, Zipf(1.1) router bias,
per-layer seeds 1..30), pre-RMSNorm and residual per layer, a final RMSNorm,
the 262,144 x 2816 bf16 tied lm_head with argmax, and greedy acceptance of 4
drafts that copy the target's argmax with probability 0.7. Eight input batches
(hidden seeds 31..38) and 64 draft seeds (33..96, seed k on batch k mod 8)
rotate across steps. Weights are random-init, inputs synthetic.

Metric: verified tokens/s with every input resident in HBM, and the achieved
HBM GB/s of the step's unique weight bytes against the measured copy
bandwidth. `value` counts 1 + E[a] tokens per step, E[a] = 0.7 + 0.7^2 +
0.7^3 + 0.7^4 = 1.7731 being the expected accepted count of the draft recipe;
the line also gives tokens/s at the accepted counts of the timed steps and the
mean accepted count over all 64 draft seeds. A step streams > 5 GB of weights,
far above the 129 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified tokens/s at batch 1 (gamma=4); achieved HBM GB/s vs 8 TB/s roofline"
M = 5
GAMMA = M - 1
S_ZIPF = 1.1
N_LAYERS = 30
N_BATCHES = 8
HIDDEN_SEED0 = 31
DRAFT_SEED0 = 33
N_DRAFT_SEEDS = 64
P_COPY = 0.7   # probability that a draft copies the target's argmax
EMB_SEED = 32
# --path names and the library's path constants
PATHS = {"fused": "PATH_FUSED", "staged": "PATH_STAGED", "fused_tc": "PATH_FUSED_TC", "fused_mma": "PATH_FUSED_MMA"}
WORKLOAD = ("full verify step: 30-layer FP8 MoE stack (Gemma-4-26B-A4B shape, Zipf s=1.1) + "
            "final RMSNorm + 262144x2816 bf16 tied lm_head argmax + greedy accept, M=5 (gamma=4)")
FALLBACK_HBM_GBS = 6800.0
ROOFLINE_TARGET_GBS = 8000.0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def expected_accept(gamma: int, p: float = P_COPY) -> float:
    """Expected greedy accepted count when each draft copies the target's argmax
    with probability p, independently: a >= j exactly when the first j drafts
    all copy it, so E[a] = sum_{j=1..gamma} p^j (a uniform draft that hits the
    argmax by chance, 1 in 262,144, is neglected)."""
    return sum(p ** j for j in range(1, gamma + 1))


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------- ncu traffic
KERNEL_SOURCES = ("fine_grained_moe_gb300/csrc/fused_step.cuh", "fine_grained_moe_gb300/csrc/common.cuh",
                  "fine_grained_moe_gb300/csrc/fgm.cu")
TRAFFIC_PROFILE = os.path.join("profiles", "k_fused_verify_step_traffic.md")


def kernel_source_hash():
    """sha256 over the sources of the persistent kernel (a changed kernel voids
    a traffic figure taken on an older one)."""
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def captured_traffic():
    """DRAM bytes (read + write) of one verify-step launch from the committed ncu
    summary, or None when that summary was taken on other kernel sources."""
    try:
        with open(os.path.join(ROOT, TRAFFIC_PROFILE)) as f:
            text = f.read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if ":" in line and line.startswith("- "):
            k, v = line[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel sources sha256") != kernel_source_hash():
        return None
    try:
        return int(fields["traffic per launch (bytes)"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- workload
def make_workload(device, n_layers=N_LAYERS, vocab=262144):
    import torch

    import synth
    t0 = time.time()
    layers = [synth.layer(l + 1, device=device, s=S_ZIPF) for l in range(n_layers)]
    emb = synth.embedding(EMB_SEED, device=device, vocab=vocab)
    xs = [synth.hidden_states(HIDDEN_SEED0 + b, M, device=device) for b in range(N_BATCHES)]
    torch.cuda.synchronize()
    log(f"[bench] generated weights in {time.time() - t0:.1f}s")
    return layers, emb, xs


def cpu_oracle_step(layers, emb, x, draft_seed, log_prefix="[oracle]"):
    """One full verify step of the oracle on host copies of the same inputs.
    Returns (seconds of oracle compute, accepted, next, cores). Host copies are
    made layer by layer and are not timed."""
    import numpy as np
    import torch

    import oracle
    import synth
    h = x.detach().cpu().double().numpy()
    compute = 0.0
    for p in layers:
        host = {k: (None if v is None else v.detach().cpu()) for k, v in p.items()}
        L = oracle.LayerParams(
            router_w=host["router_w"].view(torch.int16).numpy().view(np.uint16),
            router_b=None if host["router_b"] is None else host["router_b"].numpy(),
            gate_q=host["gate_q"].numpy(), gate_s=host["gate_s"].numpy(), up_q=host["up_q"].numpy(),
            up_s=host["up_s"].numpy(), down_q=host["down_q"].numpy(), down_s=host["down_s"].numpy())
        t0 = time.perf_counter()
        h = oracle.stack_layer(L, h).y
        compute += time.perf_counter() - t0
        del L, host
    e = emb.detach().cpu().view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    hn = oracle.bf16_to_f64(oracle.bf16_round(oracle.rmsnorm(h)))
    am, _, _ = oracle.lm_head(e, hn)
    compute += time.perf_counter() - t0
    draft = synth.drafts(draft_seed, am).numpy()
    a, nxt = oracle.spec_verify(am, draft)
    log(f"{log_prefix} full step: {compute:.2f}s compute, accepted {a}, cores {oracle.num_threads()}")
    return compute, a, nxt, oracle.num_threads()


def cpu_oracle_single_thread(layers, emb, x, n_layers=2):
    """The oracle on one thread, on a bounded sample of the step: the first
    n_layers layers and the same fraction of the lm_head rows, scaled to a full
    step. Returns (seconds per full step, sample description)."""
    import numpy as np
    import torch

    import oracle
    frac = n_layers / N_LAYERS
    host = []
    for p in layers[:n_layers]:
        h = {k: (None if v is None else v.detach().cpu()) for k, v in p.items()}
        host.append(oracle.LayerParams(
            router_w=h["router_w"].view(torch.int16).numpy().view(np.uint16),
            router_b=None if h["router_b"] is None else h["router_b"].numpy(),
            gate_q=h["gate_q"].numpy(), gate_s=h["gate_s"].numpy(), up_q=h["up_q"].numpy(),
            up_s=h["up_s"].numpy(), down_q=h["down_q"].numpy(), down_s=h["down_s"].numpy()))
    v_rows = int(emb.shape[0] * frac)
    e = emb[:v_rows].detach().cpu().view(torch.int16).numpy().view(np.uint16)
    prev = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        t0 = time.perf_counter()
        h = x.detach().cpu().double().numpy()
        for L in host:
            h = oracle.stack_layer(L, h).y
        oracle.lm_head(e, oracle.bf16_to_f64(oracle.bf16_round(oracle.rmsnorm(h))))
        secs = (time.perf_counter() - t0) / frac
    finally:
        oracle.set_num_threads(prev)
    log(f"[oracle] one thread: {secs:.2f}s per full step (scaled from {n_layers} layers)")
    return secs, (f"one thread: first {n_layers} of {N_LAYERS} layers + {v_rows} of {emb.shape[0]} lm_head rows "
                  f"on batch 0, scaled x{1 / frac:.0f}")


# ---------------------------------------------------------------- phase trace
TRACE_POINTS = ("layer start", "norm/router partials", "partials reduced", "activation terms",
                "shared gate/up done", "barrier 1 passed", "routing known", "routed gate/up done",
                "barrier 2 passed", "down done", "top-k done", "expert list done")
TRACE_ORDER = (1, 2, 3, 4, 5, 10, 11, 6, 7, 8, 9)   # the points in the order a layer reaches them
NTP = len(TRACE_POINTS)
TRACE_STAGES = 48


def write_phase_trace(path, fgm, layers, emb, x, draft, ws, arr, dev):
    """One traced verify step: per layer and phase, the time at which the last
    CTA (and the median CTA) reached each phase boundary, relative to the
    first CTA starting the layer, averaged over the layers; then the ring
    stages of two layers as seen by CTA G/2."""
    import torch
    G = torch.cuda.get_device_properties(dev).multi_processor_count
    n = (N_LAYERS * NTP + 2) * G + N_LAYERS * TRACE_STAGES * 8
    buf = torch.zeros(n, dtype=torch.int64, device=dev)
    fgm.set_phase_trace(buf)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    fgm.verify_step(layers, emb, x, draft, ws=ws, _arr=arr)
    t1.record()
    torch.cuda.synchronize()
    fgm.set_phase_trace(None)
    flat = buf.cpu().double()
    tr = flat[:(N_LAYERS * NTP + 2) * G].view(-1, G)
    det = flat[(N_LAYERS * NTP + 2) * G:].view(N_LAYERS, TRACE_STAGES, 8)
    lines = [f"one traced verify step: {t0.elapsed_time(t1) * 1e3:.1f} us (CUDA events), G = {G} CTAs"]
    last = [0.0] * NTP
    med = [0.0] * NTP
    period = 0.0
    for l in range(N_LAYERS):
        base = tr[l * NTP].min()
        nxt = tr[(l + 1) * NTP].min() if l + 1 < N_LAYERS else tr[N_LAYERS * NTP].min()
        period += float(nxt - base) / 1e3 / N_LAYERS
        for k in range(NTP):
            last[k] += float(tr[l * NTP + k].max() - base) / 1e3 / N_LAYERS
            med[k] += float(tr[l * NTP + k].median() - base) / 1e3 / N_LAYERS
    lines.append(f"mean layer period (first CTA to first CTA): {period:.2f} us")
    lines.append("point                      last CTA (us)   median CTA (us)   from layer start")
    for k in TRACE_ORDER:
        lines.append(f"{TRACE_POINTS[k]:26s} {last[k]:12.2f} {med[k]:16.2f}")
    # per-CTA mean over layers of "down done" (from each layer's first start): stragglers
    dd = torch.zeros(G, dtype=torch.float64)
    gd = torch.zeros(G, dtype=torch.float64)
    for l in range(N_LAYERS):
        base = tr[l * NTP].min()
        dd += (tr[l * NTP + 9] - base) / 1e3 / N_LAYERS
        gd += (tr[l * NTP + 7] - base) / 1e3 / N_LAYERS
    order = torch.argsort(dd, descending=True)
    lines.append("slowest CTAs (mean down done / routed gate/up done, us): " + ", ".join(
        f"{int(c)}: {float(dd[c]):.2f}/{float(gd[c]):.2f}" for c in order[:8]))
    lines.append(f"down done p10/p50/p90: {float(dd.quantile(0.1)):.2f} / {float(dd.quantile(0.5)):.2f} / "
                 f"{float(dd.quantile(0.9)):.2f} us")
    tail = tr[N_LAYERS * NTP + 1].max() - tr[N_LAYERS * NTP].min()
    lines.append(f"lm_head + accept (last CTA end - first CTA after layers): {float(tail) / 1e3:.2f} us")
    for l in (1, N_LAYERS // 2):
        base = float(det[l, 0, 7])
        lines.append(f"CTA {G // 2}, layer {l}: stage  issue  wait-from  landed  products  released  posted"
                     f"  (SM cycles from its layer start)")
        for k in range(TRACE_STAGES):
            row = det[l, k]
            if row[1] == 0:
                break
            vals = ["%8d" % int(float(row[c]) - base) if row[c] != 0 else "       -" for c in (0, 5, 1, 2, 3, 4)]
            lines.append(f"  {k:3d}  " + "  ".join(vals))
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")
    log("\n".join(lines[:NTP + 3]))


# ---------------------------------------------------------------- replicas
def reduce_over_ranks(total_ms, tokens, e2e_s, e2e_tokens, device):
    """Whole-job numbers of N independent replicas: the slowest rank's time and
    the tokens of all ranks (torch.distributed all_gather; NCCL on GPUs, gloo
    in the CPU tests)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([total_ms, tokens, e2e_s, e2e_tokens], dtype=torch.float64, device=device)
    parts = [torch.zeros_like(t) for _ in range(dist.get_world_size())]
    dist.all_gather(parts, t)
    return (max(float(q[0]) for q in parts), sum(float(q[1]) for q in parts),
            max(float(q[2]) for q in parts), sum(float(q[3]) for q in parts))


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, world):
    import torch

    import fine_grained_moe_gb300 as fgm
    import synth
    from fine_grained_moe_gb300 import traffic

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    fgm.lib()
    fgm.select_path(getattr(fgm, PATHS[args.path]))
    nl, V = args.layers, args.vocab
    full_size = (nl, V) == (N_LAYERS, 262144)
    if args.phase_trace and not full_size:
        raise SystemExit("--phase-trace needs the full-size step")
    layers, emb, xs = make_workload(dev, nl, V)
    arr = fgm.layers_array(layers)
    ws = fgm.Workspace(dev)
    stream = torch.cuda.current_stream()

    # per-batch routing (unique experts per layer) and the target's argmax; draft
    # seed k drafts for batch k mod 8
    uniq, ams = [], []
    trace = torch.empty((nl, M, 8), dtype=torch.int32, device=dev)
    for b, x in enumerate(xs):
        fgm.moe_stack_fwd(layers, x, ids_trace=trace, ws=ws)
        tr = trace.cpu()
        uniq.append([len(torch.unique(tr[l])) for l in range(nl)])
        am = torch.empty(M, dtype=torch.int32, device=dev)
        fgm.verify_step(layers, emb, x, torch.zeros(GAMMA, dtype=torch.int32, device=dev), argmax=am,
                        ws=ws, _arr=arr)
        ams.append(am.cpu())
    drafts = [synth.drafts(DRAFT_SEED0 + k, ams[k % N_BATCHES]).to(dev) for k in range(N_DRAFT_SEEDS)]
    step_bytes = [traffic.step_bytes(u, vocab=V) for u in uniq]
    K, W = args.steps, args.warmup
    # accepted count of every (batch, draft seed) pair, untimed
    acc_all = torch.zeros((N_DRAFT_SEEDS, 2), dtype=torch.int32, device=dev)
    for k in range(N_DRAFT_SEEDS):
        fgm.verify_step(layers, emb, xs[k % N_BATCHES], drafts[k], out=acc_all[k], ws=ws, _arr=arr)
    accepted_mean_all = float(acc_all[:, 0].double().mean())
    outs = torch.zeros((K, 2), dtype=torch.int32, device=dev)
    for i in range(W):
        k = i % N_DRAFT_SEEDS
        fgm.verify_step(layers, emb, xs[k % N_BATCHES], drafts[k], ws=ws, _arr=arr)
    torch.cuda.synchronize()

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        ev[0].record(stream)
        for i in range(K):
            k = i % N_DRAFT_SEEDS
            fgm.verify_step(layers, emb, xs[k % N_BATCHES], drafts[k], out=outs[i], ws=ws, _arr=arr)
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    per_step = [ev[i].elapsed_time(ev[i + 1]) for i in range(K)]
    total_ms = ev[0].elapsed_time(ev[K])
    status = ws.status()
    acc = outs.cpu()
    tokens = int(acc[:, 0].sum()) + K
    bytes_total = sum(step_bytes[(i % N_DRAFT_SEEDS) % N_BATCHES] for i in range(K))

    if args.phase_trace:
        write_phase_trace(args.phase_trace, fgm, layers, emb, xs[0], drafts[0], ws, arr, dev)

    # end to end through the host-buffer entry point
    x_h = [x.cpu().pin_memory() for x in xs]
    d_h = [d.cpu().pin_memory() for d in drafts]
    o_h = torch.empty(2, dtype=torch.int32).pin_memory()
    for i in range(min(W, 3)):
        fgm.verify_step_host(layers, emb, x_h[i % N_BATCHES], d_h[i], out_host=o_h, ws=ws, _arr=arr)
    t0 = time.perf_counter()
    e2e_tokens = 0
    for i in range(K):
        k = i % N_DRAFT_SEEDS
        fgm.verify_step_host(layers, emb, x_h[k % N_BATCHES], d_h[k], out_host=o_h, ws=ws, _arr=arr)
        e2e_tokens += int(o_h[0]) + 1
    e2e_s = time.perf_counter() - t0

    # max time and summed tokens over ranks (replicas)
    if world > 1:
        total_ms_max, tokens_all, e2e_max, e2e_tok_all = reduce_over_ranks(
            total_ms, tokens, e2e_s, e2e_tokens, dev)
    else:
        total_ms_max, tokens_all, e2e_max, e2e_tok_all = total_ms, tokens, e2e_s, e2e_tokens
    if rank != 0:
        return None

    peak, peak_kind = measured_peaks()
    ms = total_ms_max / K
    achieved = bytes_total / K / (ms * 1e-3) / 1e9
    clocks = clk.summary()
    ea = expected_accept(GAMMA)
    line = {
        "metric": METRIC,
        "value": round(world * K * (1 + ea) / (total_ms_max * 1e-3), 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 weights, fp32 accumulate; bf16 lm_head",
        "data": "synthetic (random-init weights of the Gemma-4-26B-A4B MoE shape, seeded)",
        "config": {
            "workload": WORKLOAD if full_size else
            f"profiling case: {nl}-layer FP8 MoE stack + {V}-word bf16 lm_head, otherwise as the full step",
            "M": M, "gamma": GAMMA, "zipf_s": S_ZIPF, "layers": nl, "vocab": V, "batches": N_BATCHES, "parallelism": f"replicas x{world}",
            "l2": "no flush: each step streams > 5 GB of weights (L2 is 129 MB)",
            "mean_unique_experts_per_layer": round(statistics.mean(sum(uniq, [])), 2),
            "draft_seeds": N_DRAFT_SEEDS,
            "algorithmic_bytes_by_batch": [int(b) for b in step_bytes],
            "tokens_per_step": f"value counts 1 + E[a] = {1 + ea:.4f} (E[a] = sum of 0.7^j, j = 1..4)",
        },
        "hbm_gbs": round(achieved, 1),
        "frac_of_8tbs": round(achieved / ROOFLINE_TARGET_GBS, 4),
        "expected_accept": round(ea, 4),
        "tokens_per_s_measured_accept": round(tokens_all / (total_ms_max * 1e-3), 2),
        "accepted_per_step": round((tokens - K) / K, 3),
        "accepted_mean_all_draft_seeds": round(accepted_mean_all, 3),
        "p50_ms": round(statistics.median(per_step), 4),
        "p99_ms": round(sorted(per_step)[min(K - 1, int(0.99 * K))], 4),
        "path": args.path,
        "roofline": {
            "kernel": ("k_fused (one persistent launch per step)" if args.path != "staged"
                       else "verify step (all launches of one step)"),
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": f"{peak_kind} copy bandwidth",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": (captured_traffic() if args.path != "staged" and full_size else None),
            "algorithmic_bytes_per_launch": int(bytes_total / K),
        },
        "e2e": {"value": round(world * K * (1 + ea) / e2e_max, 2), "unit": "tokens/s",
                "measured_accept_value": round(e2e_tok_all / e2e_max, 2),
                "h2d_bytes_per_step": M * 2816 * 2 + GAMMA * 4, "d2h_bytes_per_step": 8},
        "gpu_launches": K * (1 if args.path != "staged" else 1 + nl * 5 + 3),
        "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                   "reasons": clocks["reasons"]},
        "status": status,
    }
    if world == 1 and full_size and not args.no_cpu_baseline:
        secs, a, _, cores = cpu_oracle_step(layers, emb, xs[0], DRAFT_SEED0)
        secs1, sample1 = cpu_oracle_single_thread(layers, emb, xs[0])
        line["cpu_baseline"] = {"value": round((1 + ea) / secs, 4), "unit": "tokens/s", "cores": cores,
                                "kind": "oracle", "cpu_model": cpu_model(),
                                "sample": "one full verify step (30 layers + lm_head + accept) on batch 0, "
                                          f"1 + E[a] tokens; host weight copies untimed; accepted count {a}",
                                "ms_per_step": round(secs * 1e3, 1),
                                "single_thread": {"value": round((1 + ea) / secs1, 4), "unit": "tokens/s",
                                                  "cores": 1, "ms_per_step": round(secs1 * 1e3, 1),
                                                  "sample": sample1}}
    return line


# ---------------------------------------------------------------- single-stage cases
def run_case(args):
    """One stage alone, for profiling: `layer` = one MoE layer at M = 5 with the
    Zipf(1.1) bias (four weight copies and eight inputs rotate, so L2 never
    serves a repeated expert); `lm_head` / `lm_head_fp8` = the 262,144-word
    lm_head argmax at M = 5, bf16 or E4M3 rows (one call = the argmax kernel
    and the cross-CTA reduction). Prints a JSON line with the stage's HBM GB/s."""
    import torch

    import fine_grained_moe_gb300 as fgm
    import synth
    from fine_grained_moe_gb300 import traffic

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fgm.lib()
    fgm.select_path(getattr(fgm, PATHS[args.path]))
    ws = fgm.Workspace(dev)
    xs = [synth.hidden_states(HIDDEN_SEED0 + b, M, device=dev) for b in range(N_BATCHES)]
    K, W = args.steps, args.warmup
    if args.case == "layer":
        copies = [synth.layer(1 + c, device=dev, s=S_ZIPF) for c in range(4)]
        ids = torch.empty((M, 8), dtype=torch.int32, device=dev)
        calls, nbytes = [], []
        for i in range(max(K, W)):
            p, x = copies[i % 4], xs[i % N_BATCHES]
            fgm.moe_layer_fwd(p, x, topk_ids=ids, ws=ws)
            u = len(torch.unique(ids.cpu()))
            nbytes.append(traffic.step_bytes([u], with_lm_head=False))
            calls.append((p, x))
        run = lambda i: fgm.moe_layer_fwd(calls[i][0], calls[i][1], ws=ws)
        unit_bytes = nbytes
        name = "one MoE layer, M=5, Zipf s=1.1 (4 weight copies rotate)"
    elif args.case == "layer_dense":
        copies = [synth.layer(1 + c, device=dev, s=S_ZIPF) for c in range(4)]
        denses = [synth.dense_mlp(100 + c, device=dev) for c in range(4)]
        ids = torch.empty((M, 8), dtype=torch.int32, device=dev)
        calls, nbytes = [], []
        for i in range(max(K, W)):
            p, d, x = copies[i % 4], denses[i % 4], xs[i % N_BATCHES]
            fgm.moe_layer_dense_fwd(p, d, x, topk_ids=ids, ws=ws)
            nbytes.append(traffic.layer_dense_bytes(len(torch.unique(ids.cpu()))))
            calls.append((p, d, x))
        run = lambda i: fgm.moe_layer_dense_fwd(calls[i][0], calls[i][1], calls[i][2], ws=ws)
        unit_bytes = nbytes
        name = ("one MoE layer with the 2816x2112 dense MLP in place of the shared expert, M=5, Zipf s=1.1 "
                "(4 weight copies rotate)")
    elif args.case == "lm_head_fp8":
        emb_q, emb_s = synth.embedding_fp8(synth.embedding(EMB_SEED, device=dev))
        torch.cuda.empty_cache()
        am = torch.empty(M, dtype=torch.int32, device=dev)
        run = lambda i: fgm.lm_head_argmax_fp8(emb_q, emb_s, xs[i % N_BATCHES], argmax=am, ws=ws)
        unit_bytes = [traffic.lm_head_fp8_bytes()] * max(K, W)
        name = "lm_head argmax, 262144 x 2816 E4M3 + fp32 row scales, M=5"
    else:
        emb = synth.embedding(EMB_SEED, device=dev)
        am = torch.empty(M, dtype=torch.int32, device=dev)
        run = lambda i: fgm.lm_head_argmax(emb, xs[i % N_BATCHES], argmax=am, ws=ws)
        unit_bytes = [traffic.lm_head_bytes()] * max(K, W)
        name = "lm_head argmax, 262144 x 2816 bf16, M=5"
    for i in range(W):
        run(i)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    ev[0].record(stream)
    for i in range(K):
        run(i)
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(K)]
    gbs = sum(unit_bytes[:K]) / (sum(times) * 1e-3) / 1e9
    peak, kind = measured_peaks()
    return {"case": args.case, "workload": name, "path": args.path, "steps": K, "warmup": W,
            "ms_per_call": round(statistics.mean(times), 4), "hbm_gbs": round(gbs, 1),
            "frac_of_peak": round(gbs / peak, 4), "peak": peak, "peak_kind": kind,
            "status": ws.status()}


def run_sweep(args):
    """The full verify step swept over M = 1..8 (gamma 0..7) and the router bias
    Zipf s in {0, 1.1, 2.0}: the 30-layer stack and lm_head of the headline
    workload, the bias swapped per s. Prints one JSON line per point (tokens/s
    counting accepted drafts + 1 per step, and algorithmic HBM GB/s); returns None."""
    import torch

    import fine_grained_moe_gb300 as fgm
    import synth
    from fine_grained_moe_gb300 import traffic

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fgm.lib()
    fgm.select_path(getattr(fgm, PATHS[args.path]))
    layers, emb, _ = make_workload(dev)
    ws = fgm.Workspace(dev)
    peak, _ = measured_peaks()
    K, W = args.steps, args.warmup
    for s_zipf in (0.0, 1.1, 2.0):
        bias = None if s_zipf == 0.0 else synth.zipf_bias(s_zipf).to(dev)
        for p in layers:
            p["router_b"] = bias
        arr = fgm.layers_array(layers)
        for m in range(1, 9):
            xs = [synth.hidden_states(HIDDEN_SEED0 + b, m, device=dev) for b in range(N_BATCHES)]
            trace = torch.empty((N_LAYERS, m, 8), dtype=torch.int32, device=dev)
            drafts, nbytes = [], []
            for b, x in enumerate(xs):
                fgm.moe_stack_fwd(layers, x, ids_trace=trace, ws=ws)
                tr = trace.cpu()
                nbytes.append(traffic.step_bytes([len(torch.unique(tr[l])) for l in range(N_LAYERS)]))
                am = torch.empty(m, dtype=torch.int32, device=dev)
                fgm.verify_step(layers, emb, x, torch.zeros(max(m - 1, 1), dtype=torch.int32, device=dev),
                                argmax=am, ws=ws, _arr=arr)
                drafts.append(synth.drafts(DRAFT_SEED0 + b, am.cpu()).to(dev) if m > 1 else None)
            outs = torch.zeros((K, 2), dtype=torch.int32, device=dev)
            for i in range(W):
                fgm.verify_step(layers, emb, xs[i % N_BATCHES], drafts[i % N_BATCHES], ws=ws, _arr=arr)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for i in range(K):
                b = i % N_BATCHES
                fgm.verify_step(layers, emb, xs[b], drafts[b], out=outs[i], ws=ws, _arr=arr)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            tokens = int(outs[:, 0].sum()) + K
            gbs = sum(nbytes[i % N_BATCHES] for i in range(K)) / (ms * 1e-3) / 1e9
            print(json.dumps({"case": "sweep", "M": m, "gamma": m - 1, "zipf_s": s_zipf,
                              "tokens_per_s": round(tokens / (ms * 1e-3), 1),
                              "tokens_per_s_at_expected_accept": round(K * (1 + expected_accept(m - 1))
                                                                       / (ms * 1e-3), 1),
                              "ms_per_step": round(ms / K, 4), "accepted_per_step": round((tokens - K) / K, 3),
                              "hbm_gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                              "status": ws.status()}), flush=True)
    return None


def run_verify_dense(args):
    """The verify step of the model variant whose every layer carries a 2816 x
    2112 dense MLP in place of the 704-wide shared expert: same 30 routed
    stacks, inputs and draft recipe (drafts copy this step's own argmax with
    probability 0.7), MLP seeds 40..69. Returns one JSON line (tokens/s
    counting accepted drafts + 1 per step, algorithmic HBM GB/s)."""
    import torch

    import fine_grained_moe_gb300 as fgm
    import synth
    from fine_grained_moe_gb300 import traffic

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fgm.lib()
    fgm.select_path(getattr(fgm, PATHS[args.path]))
    layers, emb, xs = make_workload(dev)
    mlps = [synth.dense_mlp(40 + l, device=dev) for l in range(N_LAYERS)]
    arr, mlp_arr = fgm.layers_array(layers), fgm.mlps_array(mlps)
    ws = fgm.Workspace(dev)
    uniq, drafts = [], []
    trace = torch.empty((N_LAYERS, M, 8), dtype=torch.int32, device=dev)
    for b, x in enumerate(xs):
        fgm.moe_stack_dense_fwd(layers, mlps, x, ids_trace=trace, ws=ws)
        tr = trace.cpu()
        uniq.append([len(torch.unique(tr[l])) for l in range(N_LAYERS)])
        am = torch.empty(M, dtype=torch.int32, device=dev)
        fgm.verify_step_dense(layers, mlps, emb, x, torch.zeros(GAMMA, dtype=torch.int32, device=dev), argmax=am,
                              ws=ws, _arr=arr, _mlp_arr=mlp_arr)
        drafts.append(synth.drafts(DRAFT_SEED0 + b, am.cpu()).to(dev))
    nbytes = [traffic.step_bytes(u, dense_width=3 * 704) for u in uniq]
    K, W = args.steps, args.warmup
    outs = torch.zeros((K, 2), dtype=torch.int32, device=dev)
    for i in range(W):
        b = i % N_BATCHES
        fgm.verify_step_dense(layers, mlps, emb, xs[b], drafts[b], ws=ws, _arr=arr, _mlp_arr=mlp_arr)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        e0.record()
        for i in range(K):
            b = i % N_BATCHES
            fgm.verify_step_dense(layers, mlps, emb, xs[b], drafts[b], out=outs[i], ws=ws, _arr=arr,
                                  _mlp_arr=mlp_arr)
        e1.record()
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    tokens = int(outs[:, 0].sum().cpu()) + K
    gbs = sum(nbytes[i % N_BATCHES] for i in range(K)) / (ms * 1e-3) / 1e9
    peak, kind = measured_peaks()
    clocks = clk.summary()
    return {"case": "verify_dense", "path": args.path,
            "workload": "full verify step, M=5 (gamma=4), Zipf s=1.1, 30 layers each with a 2816x2112 dense "
                        "MLP in place of the shared expert, 262144x2816 bf16 lm_head",
            "steps": K, "warmup": W, "tokens_per_s": round(tokens / (ms * 1e-3), 2),
            "tokens_per_s_at_expected_accept": round(K * (1 + expected_accept(GAMMA)) / (ms * 1e-3), 2),
            "ms_per_step": round(ms / K, 4), "accepted_per_step": round((tokens - K) / K, 3),
            "algorithmic_bytes_per_step": int(statistics.mean(nbytes)),
            "hbm_gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4), "peak": peak, "peak_kind": kind,
            "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                       "reasons": clocks["reasons"]},
            "status": ws.status()}


def run_verify_fp8(args):
    """The headline verify step with the FP8 lm_head in place of the bf16 one:
    same 30-layer stack, inputs and draft recipe (drafts copy the FP8 head's
    own argmax with probability 0.7). Returns one JSON line (tokens/s counting
    accepted drafts + 1 per step, algorithmic HBM GB/s)."""
    import torch

    import fine_grained_moe_gb300 as fgm
    import synth
    from fine_grained_moe_gb300 import traffic

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fgm.lib()
    fgm.select_path(getattr(fgm, PATHS[args.path]))
    layers, emb, xs = make_workload(dev)
    emb_q, emb_s = synth.embedding_fp8(emb)
    del emb
    torch.cuda.empty_cache()
    arr = fgm.layers_array(layers)
    ws = fgm.Workspace(dev)
    uniq, drafts = [], []
    trace = torch.empty((N_LAYERS, M, 8), dtype=torch.int32, device=dev)
    for b, x in enumerate(xs):
        fgm.moe_stack_fwd(layers, x, ids_trace=trace, ws=ws)
        tr = trace.cpu()
        uniq.append([len(torch.unique(tr[l])) for l in range(N_LAYERS)])
        am = torch.empty(M, dtype=torch.int32, device=dev)
        fgm.verify_step_fp8_head(layers, emb_q, emb_s, x, torch.zeros(GAMMA, dtype=torch.int32, device=dev),
                                 argmax=am, ws=ws, _arr=arr)
        drafts.append(synth.drafts(DRAFT_SEED0 + b, am.cpu()).to(dev))
    nbytes = [traffic.step_bytes(u, fp8_lm_head=True) for u in uniq]
    K, W = args.steps, args.warmup
    outs = torch.zeros((K, 2), dtype=torch.int32, device=dev)
    for i in range(W):
        b = i % N_BATCHES
        fgm.verify_step_fp8_head(layers, emb_q, emb_s, xs[b], drafts[b], ws=ws, _arr=arr)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        e0.record()
        for i in range(K):
            b = i % N_BATCHES
            fgm.verify_step_fp8_head(layers, emb_q, emb_s, xs[b], drafts[b], out=outs[i], ws=ws, _arr=arr)
        e1.record()
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    tokens = int(outs[:, 0].sum().cpu()) + K
    gbs = sum(nbytes[i % N_BATCHES] for i in range(K)) / (ms * 1e-3) / 1e9
    peak, kind = measured_peaks()
    clocks = clk.summary()
    return {"case": "verify_fp8", "path": args.path,
            "workload": "full verify step, M=5 (gamma=4), Zipf s=1.1, 30 layers, "
                        "262144x2816 E4M3 lm_head with fp32 row scales",
            "steps": K, "warmup": W, "tokens_per_s": round(tokens / (ms * 1e-3), 2),
            "tokens_per_s_at_expected_accept": round(K * (1 + expected_accept(GAMMA)) / (ms * 1e-3), 2),
            "ms_per_step": round(ms / K, 4), "accepted_per_step": round((tokens - K) / K, 3),
            "algorithmic_bytes_per_step": int(statistics.mean(nbytes)),
            "hbm_gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4), "peak": peak, "peak_kind": kind,
            "launches_per_step": 2 if args.path != "staged" else 1 + N_LAYERS * 5 + 1,
            "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                       "reasons": clocks["reasons"]},
            "status": ws.status()}


# ---------------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    """The oracle as the reference arm: one full step on batch 0 fixes the
    accepted count, then each timed step runs a bounded sample of the step
    (the first n layers plus the same fraction of the lm_head rows), scaled
    to a full step."""
    if rank != 0:
        return None
    import numpy as np
    import torch

    import oracle
    import synth

    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    layers, emb, xs = make_workload(dev)
    full_s, a, _, cores = cpu_oracle_step(layers, emb, xs[0], DRAFT_SEED0, "[reference]")
    budget = 150.0
    n_steps = args.steps + args.warmup
    frac = min(1.0, budget / max(1e-9, n_steps * full_s))
    n_layers = max(1, int(round(N_LAYERS * frac)))
    frac = n_layers / N_LAYERS
    v_rows = max(1, int(262144 * frac))
    host = []
    for p in layers[:n_layers]:
        h = {k: (None if v is None else v.detach().cpu()) for k, v in p.items()}
        host.append(oracle.LayerParams(
            router_w=h["router_w"].view(torch.int16).numpy().view(np.uint16),
            router_b=None if h["router_b"] is None else h["router_b"].numpy(),
            gate_q=h["gate_q"].numpy(), gate_s=h["gate_s"].numpy(), up_q=h["up_q"].numpy(),
            up_s=h["up_s"].numpy(), down_q=h["down_q"].numpy(), down_s=h["down_s"].numpy()))
    e = emb[:v_rows].detach().cpu().view(torch.int16).numpy().view(np.uint16)
    x0 = xs[0].detach().cpu().double().numpy()

    def sample():
        t0 = time.perf_counter()
        h = x0
        for L in host:
            h = oracle.stack_layer(L, h).y
        oracle.lm_head(e, oracle.bf16_to_f64(oracle.bf16_round(oracle.rmsnorm(h))))
        return (time.perf_counter() - t0) / frac

    for _ in range(args.warmup):
        sample()
    times = [sample() for _ in range(args.steps)]
    ms = 1e3 * statistics.mean(times)
    value = (1 + expected_accept(GAMMA)) / (ms * 1e-3)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded workload as the CUDA arm)",
        "config": {"workload": WORKLOAD, "M": M, "gamma": GAMMA, "zipf_s": S_ZIPF, "layers": N_LAYERS,
                   "vocab": 262144, "parallelism": "single process, OpenMP"},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(),
                         "sample": f"per step: first {n_layers} of 30 layers + {v_rows} of 262144 lm_head rows "
                                   f"on batch 0, scaled x{1 / frac:.2f}; 1 + E[a] tokens per step as in the "
                                   f"CUDA arm (accepted count of the full step on batch 0: {a})"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", choices=tuple(PATHS), default="fused",
                    help="persistent kernel (default), one launch per stage, the persistent kernel with the "
                         "tcgen05 FP8 lm_head, or the persistent kernel with mma.sync down products")
    ap.add_argument("--layers", type=int, default=N_LAYERS,
                    help="verify case only: stack depth (a smaller case for ncu captures; default 30)")
    ap.add_argument("--vocab", type=int, default=262144,
                    help="verify case only: lm_head rows (a smaller case for ncu captures; default 262144)")
    ap.add_argument("--phase-trace", metavar="PATH", default=None,
                    help="after timing, run one traced step and write a per-phase summary to PATH")
    ap.add_argument("--case", choices=("verify", "layer", "layer_dense", "lm_head", "lm_head_fp8", "verify_fp8",
                                       "verify_dense", "sweep"),
                    default="verify",
                    help="verify: the headline step; layer / layer_dense / lm_head / lm_head_fp8: one stage alone "
                         "(profiling); verify_fp8: the step with the FP8 lm_head; verify_dense: the step with a "
                         "2112-wide dense MLP per layer; sweep: the verify step "
                         "over M = 1..8 and Zipf s in {0, 1.1, 2} (one line each)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    try:
        if args.impl == "reference":
            line = run_reference(args, rank, world)
        elif args.case == "sweep":
            line = run_sweep(args)
        elif args.case == "verify_fp8":
            line = run_verify_fp8(args)
        elif args.case == "verify_dense":
            line = run_verify_dense(args)
        elif args.case != "verify":
            line = run_case(args)
        else:
            line = run_ours(args, rank, world)
    finally:
        if world > 1 and args.impl == "ours":
            import torch
            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
