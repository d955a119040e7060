#!/usr/bin/env python
"""Throughput of the GB300 MoE-LoRA layer (tokens/s per layer) and its roofline fraction.

One step = one pass of the whole hot path over one batch of seeded synthetic input:
route -> align -> forward (gather, gate_up shrink, gate_up GEMM + expand + SiLU,
down shrink, down GEMM + expand, weighted top-k combine).  Default workload:
the decode-sized layer (T=16 tokens, H=I=2880, E=32 top-4, 8 adapters of rank 32).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

N > 1 runs N independent replicas (one process per GPU via torch.distributed.run),
each on its own batch; value = tokens of all ranks / max-over-ranks time.
--impl reference times the fp64 CPU oracle on the host cores on a bounded sample of
the same workload.
"""
from __future__ import annotations

import argparse
import gc
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from expert_gemm_gb300 import workloads as W  # noqa: E402

METRIC = "MoE-LoRA layer tokens/s"
L2_FLUSH_BYTES = 256 << 20


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)) or None, "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# --------------------------------------------------------------- accounting --

def algorithmic(wl: W.Workload, ids: np.ndarray, lora: np.ndarray):
    """Algorithmic bytes and flops of one layer pass and of its gate_up launch.

    Bytes: weights of the distinct touched experts and distinct touched (adapter>=0,
    expert) pairs, x in and out once; padding rows, S tiles, h and zero rank padding
    are not counted.  Flops: 2 * valid pairs * (H*2I + I*H) + LoRA 2 * r * (H + 2I + I + H)
    per pair with an adapter.
    """
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    ranks = np.asarray(wl.ranks)
    valid = (ids >= 0) & (ids < E)
    experts = np.unique(ids[valid])
    a_tok = np.repeat(lora, k).reshape(T, k)
    with_a = valid & (a_tok >= 0)
    ae = np.unique(a_tok[with_a].astype(np.int64) * E + ids[with_a])
    r_ae = ranks[ae // E] if len(ae) else np.zeros(0)
    w_gu = len(experts) * 2 * I * H * 2
    w_dn = len(experts) * H * I * 2
    lora_gu = int(np.sum(r_ae * (H + 2 * I))) * 2
    lora_dn = int(np.sum(r_ae * (I + H))) * 2
    act = 2 * T * H * 2
    n_pairs = int(valid.sum())
    r_pairs = ranks[a_tok[with_a]] if with_a.any() else np.zeros(0)
    flops = 2 * n_pairs * (H * 2 * I + I * H) + 2 * int(np.sum(r_pairs)) * (H + 2 * I + I + H)
    gate_up_bytes = w_gu + int(np.sum(r_ae * 2 * I)) * 2 + T * H * 2 + n_pairs * I * 2
    return {"bytes": w_gu + w_dn + lora_gu + lora_dn + act, "flops": flops, "gate_up_bytes": gate_up_bytes,
            "gate_up_flops": 2 * n_pairs * H * 2 * I + 2 * int(np.sum(r_pairs)) * 2 * I,
            "experts": int(len(experts)), "adapter_expert_pairs": int(len(ae)), "valid_pairs": n_pairs}


# ------------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu, self.proc = gpu, None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "200"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            return None
        rows = [[c.strip() for c in line.split(",")] for line in out.strip().splitlines() if line.strip()]
        rows = [r for r in rows if len(r) >= 9]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def workload_of(args) -> W.Workload:
    wl = W.get(args.workload)
    if getattr(args, "tokens", 0):
        import dataclasses
        wl = dataclasses.replace(wl, name=f"{wl.name}_T{args.tokens}", T=args.tokens,
                                 requests=min(wl.requests, args.tokens) if wl.requests else 0)
    return wl


def workload_config(wl: W.Workload, world: int) -> dict:
    """The config keys both arms report for a workload."""
    return {"workload": f"{wl.name}: T={wl.T} H={wl.H} I={wl.I} E={wl.E} top-{wl.k} L={wl.L} "
                        f"ranks={sorted(set(wl.ranks))}", "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E,
            "k": wl.k, "L": wl.L, "global_batch": world * wl.T,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


# -------------------------------------------------------------- our arm -----

KERNEL_SOURCES = ("gemm_tc.cuh", "ptx.cuh", "common.cuh", "gemm_tc.cu", "moe_lora.cu")   # kernels and their tensor maps


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "expert_gemm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from a committed ncu capture, if it was taken of the current kernel source."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            doc = json.load(f)
    except Exception:
        return None
    e = doc.get(workload, {}).get(kernel)
    if not e or e.get("kernel_source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


def max_over_ranks(value: float, world: int) -> float:
    """The largest value over all ranks (every rank gets it); the value itself when alone."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's step time."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


def _dev(torch, a):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def measure(torch, ml, wl, wd, seed_b, K, Wm, bm, world, flush, graph=False, e2e=True, clocks=None):
    """Times K steps of one workload on resident inputs; returns a dict of measurements."""
    logits, lora = W.make_routing(wl, seed_b)
    x = W.make_activations(wl, seed_b)
    d = ml.LayerDims(T=wl.T, H=wl.H, I=wl.I, E=wl.E, k=wl.k, L=wl.L, r_max=wl.r_max, block_m=bm, ranks=wl.ranks)
    layer = ml.Layer(d, wd)
    lg, lr, xd = _dev(torch, logits), _dev(torch, lora), _dev(torch, x)
    KI = max(1, min(K, 100))                      # instrumented steps (per-stage events)
    nst = ml.NUM_STAGES + 1
    stage_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nst)] for _ in range(KI)]
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for evs in stage_ev:                          # create the CUDA events before handing them to the library
        for e in evs:
            e.record()
    for _ in range(Wm):
        layer.step(lg, lr, xd)
        flush.zero_()
    torch.cuda.synchronize()
    if int(layer.status.item()) != 0:
        raise RuntimeError(f"device status {int(layer.status.item())}")
    ids = layer.topk_ids.cpu().numpy()
    tot = layer.bufs["totals"].cpu().numpy()
    plan = ml.plan(d)
    launches_per_step = plan["launches_route_align"] + plan["launches_forward"]
    acct = algorithmic(wl, ids, lora)

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.start()
    t_wall0 = time.perf_counter()
    # headline: K plain steps (events only at step boundaries)
    for i in range(K):
        step_ev[i][0].record()
        layer.step(lg, lr, xd)
        step_ev[i][1].record()
        flush.zero_()
    # per-kernel durations: steps with an event between every two launches
    for i in range(KI):
        layer.step(lg, lr, xd, stage_events=stage_ev[i])
        flush.zero_()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop() if clocks is not None else None
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    stage_ms = np.array([[evs[j].elapsed_time(evs[j + 1]) for j in range(nst - 1)] for evs in stage_ev])
    ms = max_over_ranks(float(np.sum(step_ms)) / K, world)
    if int(layer.status.item()) != 0:
        raise RuntimeError(f"device status {int(layer.status.item())}")
    out = {"wl": wl, "bm": bm, "ms": ms, "K": K, "KI": KI, "stage_ms": stage_ms, "acct": acct, "clocks": clk,
           "t_wall": t_wall, "totals": [int(v) for v in tot], "launches": launches_per_step * (K + KI),
           "plan": plan}

    if graph:
        try:
            out["graph_ms"] = _graph_ms(torch, layer, lg, lr, xd, flush, K)
        except Exception as exc:   # report, keep the rest of the measurement
            out["graph_error"] = f"{type(exc).__name__}: {exc}"[:300]
    if e2e:
        # end to end through the host-buffer entry point (pinned host memory)
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
        lg_h, lr_h, x_h = pin(logits), pin(lora), pin(x.view(np.int16))
        out_h = torch.empty((wl.T, wl.H), dtype=torch.int16).pin_memory()
        for _ in range(max(2, min(Wm, 10))):
            layer.step_host(lg_h, lr_h, x_h, out_h)
        ke = max(1, min(K, 500))
        if world > 1:
            torch.distributed.barrier()
        # each call ends in a stream synchronise, so per-call wall times are whole steps;
        # the median keeps a host-side hiccup from standing for the step
        def timed(fn):
            per = []
            for _ in range(ke):
                t0 = time.perf_counter()
                fn()
                per.append(time.perf_counter() - t0)
            return float(np.median(per)), float(np.mean(per))
        # (1) the captured layer (moe_lora_layer_graph_run): copies in, kernels, copies out
        gstream = torch.cuda.Stream()
        graph = layer.graph_host(lg_h, lr_h, x_h, out_h, gstream)
        try:
            for _ in range(max(2, min(Wm, 10))):
                graph.run()
            if world > 1:
                torch.distributed.barrier()
            med, mean = timed(graph.run)
        finally:
            graph.close()
        out["e2e_s"] = max_over_ranks(med, world)
        out["e2e_mean_s"] = mean
        # (2) the same through moe_lora_layer_host (each call enqueues every copy and launch)
        med, mean = timed(lambda: layer.step_host(lg_h, lr_h, x_h, out_h))
        out["e2e_direct_s"] = max_over_ranks(med, world)
    del layer
    return out


def _graph_ms(torch, layer, lg, lr, xd, flush, K):
    """The same step captured once into a CUDA graph and replayed (launch overhead off the host)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.step(lg, lr, xd, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.step(lg, lr, xd)
    for _ in range(3):
        g.replay()
        flush.zero_()
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        gev[i][0].record()
        g.replay()
        gev[i][1].record()
        flush.zero_()
    torch.cuda.synchronize()
    if int(layer.status.item()) != 0:
        raise RuntimeError(f"device status {int(layer.status.item())} after graph replay")
    return float(np.mean([a.elapsed_time(b) for a, b in gev]))


def roofline_of(m, ml):
    """Dominant-kernel roofline (gate_up) and the whole-layer roofline of one measurement.

    Tensor-bound fractions are of the sustained bf16 rate (cuBLAS back to back for
    seconds, under the power cap): every leg times its kernels inside a fraction of a
    second or more of back-to-back steps, and the compute-bound legs run at the power
    cap.  The fraction of the burst rate is reported beside it (`frac_of_burst`)."""
    hbm, tc_burst, tc_sus, src = peaks()
    tc = tc_sus or tc_burst
    tc_name = "cuBLAS bf16 sustained" if tc_sus else "cuBLAS bf16 burst"
    acct, wl = m["acct"], m["wl"]
    gu_ms = float(np.mean(m["stage_ms"][:, ml.STAGES.index("gate_up")]))
    intensity = acct["gate_up_flops"] / max(acct["gate_up_bytes"], 1)
    ridge = tc * 1e12 / (hbm * 1e9)
    kname = "gate_up (tcgen05 grouped GEMM + LoRA expand + SiLU)"
    if intensity < ridge:
        ach = acct["gate_up_bytes"] / (gu_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": kname, "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "peak_source": f"{src} (HBM copy)", "algorithmic_bytes_per_launch": acct["gate_up_bytes"]}
    else:
        ach = acct["gate_up_flops"] / (gu_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": kname, "achieved": ach, "peak": tc, "unit": "TFLOP/s",
                "frac": ach / tc, "peak_source": f"{src} ({tc_name})", "frac_of_burst": ach / tc_burst,
                "algorithmic_flops_per_launch": acct["gate_up_flops"]}
    roof["launch_ms"] = gu_ms
    roof["traffic"] = committed_traffic(wl.name, "gate_up")
    layer_s = m["ms"] * 1e-3
    t_bw, t_tc = acct["bytes"] / (hbm * 1e9), acct["flops"] / (tc * 1e12)
    layer = {"alg_bytes": acct["bytes"], "alg_flops": acct["flops"], "t_roof_ms": max(t_bw, t_tc) * 1e3,
             "bound": "hbm" if t_bw >= t_tc else "tensor", "frac": max(t_bw, t_tc) / layer_s,
             "hbm_gbs_peak": hbm, "bf16_tflops_peak": tc, "bf16_tflops_peak_source": tc_name}
    if t_tc > t_bw:
        layer["frac_of_burst"] = acct["flops"] / (tc_burst * 1e12) / layer_s
    return roof, layer


# The other configurations the layer is measured on, timed after the headline (decode)
# in the default run; each gets its own clock record and CPU baseline.
# The sweep legs run last: right after their 7.9 GB of adapter banks were freed, the
# dense_decode leg's plain steps measured 0.33-0.38 ms against 0.188 ms on its own or
# earlier in the run, with unchanged per-kernel times (the host's launch loop fell
# behind the GPU), in two runs.
SECONDARY = ("prefill", "dense_decode", "wide", "sweep_T1", "sweep_T16", "sweep_T256", "sweep_T4096")


def _weights_key(wl: W.Workload):
    return (wl.H, wl.I, wl.E, wl.L, tuple(wl.ranks))


def _upload(torch, w):
    return {n: _dev(torch, w[n]) for n in ("W_gu", "W_dn", "A_gu", "B_gu", "A_dn", "B_dn")}


def clock_summary(clk, ms):
    """The leg's sampled clocks plus its step time in SM cycles (ms x median MHz)."""
    if not clk:
        return clk
    out = dict(clk)
    if clk.get("sm_mhz"):
        out["kcycles_per_step"] = ms * clk["sm_mhz"]   # ms * MHz = thousands of cycles
    return out


def secondary_steps(ms_est: float, k_arg: int) -> int:
    """Steps of a secondary leg: about 0.6 s of timed work with the L2 flushes between
    steps (~0.07 ms each), so that the 200 ms clock sampler sees the leg; at least 10
    and at least the headline's steps, at most 5000."""
    k = int(0.6e3 / (max(ms_est, 1e-3) + 0.07))
    return max(10, min(k_arg, 5000), min(k, 5000))


def secondary_warmup(ms_est: float) -> int:
    """Untimed steps before a secondary leg: about 0.1 s of them (at least 3, at most 1000),
    so that the host's launch loop runs ahead of the GPU when the timed steps start.  The
    legs of a few tens of microseconds are host-launch sensitive: with 3 warm-up steps
    right after the sweep layer's 7.9 GB of adapter banks were drawn and uploaded, the
    one-token leg once measured 59.4 us a step with unchanged per-kernel times (52.7 us in
    other runs)."""
    return max(3, min(1000, int(0.1e3 / (max(ms_est, 1e-3) + 0.07))))


def run_secondary(torch, ml, name, wd, w_host, rank, world, flush, args):
    """One secondary configuration: device timing, roofline, clocks, oracle baseline."""
    wl = W.get(name)
    bm = ml.pick_block_m(wl.T, wl.k, wl.E, wl.L, wl.H, wl.I)
    probe = measure(torch, ml, wl, wd, rank, 3, 3, bm, world, flush, graph=False, e2e=False)
    k = secondary_steps(probe["ms"], args.steps)
    wu = secondary_warmup(probe["ms"])
    m = measure(torch, ml, wl, wd, rank, k, wu, bm, world, flush, graph=False, e2e=False,
                clocks=ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))))
    roof, layer = roofline_of(m, ml)
    res = {"workload": workload_config(wl, world)["workload"], "T": wl.T,
           "value": job_throughput(wl.T, world, m["ms"]), "unit": "tokens/s", "ms_per_step": m["ms"],
           "steps": k, "warmup": wu, "block_m": bm, "roofline": roof, "layer_roofline": layer,
           "stage_ms": {n: float(np.mean(m["stage_ms"][:, j])) for j, n in enumerate(ml.STAGES)},
           "touched": {k_: m["acct"][k_] for k_ in ("experts", "adapter_expert_pairs", "valid_pairs")},
           "clocks": clock_summary(m["clocks"], m["ms"]), "gpu_launches": probe["launches"] + m["launches"],
           "plan": m["plan"]}
    if world == 1 and args.secondary_cpu_s > 0:
        res["cpu_baseline"] = cpu_baseline(wl, args.secondary_cpu_s, w_host)
    return res


def run_ours(args, rank, world, local_rank):
    import torch
    from expert_gemm_gb300 import build, moe_lora as ml
    torch.cuda.set_device(local_rank)
    build.build()
    ml.load()
    wl = workload_of(args)
    w_host = W.make_weights(wl, 0)                # same weights on every replica, own batch per rank
    wd = _upload(torch, w_host)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    bm = args.block_m or ml.pick_block_m(wl.T, wl.k, wl.E, wl.L, wl.H, wl.I)
    m = measure(torch, ml, wl, wd, rank, args.steps, args.warmup, bm, world, flush,
                graph=not args.no_graph, clocks=ClockSampler(local_rank))
    roof, layer = roofline_of(m, ml)
    stage_ms = m["stage_ms"]
    res = {
        "metric": METRIC, "value": job_throughput(wl.T, world, m["ms"]), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": m["ms"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded normals, bf16)",
        "config": {**workload_config(wl, world), "block_m": bm,
                   "l2": "flushed between timed steps (256 MiB write)"},
        "roofline": roof,
        "layer_roofline": layer,
        "stage_ms": {n: float(np.mean(stage_ms[:, j])) for j, n in enumerate(ml.STAGES)},
        "instrumented_ms_per_step": float(np.mean(np.sum(stage_ms, axis=1))),
        "instrumented_steps": m["KI"],
        "touched": {k_: m["acct"][k_] for k_ in ("experts", "adapter_expert_pairs", "valid_pairs")},
        "e2e": {"value": job_throughput(wl.T, world, m["e2e_s"] * 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": wl.T * (wl.E * 4 + 4 + wl.H * 2),
                "d2h_bytes_per_step": wl.T * wl.H * 2 + 32, "ms_per_step": m["e2e_s"] * 1e3,
                "stat": "median of per-step wall times", "mean_ms_per_step": m["e2e_mean_s"] * 1e3,
                "entry": "moe_lora_layer_graph_run (pinned host buffers of at most 4 MB, x while its "
                         "gather reads stay within 1 MB, read and written in place by the kernels over the "
                         "CPU-GPU link, the rest copied; the status record copied back; all in the graph)",
                "direct": {"entry": "moe_lora_layer_host", "ms_per_step": m["e2e_direct_s"] * 1e3,
                           "value": job_throughput(wl.T, world, m["e2e_direct_s"] * 1e3)}},
        "gpu_launches": m["launches"],
        "clocks": clock_summary(m["clocks"], m["ms"]),
        "wall_s_timed": m["t_wall"],
        "align_totals": m["totals"],
        "plan": m["plan"],
    }
    if "graph_ms" in m:
        res["cuda_graph"] = {"ms_per_step": m["graph_ms"], "value": world * wl.T / (m["graph_ms"] * 1e-3),
                             "unit": "tokens/s", "note": "the same step captured once and replayed"}
    elif "graph_error" in m:
        res["cuda_graph"] = {"error": m["graph_error"]}
    if world == 1 and args.cpu_baseline_s > 0:
        res["cpu_baseline"] = cpu_baseline(wl, args.cpu_baseline_s, w_host)
    # the other configurations, each a full pass of the same hot path at its own shapes
    if args.secondary and wl.name == "decode":
        res["secondary"] = {}
        cur_key = _weights_key(wl)
        for name in SECONDARY:
            sw = W.get(name)
            if _weights_key(sw) != cur_key:
                del wd
                wd = None
                torch.cuda.empty_cache()
                w_host = None
                gc.collect()
                w_host = W.make_weights(sw, 0)
                wd = _upload(torch, w_host)
                cur_key = _weights_key(sw)
                time.sleep(1.0)   # let the host settle after gigabytes of fresh pages
            r = run_secondary(torch, ml, name, wd, w_host, rank, world, flush, args)
            res["secondary"][name] = r
            res["gpu_launches"] += r["gpu_launches"]
        res["prefill"] = res["secondary"]["prefill"]   # the compute-bound headline beside decode
    return res


# --------------------------------------------------------- oracle timings ---

def oracle_sample_rate(wl: W.Workload, n_tokens: int, budget_s: float, seed: int = 0, threads: int = 0, w=None):
    """Oracle (route + align + fp64 forward) on the first n_tokens tokens, repeated for ~budget_s.

    threads > 0 caps the oracle's OpenMP threads for this sample (0: one per processor);
    w: the workload's host weights (drawn here when None)."""
    from oracle import Oracle
    o = Oracle()
    o.set_threads(threads)
    logits, lora = W.make_routing(wl, seed)
    x = W.make_activations(wl, seed)
    if w is None:
        w = W.make_weights(wl, seed)
    n = max(1, min(n_tokens, wl.T))
    lg, lr, xs = logits[:n], lora[:n], x[:n]
    bm = 16
    reps, t0 = 0, time.perf_counter()
    while True:
        ids, tw = o.route(lg, wl.k)
        o.align(ids, lr, wl.E, wl.L, bm)
        o.forward(xs, ids, tw.astype(np.float32), lr, w)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    o.set_threads(0)
    return n * reps / el, n, reps, el


def cores_used():
    try:
        n = len(os.sched_getaffinity(0))
    except Exception:
        n = os.cpu_count() or 1
    return int(os.environ.get("OMP_NUM_THREADS", n))


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
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
    except Exception:
        pass
    return None


def cpu_baseline(wl, budget_s, w=None):
    """The oracle on all host cores and on one, over the same bounded token sample.

    The oracle's forward is parallel over tokens, so the threads it uses are at most the
    sample's token count."""
    n = min(wl.T, 16)
    v, n, reps, el = oracle_sample_rate(wl, n, budget_s, w=w)
    v1, _, reps1, el1 = oracle_sample_rate(wl, n, budget_s / 3, threads=1, w=w)
    return {"value": v, "unit": "tokens/s", "cores": min(cores_used(), n), "kind": "oracle",
            "sample": f"first {n} of {wl.T} tokens, {reps} passes in {el:.1f} s (route + align + fp64 forward)",
            "one_core": {"value": v1, "unit": "tokens/s", "cores": 1,
                         "sample": f"the same {n} tokens, {reps1} passes in {el1:.1f} s"},
            "host_cores": cores_used(), "cpu_model": cpu_model()}


def run_reference(args):
    """The fp64 oracle as the reference arm: each step is a bounded token sample of the workload."""
    from oracle import Oracle
    wl = workload_of(args)
    o = Oracle()
    logits, lora = W.make_routing(wl, 0)
    x = W.make_activations(wl, 0)
    w = W.make_weights(wl, 0)
    # calibrate: cost of one token, then size the per-step sample to ~150 s in total
    def one_step(n):
        ids, tw = o.route(logits[:n], wl.k)
        o.align(ids, lora[:n], wl.E, wl.L, 16)
        o.forward(x[:n], ids, tw.astype(np.float32), lora[:n], w)
    n_cal = min(wl.T, 8)
    t0 = time.perf_counter()
    one_step(n_cal)
    per_tok = (time.perf_counter() - t0) / n_cal
    budget = 150.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(wl.T, budget / max(per_tok, 1e-9))))
    for _ in range(args.warmup):
        one_step(n)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step(n)
    el = time.perf_counter() - t0
    v = n * args.steps / el
    return {"metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded normals, bf16)",
            "impl": "reference",
            "config": workload_config(wl, args.gpus),
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": min(cores_used(), n), "kind": "oracle",
                             "sample": f"first {n} of {wl.T} tokens per step (route + align + fp64 forward)",
                             "host_cores": cores_used(), "cpu_model": cpu_model()},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode", choices=sorted(W.WORKLOADS))
    ap.add_argument("--block-m", type=int, default=0)
    ap.add_argument("--tokens", type=int, default=0, help="override T of the workload (small profiling cases)")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timing")
    ap.add_argument("--no-secondary", dest="secondary", action="store_false",
                    help="skip the other configurations that accompany the decode workload")
    ap.add_argument("--cpu-baseline-s", type=float, default=12.0, help="seconds of oracle time (0 = skip)")
    ap.add_argument("--secondary-cpu-s", type=float, default=2.0,
                    help="seconds of oracle time per secondary configuration (0 = skip)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
