"""Benchmark: ms per 10-step action decision on one GB300 (18 layers x 10 Euler
steps, M = 50 action rows, prefix KV 788 tokens, FP8 weights and activations),
with the achieved HBM bandwidth of the decision and of the dominant kernel.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). A "step" is one whole decision (all layers, all
Euler steps) on synthetic seeded inputs; the weights streamed per decision
(2.7 GB) are far larger than L2 (129 MB), so no L2 flush is needed between steps.
N > 1 (torchrun) runs one independent policy replica per GPU: the path does not
shard, there is no collective on the data path.

--impl reference times the CPU oracle (the plain FP64 restatement of the same
method) on this host's cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import fm_synth  # noqa: E402

WORKLOAD = "expert_fp8_m50"
METRIC = "ms per 10-step action decision at 1 GB300; achieved HBM GB/s vs 8 TB/s roofline"
UNIT = "ms/decision"


def algorithmic_bytes(cfg) -> dict:
    """Bytes a decision must move at least once: packed weights every layer-step,
    the prefix K/V every layer-step, the modulation table once per step and layer,
    the in/out projections once per step (activations are < 0.1% and excluded)."""
    wb = {"fp8": 1.0, "bf16": 2.0, "nvfp4": 0.5625}[cfg.weight_fmt]
    w_layer = sum(n * k for n, k in cfg.gemm_shapes) * wb
    kv_layer = 2 * cfg.P * cfg.Hkv * cfg.Dh * 2
    mod = cfg.S * cfg.L * 6 * cfg.d * 4 + cfg.S * 2 * cfg.d * 4
    io = cfg.S * 2 * cfg.d * cfg.A * 2
    total = cfg.S * cfg.L * (w_layer + kv_layer) + mod + io
    return {"weights": cfg.S * cfg.L * w_layer, "kv": cfg.S * cfg.L * kv_layer, "mod": mod, "io": io,
            "total": total}


def layer_bytes(cfg) -> int:
    """Bytes one layer-step must move at least once: its packed weights, its prefix
    K/V and its own modulation rows (the single-layer protocol's unit)."""
    ab = algorithmic_bytes(dataclasses.replace(cfg, L=1, S=1))
    return int(ab["weights"] + ab["kv"] + 6 * cfg.d * 4)


def algorithmic_flops(cfg) -> dict:
    """GEMM and attention FLOPs of one decision (2 per multiply-add)."""
    gemm = 2 * cfg.M * sum(n * k for n, k in cfg.gemm_shapes)
    attn = 2 * 2 * cfg.M * cfg.H * (cfg.P + cfg.M) * cfg.Dh   # Q K^T and P V
    return {"gemm": cfg.S * cfg.L * gemm, "attn": cfg.S * cfg.L * attn, "total": cfg.S * cfg.L * (gemm + attn)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_tensor_peak(sustained=False):
    """Dense bf16 (= f16) tensor peak in TFLOP/s: burst for a kernel timed alone,
    sustained for a kernel inside a long step."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained" if sustained else "bf16_tflops"]), "measured"
    return (1700.0 if sustained else 1900.0), "fallback"


class ClockSampler:
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
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- our arm

def run_ours(args, rank, world, local_rank):
    import torch
    import flow_matching_action_denoise_gb300 as fmad

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    fmad.load()
    cfg = fm_synth.config(args.workload)
    layers = [fm_synth.layer_weights(cfg, l) for l in range(cfg.L)]
    final = fm_synth.final_weights(cfg)
    scales = fm_synth.default_act_scales(cfg)
    weights = fmad.DeviceWeights(cfg, layers, final, device=device)
    del layers
    pol = fmad.Policy(cfg, act_scales=scales, weights=weights, device=device)
    # the one-step warm start needs its flow time in the plan: a policy of its own
    weights_for_warm = weights if cfg.weight_fmt != "nvfp4" else None
    # launch-mode variants of the same policy (same kernels): graph without PDL, no graph
    variants = {}
    if not args.no_variants:
        variants = {"graph_no_pdl": fmad.Policy(cfg, act_scales=scales, weights=weights, device=device,
                                                flags=fmad.FLAG_USE_GRAPH),
                    "eager_pdl": fmad.Policy(cfg, act_scales=scales, weights=weights, device=device,
                                             flags=fmad.FLAG_USE_PDL)}
        if cfg.weight_fmt != "nvfp4":   # the other consumer placement: inside the GEMMs
            variants["graph_pdl_fused_consumers"] = fmad.Policy(
                cfg, act_scales=scales, weights=weights, device=device,
                flags=fmad.FLAG_USE_GRAPH | fmad.FLAG_USE_PDL | fmad.FLAG_FUSED_CONSUMERS)
            variants["graph_pdl_o_consumer_in_gemm"] = fmad.Policy(
                cfg, act_scales=scales, weights=weights, device=device,
                flags=fmad.FLAG_USE_GRAPH | fmad.FLAG_USE_PDL | fmad.FLAG_O_CONSUMER_IN_GEMM)
    del weights
    kp, vp = fm_synth.prefix_kv(cfg)
    k_dev = torch.from_numpy(kp).to(device, torch.bfloat16)
    v_dev = torch.from_numpy(vp).to(device, torch.bfloat16)
    pol.set_prefix_kv(k_dev, v_dev)
    for vpol in variants.values():
        vpol.set_prefix_kv(k_dev, v_dev)
    noise = torch.from_numpy(fm_synth.noise(cfg, 0)).to(device)
    actions = torch.empty_like(noise)
    stream = torch.cuda.current_stream(device)
    per_layer, per_decision = fmad.kernel_count(pol.handle)
    pol_ws_bytes = pol.ws_bytes

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(device)

    for _ in range(args.warmup):
        pol.decode(noise, actions)
    barrier()

    # ---- device-resident timed region: per-decision events on the launching stream
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with ClockSampler(local_rank) as clocks:
        barrier()
        evs[0].record(stream)
        for i in range(args.steps):
            pol.decode(noise, actions)
            evs[i + 1].record(stream)
        barrier()
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)]
    total_ms = evs[0].elapsed_time(evs[-1])
    status = fmad.device_status(pol.handle)
    if status:
        raise RuntimeError(f"device error word {status}")

    # ---- end to end through the C ABI with host buffers (copies inside the timed region)
    h_noise = torch.from_numpy(fm_synth.noise(cfg, 1)).pin_memory()
    h_act = torch.empty_like(h_noise).pin_memory()
    for _ in range(max(1, args.warmup // 2)):
        fmad.decode_actions_host(pol.handle, h_noise, h_act)
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fmad.decode_actions_host(pol.handle, h_noise, h_act)
    barrier()
    e2e_ms = (time.perf_counter() - t0) * 1e3

    # ---- the same policy's other entry points: device-generated noise (Philox) with the
    # decision's own timestamps, and a session of the policy (shared weights, own state)
    for _ in range(2):
        fmad.decode_actions_seeded(pol.handle, 1234, 0, actions)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_infer = []
    e0.record(stream)
    for i in range(args.steps):
        fmad.decode_actions_seeded(pol.handle, 1234, i, actions)
        if i < 3:
            t_infer.append(fmad.last_timing(pol.handle)["t_infer_ns"] * 1e-6)
    e1.record(stream)
    torch.cuda.synchronize(device)
    seeded_ms = e0.elapsed_time(e1) / args.steps
    sess = pol.session()
    sess.set_prefix_kv(k_dev, v_dev)
    for _ in range(2):
        sess.decode(noise, actions)
    torch.cuda.synchronize(device)
    e0.record(stream)
    for _ in range(args.steps):
        sess.decode(noise, actions)
    e1.record(stream)
    torch.cuda.synchronize(device)
    session_ms = e0.elapsed_time(e1) / args.steps
    session_bytes = sess.ws_bytes
    sess.close()
    warm = time_warm_start(cfg, weights_for_warm, scales, k_dev, v_dev, noise, device, stream, args)

    # ---- dominant kernel timed alone: the gate|up GEMM, rotating weight copies; the
    # decision's own variant (GeGLU + E4M3 epilogue) and the fp32-plane building block
    if cfg.weight_fmt == "fp8":
        gemm = time_decision_gemm(cfg, scales, device)
        gemm_planes = time_dominant_gemm(cfg, pol, device, stream)
    else:
        gemm, gemm_planes = time_dominant_gemm_nvfp4(cfg, device, stream), None

    # ---- launch-mode variants (PDL off, graph off), same kernels and inputs
    variant_ms = {}
    for name, vpol in variants.items():
        for _ in range(args.warmup):
            vpol.decode(noise, actions)
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            vpol.decode(noise, actions)
        e1.record(stream)
        torch.cuda.synchronize(device)
        variant_ms[name] = round(e0.elapsed_time(e1) / args.steps, 4)
        vpol.close()

    # ---- max over ranks
    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], device)
    pol.close()
    if rank != 0:
        return None

    peak_gbs, peak_kind = measured_peaks()
    ab = algorithmic_bytes(cfg)
    lat_ms = total_ms / args.steps
    value = aggregate_ms_per_decision(total_ms, args.steps, world)
    achieved_gbs = ab["total"] / (lat_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 4),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(lat_ms, 4),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("fp8_e4m3" + (" (attention too)" if cfg.attn_fmt == "fp8" else "")) if cfg.weight_fmt == "fp8"
        else f"nvfp4 weights, {'nvfp4' if cfg.act_fmt == 'nvfp4' else 'fp8_e4m3'} activations, f16 MMA",
        "data": "synthetic (seeded N(0,1)/N(0,0.02) weights, prefix KV, noise; no trained weights)",
        "config": {"workload": cfg.name, "layers": cfg.L, "euler_steps": cfg.S, "action_rows": cfg.M,
                   "d_model": cfg.d, "heads": f"{cfg.H}x{cfg.Dh} (kv {cfg.Hkv})", "prefix_tokens": cfg.P,
                   "mlp": f"GeGLU {cfg.d}->2x{cfg.F}->{cfg.d}", "weights": cfg.weight_fmt,
                   "activations": cfg.act_fmt, "launch": "CUDA graph + PDL",
                   "l2": f"no flush: {ab['weights'] / 1e9:.1f} GB of weights streamed per decision >> 129 MB L2",
                   "parallelism": f"replicas x{world}"},
        "latency_ms": {"median": round(statistics.median(per), 4),
                       "p99": round(float(np.percentile(per, 99)), 4),
                       "min": round(min(per), 4)},
        "decision_hbm": {"algorithmic_bytes": int(ab["total"]), "achieved_gbs": round(achieved_gbs, 1),
                         "peak_gbs": peak_gbs, "frac": round(achieved_gbs / peak_gbs, 4),
                         "peak_kind": peak_kind},
        "e2e": {"value": round(e2e_ms / args.steps, 4), "unit": UNIT,
                "h2d_bytes_per_step": int(h_noise.numel() * 4), "d2h_bytes_per_step": int(h_act.numel() * 4)},
        "roofline": gemm,
        **({"roofline_planes_variant": gemm_planes} if gemm_planes else {}),
        "gpu_launches": int(per_decision * args.steps),
        "kernels_per_layer": per_layer,
        "launch_variants_ms": variant_ms,
        "clocks": clocks.summary(),
        "entry_points_ms": {
            "decode_actions_seeded": round(seeded_ms, 4),
            "t_infer_device": [round(t, 4) for t in t_infer],
            "session_decision": round(session_ms, 4),
            "session_workspace_mb": round(session_bytes / 2 ** 20, 1),
            "policy_workspace_mb": round(pol_ws_bytes / 2 ** 20, 1),
            **warm,
        },
    }
    if cfg.weight_fmt == "nvfp4":
        fl = algorithmic_flops(cfg)
        tpk, tkind = measured_tensor_peak(sustained=True)
        tf = fl["total"] / (lat_ms * 1e-3) / 1e12
        line["decision_tensor"] = {"algorithmic_flops": int(fl["total"]), "achieved_tflops": round(tf, 1),
                                   "peak_tflops": tpk, "frac": round(tf / tpk, 4),
                                   "peak_kind": f"{peak_kind_note(tkind)} sustained dense bf16"}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg)
    return line


def time_warm_start(cfg, weights, scales, k_dev, v_dev, noise, device, stream, args):
    """The one-step warm start (warm_t = 0.5, 3 actions executed) against the full
    decision, on a policy created with that flow time (CUDA events)."""
    import torch
    import flow_matching_action_denoise_gb300 as fmad
    if weights is None:
        return {}
    wcfg = dataclasses.replace(cfg, warm_t=0.5)
    pol = fmad.Policy(wcfg, act_scales=scales, weights=weights, device=device)
    pol.set_prefix_kv(k_dev, v_dev)
    out = torch.empty_like(noise)
    pol.decode(noise, out)
    for _ in range(3):
        pol.decode_warm(noise, 3, out)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        pol.decode_warm(noise, 3, out)
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / args.steps
    if fmad.device_status(pol.handle):
        raise RuntimeError("device error word set (warm start)")
    pol.close()
    return {"decode_warm_one_step": round(ms, 4), "warm_t": 0.5}


def time_graph(device, launches, replays=5):
    """Capture `launches` (callables taking a stream) back to back into one CUDA graph,
    replay it, and return the device time per launch in microseconds (CUDA events on
    the replay stream): kernel durations without host launch gaps."""
    import torch
    s = torch.cuda.Stream(device)
    for f in launches[:2]:   # one-time setup (function attributes, module load) outside the capture
        f(s)
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for f in launches:
            f(s)
    g.replay()
    torch.cuda.synchronize(device)
    cur = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for _ in range(replays):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize(device)
    us = e0.elapsed_time(e1) * 1e3 / (replays * len(launches))
    del g
    return us


def time_decision_gemm(cfg, scales, device, index=None):
    """The gate|up GEMM exactly as the decision launches it (GeGLU + E4M3 epilogue,
    the decision's split and cluster; kernel `index` of a layer-step; programmatic
    dependent launch), launched back to back through fm_test_launch_kernel over the
    layers of a policy whose packed weights rotate through more than 2x L2, timed with
    CUDA events on the replay stream: the average launch duration is the graph's time
    over its launches, so a launch's weight copies may overlap its predecessor's tail
    as they do in the decision. The same without programmatic dependent launch (each
    launch starts after the previous one has finished) is reported as `no_pdl`.
    Algorithmic bytes per launch: weights N K + activations M K + GeGLU codes M N / 2."""
    import torch
    import flow_matching_action_denoise_gb300 as fmad

    N, K, M = 2 * cfg.F, cfg.d, cfg.M
    l2 = l2_bytes(device)
    R = int(np.ceil(2 * l2 / (N * K))) + 1
    rcfg = dataclasses.replace(cfg, L=R, S=1)
    layer = fm_synth.layer_weights(rcfg, 0)
    kp, vp = fm_synth.prefix_kv(dataclasses.replace(rcfg, L=1))
    algo = N * K + M * K + M * (N // 2)

    def timed(flags):
        nonlocal index
        pol = fmad.Policy(rcfg, [layer] * R, fm_synth.final_weights(rcfg), act_scales=np.tile(scales[:1], (R, 1)),
                          device=device, flags=flags)
        pol.set_prefix_kv(torch.from_numpy(np.repeat(kp, R, 0)).to(device, torch.bfloat16),
                          torch.from_numpy(np.repeat(vp, R, 0)).to(device, torch.bfloat16))
        noise = torch.from_numpy(fm_synth.noise(rcfg, 0)).to(device)
        pol.decode(noise)   # fills every buffer the kernel reads
        torch.cuda.synchronize(device)
        if index is None:   # the gate|up GEMM's position in a layer-step: after the O GEMM's consumer
            index = 4 if fmad.kernel_count(pol.handle)[0] == 7 else 3
        launches = [lambda st, l=l: fmad.launch_kernel(pol.handle, l, 0, index, st) for l in range(R)] * 2
        us = time_graph(device, launches)
        if fmad.device_status(pol.handle):
            raise RuntimeError("device error word set (decision GEMM timing)")
        pol.close()
        return us

    us = timed(fmad.FLAG_USE_GRAPH | fmad.FLAG_USE_PDL)
    us_plain = timed(fmad.FLAG_USE_GRAPH)
    peak, kind = measured_peaks()
    achieved = algo / (us * 1e-6) / 1e9
    achieved_plain = algo / (us_plain * 1e-6) / 1e9
    return {"kernel": f"skinny_gemm_kernel<fp8> gate|up + GeGLU epilogue as in the decision (N={N}, K={K}, M={M})",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_kind": peak_kind_note(kind),
            "traffic": profiled_traffic(), "algorithmic_bytes": int(algo), "avg_launch_us": round(us, 3),
            "timing": f"CUDA graph of back-to-back launches with programmatic dependent launch, as in the "
                      f"decision, over {R} layers' weights (> 2x L2); graph time / launches, CUDA events",
            "no_pdl": {"avg_launch_us": round(us_plain, 3), "achieved": round(achieved_plain, 1),
                       "frac": round(achieved_plain / peak, 4)}}


def time_dominant_gemm(cfg, pol, device, stream):
    """Average duration of the gate|up GEMM (the largest weight stream of a layer) as the
    building block fm_test_skinny_gemm (fp32 partial planes), launched back to back through
    the C ABI over rotating packed weights (> 2x L2), timed with CUDA events on the
    launching stream."""
    import torch
    import flow_matching_action_denoise_gb300 as fmad

    N, K = 2 * cfg.F, cfg.d
    M = cfg.M
    nkb = K // 128
    s = next(s for s in range(1, nkb + 1) if nkb % s == 0 and (N // 128) * s >= 114)
    cs = 8
    while s % cs:
        cs //= 2
    nparts = s // cs
    nbytes = fmad.fm_packed_weight_bytes(N, K, fmad.FMT_FP8)
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    copies = max(4, int(np.ceil(2 * l2 / nbytes)) + 1)
    rng = np.random.default_rng(0)
    w = torch.from_numpy((rng.standard_normal((N, K)) * 0.02).astype(np.float32)).to(device)
    bufs = []
    scale = torch.empty(1, dtype=torch.float32, device=device)
    for _ in range(copies):
        b = torch.empty(nbytes + 1024, dtype=torch.uint8, device=device)
        ptr = b.data_ptr() + ((-b.data_ptr()) % 1024)
        fmad.fm_pack_weight(w, None, N, K, fmad.FMT_FP8, ptr, scale)
        bufs.append((b, ptr))
    del w
    a = torch.randint(0, 0x7E, (M, K), dtype=torch.uint8, device=device)
    out = torch.empty((nparts, M, N), dtype=torch.float32, device=device)
    launches = [lambda st, ptr=ptr: fmad.fm_test_skinny_gemm(a, M, K, ptr, N, fmad.FMT_FP8, s, cs, out, st)
                for _, ptr in bufs] * 4
    us = time_graph(device, launches)
    algo = N * K + M * K + nparts * M * N * 4
    peak, kind = measured_peaks()
    achieved = algo / (us * 1e-6) / 1e9
    return {"kernel": "skinny_gemm_kernel<fp8> gate|up (N=8192, K=1024, M=50, "
                      f"split {s}, cluster {cs})",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_kind": peak_kind_note(kind),
            "traffic": None, "algorithmic_bytes": int(algo), "avg_launch_us": round(us, 3),
            "timing": "CUDA graph of back-to-back launches over rotating weights (> 2x L2), CUDA events"}


def time_dominant_gemm_nvfp4(cfg, device, stream):
    """The NVFP4 gate|up GEMM (N = 2F, K = d, M rows, one K slice) launched back to
    back through the C ABI over rotating packed weights (> 2x L2); tensor-bound at
    M = 256, so reported against the dense bf16/f16 tensor peak."""
    import torch
    import flow_matching_action_denoise_gb300 as fmad

    N, K, M = 2 * cfg.F, cfg.d, cfg.M
    nbytes = fmad.fm_packed_weight_bytes(N, K, fmad.FMT_NVFP4)
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    copies = max(4, int(np.ceil(2 * l2 / nbytes)) + 1)
    rng = np.random.default_rng(0)
    w = torch.from_numpy((rng.standard_normal((N, K)) * 0.02).astype(np.float32)).to(device)
    bufs = []
    scale = torch.empty(1, dtype=torch.float32, device=device)
    for _ in range(copies):
        b = torch.empty(nbytes + 1024, dtype=torch.uint8, device=device)
        ptr = b.data_ptr() + ((-b.data_ptr()) % 1024)
        fmad.fm_pack_weight(w, None, N, K, fmad.FMT_NVFP4, ptr, scale)
        bufs.append((b, ptr))
    del w
    a = (torch.randn((M, K), device=device) * 4).to(torch.float16)
    out = torch.empty((1, M, N), dtype=torch.float32, device=device)
    launches = [lambda st, ptr=ptr: fmad.fm_test_skinny_gemm(a, M, K, ptr, N, fmad.FMT_NVFP4, 1, 1, out, st)
                for _, ptr in bufs] * 4
    us = time_graph(device, launches)
    flops = 2 * M * N * K
    peak, kind = measured_tensor_peak(sustained=False)
    achieved = flops / (us * 1e-6) / 1e12
    hbm = (nbytes + M * K * 2 + M * N * 4) / (us * 1e-6) / 1e9
    hpk, hkind = measured_peaks()
    return {"kernel": f"nvfp4_gemm_kernel gate|up (N={N}, K={K}, M={M}, split 1)",
            "bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind_note(kind)} dense bf16 burst (f16 same rate)",
            "traffic": None, "algorithmic_flops": int(flops), "avg_launch_us": round(us, 3),
            "hbm": {"achieved_gbs": round(hbm, 1), "peak_gbs": hpk, "frac": round(hbm / hpk, 4)},
            "timing": "CUDA graph of back-to-back launches over rotating weights (> 2x L2), CUDA events"}


def profiled_traffic(name="skinny_gemm_gu_m50.md"):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary,
    only while the kernel source is the one that was profiled (else None)."""
    import hashlib
    import re
    try:
        text = open(os.path.join(ROOT, "profiles", name)).read()
        src = open(os.path.join(ROOT, "flow_matching_action_denoise_gb300", "csrc", "gemm.cu"), "rb").read()
    except OSError:
        return None
    sha = re.search(r"sha256 prefix: ([0-9a-f]+)", text)
    traffic = re.search(r"traffic_bytes_per_launch: (\d+)", text)
    if not sha or not traffic or hashlib.sha256(src).hexdigest()[:len(sha.group(1))] != sha.group(1):
        return None
    return int(traffic.group(1))


def peak_kind_note(kind):
    return "of measured" if kind == "measured" else "of fallback"


# ---------------------------------------------------------------- CPU oracle (baseline / reference arm)

def host_cores() -> dict:
    try:
        aff = len(os.sched_getaffinity(0))
    except AttributeError:
        aff = os.cpu_count()
    return {"affinity": aff, "os_cpu_count": os.cpu_count()}


def oracle_layer_steps_ms(cfg, n_layers: int, n_steps: int) -> float:
    """Time the FP64 oracle as it stands on n_steps Euler steps through the first
    n_layers layers of `cfg` (weights prepared outside the timing), in ms per
    layer-step."""
    from oracle import model as O
    sub = dataclasses.replace(cfg, L=n_layers)
    layers = [fm_synth.layer_weights(sub, l) for l in range(n_layers)]
    conds = fm_synth.step_conds(sub) if sub.cond == "given" else None
    model = O.Model(sub, layers, fm_synth.final_weights(sub), conds)
    del layers
    kp, vp = fm_synth.prefix_kv(sub)
    kp, vp = kp.astype(np.float64), vp.astype(np.float64)
    scales = fm_synth.default_act_scales(sub)
    a = fm_synth.noise(sub, 0).astype(np.float64)
    t0 = time.perf_counter()
    for k in range(n_steps):
        a = O.euler_step(model, k, a, kp, vp, scales)
    return (time.perf_counter() - t0) * 1e3 / (n_layers * n_steps)


ONE_THREAD_ENV = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1",
                  "BLIS_NUM_THREADS": "1", "VECLIB_MAXIMUM_THREADS": "1"}


def oracle_one_thread_ms(workload: str) -> float | None:
    """The same single-layer oracle timing in a fresh process whose BLAS runs one thread."""
    code = ("import sys; sys.path.insert(0, %r); import bench, fm_synth; "
            "print(bench.oracle_layer_steps_ms(fm_synth.config(%r), 1, 1))" % (ROOT, workload))
    try:
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300,
                           env={**os.environ, **ONE_THREAD_ENV})
        return float(r.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError):
        return None


def cpu_baseline(cfg, samples: int = 1):
    """Time the FP64 oracle as it stands on this host's cores (BLAS threads = numpy's
    default, all cores) on a bounded sample of the workload: two Euler steps of all 18
    layers of the expert (the first layers of one step for larger decoders), scaled to
    ms per decision. Also one bounded oracle timing per other workload (each scaled to
    its own decision) and the single-layer workload with one BLAS thread."""
    big = cfg.M * cfg.d > 100_000
    n_layers = min(cfg.L, 2) if big else cfg.L
    steps = 1 if big else 2
    times = [oracle_layer_steps_ms(cfg, n_layers, steps) * cfg.S * cfg.L for _ in range(samples)]
    what = (f"{n_layers} layers of Euler step 0" if big else f"{steps} Euler steps x {cfg.L} layers")
    out = {"value": round(statistics.median(times), 1), "unit": UNIT, "cores": host_cores()["affinity"],
           "kind": "oracle",
           "sample": f"{what} of {cfg.name} (FP64 numpy, weights prepared outside the timing), "
                     f"scaled to one {cfg.L}-layer x {cfg.S}-step decision",
           "sampled_layer_steps": n_layers * steps, "scaled_to_layer_steps": cfg.L * cfg.S,
           "host": host_cores(), "blas_threads": "numpy default (all cores)"}
    per = {}
    l0 = fm_synth.config("layer_fp8_m10")
    per["layer_fp8_m10"] = {"ms_per_decision": round(oracle_layer_steps_ms(l0, 1, 1), 2),
                            "sample": "the whole 1-layer x 1-step decision"}
    one = oracle_one_thread_ms("layer_fp8_m10")
    per["layer_fp8_m10_one_thread"] = {"ms_per_decision": None if one is None else round(one, 2),
                                       "sample": "the whole 1-layer x 1-step decision, BLAS limited to 1 thread"}
    for name, nl in (("expert_bf16_m63", 2), ("wam_nvfp4_m256", 1)):
        if name == cfg.name:
            continue
        c = fm_synth.config(name)
        per[name] = {"ms_per_decision": round(oracle_layer_steps_ms(c, nl, 1) * c.L * c.S, 1),
                     "sample": f"{nl} layer(s) x 1 Euler step, scaled to {c.L} x {c.S}"}
    out["per_workload"] = per
    return out


def max_over_ranks(values, device):
    """Element-wise max of per-rank timings (every rank calls it; one rank returns
    its own): the slowest replica sets the job's time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def aggregate_ms_per_decision(total_ms: float, steps: int, world: int) -> float:
    """Whole-job figure for N replicas that each ran `steps` decisions in (the max of)
    total_ms: time per decision of the job."""
    return total_ms / (steps * world)


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each of the K timed steps (after W warm-up
    steps) is one Euler step through all layers of the workload - a bounded sample, one
    S-th of a decision - and the reported value is the median step scaled by S to ms
    per decision. Rank 0 only."""
    if rank != 0:
        return None
    from oracle import model as O
    cfg = fm_synth.config(args.workload)
    big = cfg.M * cfg.d > 100_000
    n_layers = min(cfg.L, 2) if big else cfg.L
    sub = dataclasses.replace(cfg, L=n_layers)
    layers = [fm_synth.layer_weights(sub, l) for l in range(n_layers)]
    model = O.Model(sub, layers, fm_synth.final_weights(sub))
    del layers
    kp, vp = fm_synth.prefix_kv(sub)
    kp, vp = kp.astype(np.float64), vp.astype(np.float64)
    scales = fm_synth.default_act_scales(sub)
    a = fm_synth.noise(sub, 0).astype(np.float64)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        O.euler_step(model, i % cfg.S, a, kp, vp, scales)
        if i >= args.warmup:
            times.append((time.perf_counter() - t0) * 1e3)
    step_ms = statistics.median(times)
    scale = cfg.S * cfg.L / n_layers
    value = step_ms * scale
    cores = host_cores()
    sample = (f"one Euler step x {n_layers} of {cfg.L} layers of {cfg.name} per timed step (FP64 numpy, BLAS "
              f"on all cores, weights prepared outside the timing); value = median step x {scale:g}")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 2),
            "step": f"one Euler step through {n_layers} layers (1/{scale:g} of a decision)",
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "layers": cfg.L, "euler_steps": cfg.S, "action_rows": cfg.M},
            "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": cores["affinity"], "kind": "oracle",
                             "sample": sample, "host": cores},
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def profile_case(workload=WORKLOAD):
    """Small ncu target: a 1-layer, 1-step policy of the bench workload (about 18 MiB
    on the device); the second decision runs inside a cudaProfilerStart/Stop range
    (ncu --profile-from-start off)."""
    import torch
    import flow_matching_action_denoise_gb300 as fmad
    cfg = fm_synth.config(workload, L=1, S=1)
    pol = fmad.Policy(cfg, [fm_synth.layer_weights(cfg, 0)], fm_synth.final_weights(cfg),
                      act_scales=fm_synth.default_act_scales(cfg))
    kp, vp = fm_synth.prefix_kv(cfg)
    pol.set_prefix_kv(torch.from_numpy(kp).cuda().to(torch.bfloat16), torch.from_numpy(vp).cuda().to(torch.bfloat16))
    noise = torch.from_numpy(fm_synth.noise(cfg, 0)).cuda()
    pol.decode(noise)
    torch.cuda.synchronize()
    torch.cuda.profiler.start()
    pol.decode(noise)
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    pol.close()


def run_bf16_protocol(args):
    """Matched 16-bit workload (bf16 weights and activations, M = 63, 18 layers x 10
    steps, prefix 788): 100 consecutive decisions on one policy with new noise each,
    the 768 image-token rows of the prefix refreshed before every 5th decision.
    Reports the mean decision latency without the refresh, the refresh latency, the
    mean per decision including refreshes, and capsule restore + decision against
    set_prefix_kv + decision. Every input is resident on the device beforehand."""
    import torch
    import flow_matching_action_denoise_gb300 as fmad
    device = torch.device("cuda", 0)
    fmad.load()
    cfg = fm_synth.config("expert_bf16_m63")
    rows, every, n_dec = 768, 5, 100
    layers = [fm_synth.layer_weights(cfg, l) for l in range(cfg.L)]
    weights = fmad.DeviceWeights(cfg, layers, fm_synth.final_weights(cfg), device=device)
    del layers
    pol = fmad.Policy(cfg, weights=weights, device=device)
    del weights
    bf = lambda a: torch.from_numpy(a).to(device, torch.bfloat16)
    kp, vp = fm_synth.prefix_kv(cfg)
    k_dev, v_dev = bf(kp), bf(vp)
    pol.set_prefix_kv(k_dev, v_dev)
    refresh = {d: tuple(bf(a) for a in fm_synth.prefix_kv_rows(cfg, d // every, rows))
               for d in range(every, n_dec, every)}
    noise = [torch.from_numpy(fm_synth.noise(cfg, d)).to(device) for d in range(n_dec)]
    actions = torch.empty_like(noise[0])
    stream = torch.cuda.current_stream(device)
    for _ in range(max(3, args.warmup)):
        pol.decode(noise[0], actions)
    pol.set_prefix_kv(k_dev, v_dev)
    torch.cuda.synchronize(device)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    marks = []
    with ClockSampler(0) as clocks:
        start = ev()
        start.record(stream)
        for d in range(n_dec):
            r0 = r1 = None
            if d in refresh:
                r0, r1 = ev(), ev()
                r0.record(stream)
                pol.refresh_prefix(0, rows, *refresh[d])
                r1.record(stream)
            d0, d1 = ev(), ev()
            d0.record(stream)
            pol.decode(noise[d], actions)
            d1.record(stream)
            marks.append((r0, r1, d0, d1))
        end = ev()
        end.record(stream)
        torch.cuda.synchronize(device)
    if fmad.device_status(pol.handle):
        raise RuntimeError("device error word set")
    dec = [d0.elapsed_time(d1) for _, _, d0, d1 in marks]
    ref = [r0.elapsed_time(r1) for r0, r1, _, _ in marks if r0 is not None]
    total = start.elapsed_time(end)

    # capsule restore + decision vs re-set prefix + decision (same resulting state)
    n = fmad.state_size(pol.handle)
    cap = torch.empty(n, dtype=torch.uint8, device=device)
    fmad.snapshot_state(pol.handle, cap, n, True)
    reps = 20
    t = {}
    for name in ("restore", "set_prefix"):
        e0, e1 = ev(), ev()
        e0.record(stream)
        for _ in range(reps):
            if name == "restore":
                fmad.restore_state(pol.handle, cap, n, True)
            else:
                pol.set_prefix_kv(k_dev, v_dev)
            pol.decode(noise[0], actions)
        e1.record(stream)
        torch.cuda.synchronize(device)
        t[name] = e0.elapsed_time(e1) / reps
    pol.close()
    peak_gbs, peak_kind = measured_peaks()
    ab = algorithmic_bytes(cfg)["total"]
    mean_dec = statistics.fmean(dec)
    return {"protocol": "bf16 persistent prefix, refresh every 5th decision", "workload": cfg.name,
            "decisions": n_dec, "unit": "ms",
            "decision_mean_excl_refresh": round(mean_dec, 4),
            "decision_p99": round(float(np.percentile(dec, 99)), 4),
            "refresh_mean": round(statistics.fmean(ref), 4), "refreshes": len(ref),
            "mean_per_decision_incl_refresh": round(total / n_dec, 4),
            "restore_plus_decision": round(t["restore"], 4),
            "set_prefix_plus_decision": round(t["set_prefix"], 4),
            "state_bytes": n,
            "decision_hbm": {"algorithmic_bytes": int(ab), "achieved_gbs": round(ab / (mean_dec * 1e-3) / 1e9, 1),
                             "peak_gbs": peak_gbs, "frac": round(ab / (mean_dec * 1e-3) / 1e9 / peak_gbs, 4),
                             "peak_kind": peak_kind},
            "clocks": clocks.summary()}


def l2_bytes(device):
    import torch
    props = torch.cuda.get_device_properties(device)
    return getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)


def run_layer_protocol(args):
    """Single decoder layer, one denoise step (M = 10, d = 1024, prefix 64, FP8): R
    copies of the layer's weights in separate buffers, R * 15 MB >= 2x L2, run as one
    R-layer, 1-step policy (one CUDA graph with PDL); time per layer = decision time / R
    (the step head and tail are included, spread over the R layers)."""
    import torch
    import flow_matching_action_denoise_gb300 as fmad
    device = torch.device("cuda", 0)
    fmad.load()
    base = fm_synth.config("layer_fp8_m10")
    layer = fm_synth.layer_weights(base, 0)
    per_layer = layer_bytes(base)
    R = int(np.ceil(2 * l2_bytes(device) / per_layer)) + 1
    cfg = fm_synth.config("layer_fp8_m10", L=R)
    conds = fm_synth.step_conds(cfg)
    scales = np.tile(np.loadtxt(os.path.join(ROOT, "tests", "golden", "act_scales_layer_fp8_m10.txt"),
                                ndmin=2).astype(np.float32), (R, 1))
    flags = fmad.FLAG_USE_GRAPH | fmad.FLAG_USE_PDL | (fmad.FLAG_FUSED_CONSUMERS if args.fused_consumers else 0)
    pol = fmad.Policy(cfg, [layer] * R, fm_synth.final_weights(cfg), act_scales=scales, conds=conds, device=device,
                      flags=flags)
    kernels_per_layer = fmad.kernel_count(pol.handle)[0]
    kp, vp = fm_synth.prefix_kv(cfg)
    pol.set_prefix_kv(torch.from_numpy(kp).to(device, torch.bfloat16), torch.from_numpy(vp).to(device, torch.bfloat16))
    noise = torch.from_numpy(fm_synth.noise(cfg, 0)).to(device)
    actions = torch.empty_like(noise)
    stream = torch.cuda.current_stream(device)
    for _ in range(max(3, args.warmup)):
        pol.decode(noise, actions)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clocks:
        e0.record(stream)
        for _ in range(args.steps):
            pol.decode(noise, actions)
        e1.record(stream)
        torch.cuda.synchronize(device)
    if fmad.device_status(pol.handle):
        raise RuntimeError("device error word set")
    us = e0.elapsed_time(e1) * 1e3 / args.steps / R
    peak, kind = measured_peaks()
    gbs = per_layer / (us * 1e-6) / 1e9
    pol.close()
    return {"protocol": "single layer, rotating weight copies", "workload": base.name, "copies": R,
            "bytes_per_layer": int(per_layer), "us_per_layer": round(us, 3), "achieved_gbs": round(gbs, 1),
            "peak_gbs": peak, "frac": round(gbs / peak, 4), "peak_kind": peak_kind_note(kind),
            "kernels_per_layer": kernels_per_layer, "fused_consumers": bool(args.fused_consumers),
            "steps": args.steps, "clocks": clocks.summary()}


def run_handoff_protocol(args):
    """What a stage boundary costs by itself: (a) a CUDA graph of dependent empty kernels
    (programmatic dependent launch, as the decision launches its kernels, and plain
    stream order; also in thread-block clusters and with every thread storing 16 words
    after its wait), microseconds per kernel; (b) grid-wide barriers inside one cooperative
    launch (release/acquire at gpu scope, and fences around relaxed atomics), the median
    over CTAs of nanoseconds per round. Both at 1 CTA, at the decision's typical grid
    sizes and at one and two CTAs per SM."""
    import torch
    import flow_matching_action_denoise_gb300 as fmad
    device = torch.device("cuda", 0)
    fmad.load()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    grids = [1, 64, sms, 2 * sms]
    writes_max = 16
    scratch = torch.zeros(1 + 2 * sms * 256 * writes_max, dtype=torch.int32, device=device)
    chain, barrier = [], []
    with ClockSampler(0) as clocks:
        for ctas in grids:
            for pdl in (True, False):
                us = fmad.pdl_chain(ctas, 256, 1000, 10, pdl, scratch)
                chain.append({"ctas": ctas, "threads": 256, "pdl": pdl, "cluster": 1, "writes": 0,
                              "us_per_kernel": round(us, 3)})
        for cluster in (1, 2, 8):   # the decision's kernels run in clusters and store their outputs
            for writes in (0, writes_max):
                us = fmad.pdl_chain(64, 256, 1000, 10, True, scratch, cluster, writes)
                chain.append({"ctas": 64, "threads": 256, "pdl": True, "cluster": cluster, "writes": writes,
                              "us_per_kernel": round(us, 3)})
        for ctas in grids:
            for mode, name in ((0, "release/acquire"), (1, "fences + relaxed atomics")):
                out = torch.zeros(2 * ctas, dtype=torch.int64, device=device)
                rounds = 2000
                if fmad.grid_barrier(ctas, 256, rounds, mode, 10 ** 9, scratch, out) != 0:
                    raise RuntimeError("grid barrier wait ran out")
                o = out.cpu().numpy().reshape(ctas, 2)
                barrier.append({"ctas": ctas, "threads": 256, "ordering": name,
                                "ns_per_round": round(float(np.median(o[:, 0] / o[:, 1])), 1)})
    return {"protocol": "stage hand-off cost", "kernels_per_graph": 1000, "barrier_rounds": 2000,
            "pdl_chain": chain, "grid_barrier": barrier, "clocks": clocks.summary()}


def run_timeline(args):
    """Where a decision's time goes: one decision replayed as the same CUDA graph with a
    per-CTA timeline (fm_decode_timeline), summarised per kernel position in a
    layer-step: the hand-off (the previous kernel's last CTA exit -> this kernel's last
    programmatic-dependent-launch wait return), the kernel's own time after that wait,
    and the median of each recorded stamp after the wait (us), averaged over every
    layer-step but the first two."""
    import collections
    import torch
    import flow_matching_action_denoise_gb300 as fmad
    device = torch.device("cuda", 0)
    fmad.load()
    cfg = fm_synth.config(args.workload, S=args.timeline_steps) if args.timeline_steps else fm_synth.config(args.workload)
    layers = [fm_synth.layer_weights(cfg, l) for l in range(cfg.L)]
    scales = fm_synth.default_act_scales(cfg) if cfg.act_fmt in ("fp8", "nvfp4") else None
    pol = fmad.Policy(cfg, layers, fm_synth.final_weights(cfg), act_scales=scales, device=device)
    del layers
    kp, vp = fm_synth.prefix_kv(cfg)
    pol.set_prefix_kv(torch.from_numpy(kp).to(device, torch.bfloat16), torch.from_numpy(vp).to(device, torch.bfloat16))
    noise = torch.from_numpy(fm_synth.noise(cfg, 0)).to(device)
    act = torch.empty_like(noise)
    for _ in range(max(3, args.warmup)):
        pol.decode(noise, act)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        pol.decode(noise, act)
    e1.record()
    torch.cuda.synchronize(device)
    plain_ms = e0.elapsed_time(e1) / args.steps
    nrec = 2 * (1 + cfg.L * cfg.S * 8) * 256
    buf = torch.zeros(64 + 128 * nrec, dtype=torch.uint8, device=device)
    fmad.decode_timeline(pol.handle, noise, act, buf, buf.numel())
    if fmad.device_status(pol.handle):
        raise RuntimeError("device error word set (timeline)")
    pol.close()
    recs = fmad.parse_timeline(buf.cpu().numpy())
    by = collections.defaultdict(list)
    for r in recs:
        by[(r["kind"], r["grid"])].append(r)
    inst = []
    for sig, rs in by.items():
        n = sig[1][0] * sig[1][1]
        rs.sort(key=lambda r: r["t"][0])
        inst += [(sig, rs[i:i + n]) for i in range(0, len(rs), n)]
    inst.sort(key=lambda x: min(r["t"][0] for r in x[1]))
    kinds = {1: "gemm", 2: "attention", 3: "row", 4: "nvfp4_gemm"}
    kpl = (len(inst) - 1) // (cfg.L * cfg.S)
    per = collections.defaultdict(list)
    prev_exit = None
    for i, (sig, rs) in enumerate(inst):
        wait = max(r["t"][1] for r in rs)
        ex = max(max(r["t"]) for r in rs)
        stamps = [float(np.median([r["t"][j] - wait for r in rs if r["t"][j]])) / 1e3
                  if any(r["t"][j] for r in rs) else None for j in range(2, 15)]
        if i >= 1 and (i - 1) // kpl >= 2:
            per[((i - 1) % kpl, f"{kinds[sig[0]]} grid {sig[1][0]}x{sig[1][1]}")].append(
                ((wait - prev_exit) / 1e3, (ex - wait) / 1e3, stamps))
        prev_exit = ex
    rows = []
    for (pos, name), v in sorted(per.items()):
        st = [round(float(np.mean([s[j] for _, _, s in v])), 2) if v[0][2][j] is not None else None for j in range(13)]
        rows.append({"position": pos, "kernel": name, "handoff_us": round(float(np.mean([a for a, _, _ in v])), 2),
                     "own_us": round(float(np.mean([b for _, b, _ in v])), 2),
                     "stamps_after_wait_us": [x for x in st if x is not None]})
    t0 = min(r["t"][0] for r in recs)
    t1 = max(max(r["t"]) for r in recs)
    return {"protocol": "in-graph kernel timeline (fm_decode_timeline)", "workload": cfg.name, "layers": cfg.L,
            "euler_steps": cfg.S, "decision_ms": round(plain_ms, 4), "timeline_decision_ms": round((t1 - t0) / 1e6, 4),
            "kernels_per_layer_recorded": kpl,
            "per_layer_step_us": round(sum(r["handoff_us"] + r["own_us"] for r in rows), 2), "kernels": rows}


def run_gemm_sweep(args):
    """Skinny GEMM + fused consumer (fm_gemm_consumer: bias + gated residual + AdaRMSNorm
    + static E4M3 quantise) over M in {1, 10, 50, 63}, K in {1024, 2048, 4096},
    N in {1024, 4096, 8192, 16384}, K-split s in {1, 2, 4, 8, 16}: back-to-back calls
    over rotating packed weights (> 2x L2), captured in a CUDA graph, CUDA events.
    Algorithmic bytes per call:
    K N (weights) + M K (activations) + 9 M N (x read/write, partial write/read, codes)
    + 16 N (bias, gate, scale, shift)."""
    import torch
    import flow_matching_action_denoise_gb300 as fmad
    device = torch.device("cuda", 0)
    fmad.load()
    stream = torch.cuda.current_stream(device)
    peak, kind = measured_peaks()
    l2 = l2_bytes(device)
    rows = []
    f32 = lambda n, v=0.1: torch.full((n,), v, dtype=torch.float32, device=device)
    for K in (1024, 2048, 4096):
        for N in (1024, 4096, 8192, 16384):
            nbytes = fmad.fm_packed_weight_bytes(N, K, fmad.FMT_FP8)
            copies = min(256, int(np.ceil(2 * l2 / nbytes)) + 1)
            w = (torch.randn(N, K, device=device) * 0.02)
            pool = torch.empty(copies * (nbytes + 1024), dtype=torch.uint8, device=device)
            base = pool.data_ptr() + ((-pool.data_ptr()) % 1024)
            ptrs = [base + i * (nbytes + 1024) for i in range(copies)]
            s_w = torch.empty(1, dtype=torch.float32, device=device)
            for ptr in ptrs:
                fmad.fm_pack_weight(w, None, N, K, fmad.FMT_FP8, ptr, s_w)
            del w
            for M in (1, 10, 50, 63):
                a = torch.randint(0, 0x70, (M, K), dtype=torch.uint8, device=device)
                x = torch.randn(M, N, device=device)
                q = torch.empty((M, N), dtype=torch.uint8, device=device)
                bias, gate, scale, shift = f32(N, 0.01), f32(N, 0.1), f32(N, 0.1), f32(N, 0.0)
                s_a, s_q = f32(1, 0.02), f32(1, 0.05)
                for s in (1, 2, 4, 8, 16):
                    row = {"M": M, "K": K, "N": N, "s": s}
                    try:
                        sb = fmad.gemm_consumer_scratch_bytes(M, N, K, fmad.FMT_FP8, s)
                    except fmad.FmError as e:
                        row["skipped"] = str(e).split(":")[-1].strip()[:80]
                        rows.append(row)
                        continue
                    scratch = torch.empty(max(sb // 4, 1), dtype=torch.float32, device=device)
                    launches = [lambda st, ptr=ptr: fmad.fm_gemm_consumer(a, M, K, ptr, N, fmad.FMT_FP8, s, s_a, s_w,
                                                                          bias, x, gate, scale, shift, 1e-6, s_q, q,
                                                                          scratch, sb, st)
                                for ptr in ptrs] * max(1, 24 // copies)
                    us = time_graph(device, launches, replays=3)
                    algo = K * N + M * K + 9 * M * N + 16 * N
                    gbs = algo / (us * 1e-6) / 1e9
                    row.update({"us": round(us, 3), "algorithmic_bytes": algo, "gbs": round(gbs, 1),
                                "frac": round(gbs / peak, 4)})
                    rows.append(row)
            del pool
            torch.cuda.empty_cache()
    done = [r for r in rows if "us" in r]
    best = max(done, key=lambda r: r["frac"])
    return {"protocol": "skinny GEMM + fused consumer sweep (FP8)", "points": len(rows), "measured": len(done),
            "peak_gbs": peak, "peak_kind": peak_kind_note(kind), "best": best, "rows": rows}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["expert_fp8_m50", "expert_fp8attn_m50", "wam_nvfp4_m256", "wam_w4a4_m256",
                                           "expert_bf16_m63"],
                    default=WORKLOAD,
                    help="decoder workload (default: the 18-layer FP8 action expert, M = 50)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-variants", action="store_true", help="skip the PDL-off / graph-off timings")
    ap.add_argument("--profile-case", action="store_true",
                    help="run only the small 1-layer, 1-step case for ncu (profiler range on its 2nd decision)")
    ap.add_argument("--fused-consumers", action="store_true",
                    help="with --layer-protocol: run the consumers inside the GEMMs")
    ap.add_argument("--layer-protocol", action="store_true",
                    help="run only the single-layer protocol (M = 10, rotating weight copies > 2x L2)")
    ap.add_argument("--gemm-sweep", action="store_true",
                    help="run only the skinny GEMM + fused consumer sweep (240 points)")
    ap.add_argument("--handoff-protocol", action="store_true",
                    help="cost of a kernel boundary (PDL graph chain) and of an in-kernel grid barrier")
    ap.add_argument("--timeline", action="store_true",
                    help="run only the in-graph kernel timeline of one decision of --workload")
    ap.add_argument("--timeline-steps", type=int, default=0,
                    help="with --timeline: Euler steps of the timed policy (0 = the workload's)")
    ap.add_argument("--bf16-protocol", action="store_true",
                    help="run only the matched 16-bit persistence protocol (100 decisions, refresh every 5th)")
    args = ap.parse_args()
    if args.bf16_protocol:
        print(json.dumps(run_bf16_protocol(args)), flush=True)
        return
    if args.timeline:
        print(json.dumps(run_timeline(args)), flush=True)
        return
    if args.handoff_protocol:
        print(json.dumps(run_handoff_protocol(args)), flush=True)
        return
    if args.layer_protocol:
        print(json.dumps(run_layer_protocol(args)), flush=True)
        return
    if args.gemm_sweep:
        print(json.dumps(run_gemm_sweep(args)), flush=True)
        return
    if args.profile_case:
        profile_case(args.workload)
        return
    if args.workload == "expert_bf16_m63":
        raise SystemExit("expert_bf16_m63 is measured by --bf16-protocol (and profiled with --profile-case)")
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
        line = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
