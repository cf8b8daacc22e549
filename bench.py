#!/usr/bin/env python3
"""Benchmark of the routed-expert RVQ MoE step on one GB300 (or N replicas).

Default workload: one decode layer with the pages' expert shape -- d=7168,
f=1536, E=384 experts, top-16, one token per step, fp32 activations (the
configuration the metric is quoted on).  A step = router GEMV + top-k/softmax
+ fused RVQ gate/up + SwiGLU + down + gate-weighted combine for one token.
Per step a fresh token is taken from a pool of 64; L2 is flushed between steps
(a 256 MiB write outside the timed events), so every step streams its ~210 MB
from HBM.

Also measured (extra keys of the same line): batched decode (128 tokens) and a
prefill chunk (512 tokens) on the grouped tensor-core path, the full-depth
decode stack (92 layers x 64 experts, lookahead 6 vs off, captured in CUDA
graphs), a tiered expert bank (16 layers x 64 experts in pinned host memory
behind HBM caches of three sizes, lookahead 0/6/16), the RVQ encoder on one expert,
the end-to-end number
through the C ABI with host buffers, and the CPU oracle on the host cores.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
For N > 1 it is launched once per GPU by torch.distributed.run; every rank
runs its own replica (the step does not shard) and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "routed-expert tokens/s per MoE layer"
UNIT = "tok/s"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0
DECODE_POOL = 64


# ---------------------------------------------------------------- helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's x: the job's time is its slowest rank's."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured", p
    except Exception:
        return FALLBACK_HBM_GBS, "fallback", None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.lines = []
        self.windows = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        import threading
        self.t0 = time.time()
        self.thread = None
        if self.proc:
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, start: float, end: float):
        self.windows.append((start, end))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        inside = [l for (ts, l) in self.lines
                  if any(a - 0.05 <= ts <= b + 0.05 for a, b in self.windows)]
        rows = []
        for l in inside:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]), active=parts[4],
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows)}


def source_hash(*rel_paths) -> str:
    h = hashlib.sha256()
    for p in rel_paths:
        with open(os.path.join(ROOT, p), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_tag: str):
    """DRAM bytes per launch of a kernel from the committed ncu summary, if the summary was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as fh:
        for line in fh:
            if ":" in line and not line.lstrip().startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    try:
        if vals.get("source_sha256_16") != source_hash(*vals["sources"].split()):
            return None
        return float(vals["dram_bytes_per_launch_full_size"])
    except Exception:
        return None


# ---------------------------------------------------------------- native arm

def expert_code_bytes(d: int, f: int) -> int:
    """Code bytes of one expert: 3 matrices of d x f weights, 3 stages x 1 byte per 8 weights
    (12,386,304 B at d=7168, f=1536)."""
    return 3 * 3 * d * f // 8


def host_description() -> dict:
    """The host cores the CPU baseline runs on: count and model name."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":", 1)[0].strip() == "Model name":
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as fh:
                for line in fh:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    import platform
    return {"nproc": os.cpu_count(), "cpu_model": model, "machine": platform.machine()}


def decode_algorithmic_bytes(w):
    """Algorithmic bytes per decode step and per gate/up and down launch."""
    codes = expert_code_bytes(w.d, w.f)
    cb_mat = 3 * 256 * 8 * 4
    gate_up = w.top_k * (2 * codes // 3 + 2 * cb_mat) + w.d * 4
    down = w.top_k * (codes // 3 + cb_mat)
    router = w.n_experts * w.d * 4 + w.d * 4
    step = gate_up + down + router + 2 * w.d * 4  # + out write
    return step, gate_up, down


def run_decode(args, dev, out):
    from rvq_compressed_expert_gb300 import binding as B
    from rvq_compressed_expert_gb300 import synth
    from rvq_compressed_expert_gb300.layer import MoELayer

    w = synth.WORKLOADS["decode"]
    layer = MoELayer(w, seed=0, layer=0, device=dev, crc=True)
    # opening the layer with every record's payload crc32 checked on the device
    # (create + destroy with and without the check, each after one untimed call; the check's
    # cost is the difference)
    def create_s(flags, reps=5):
        c = B.make_config(w.d, w.f, w.n_experts, w.top_k, w.act_dtype, 1, 0, flags, layer.layer)
        B.waste_moe_destroy(B.waste_moe_create(c, layer.router_w, layer.router_b, layer.records, layer.stride,
                                               layer.codebooks))
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            t0 = time.perf_counter()
            B.waste_moe_destroy(B.waste_moe_create(c, layer.router_w, layer.router_b, layer.records, layer.stride,
                                                   layer.codebooks))
            best = min(best, time.perf_counter() - t0)
        return best
    plain_s = create_s(0)
    with_s = create_s(B.FLAG_VERIFY_CRC)
    verify_s = max(with_s - plain_s, 1e-9)
    out["verify_crc"] = dict(create_seconds=plain_s, create_with_verify_seconds=with_s, verify_seconds=verify_s,
                             bank_bytes=w.n_experts * layer.stride,
                             verify_gb_per_s=w.n_experts * layer.stride / verify_s / 1e9)
    pool = [synth.hidden(100 + i, 1, w.d, "f32", dev) for i in range(DECODE_POOL)]
    idx, gate, logits, y = layer.alloc_outputs(1)
    h_in = torch.empty(1, w.d, dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    K = args.steps

    def step():
        layer.step(h_in, 1, idx, gate, y, 0, logits)

    # the decode step (one persistent kernel) captured in a CUDA graph, replayed per token
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(3):
            h_in.copy_(pool[i])
            step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        h_in.copy_(pool[i % DECODE_POOL])
        flush.zero_()
        graph.replay()
    torch.cuda.synchronize()
    layer.reset_stats()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if args.world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start = time.time()
    for i in range(K):
        h_in.copy_(pool[i % DECODE_POOL])
        flush.zero_()
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    t_end = time.time()
    if args.world > 1:
        torch.distributed.barrier()
    args.sampler.mark(t_start, t_end)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), args.world, dev)
    st = layer.stats()

    # the same step as one persistent kernel (router, top-k, expert units and combine from a
    # device queue), on a second handle over the same weights, for comparison
    ucfg = B.make_config(w.d, w.f, w.n_experts, w.top_k, w.act_dtype, 1, 0,
                         B.FLAG_STEP_KERNEL, layer.layer)
    uh = B.waste_moe_create(ucfg, layer.router_w, layer.router_b, layer.records, layer.stride,
                            layer.codebooks)
    with torch.cuda.stream(side):
        for i in range(3):
            B.waste_moe_step(uh, h_in, 1, idx, gate, logits, y, 0)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ug = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ug):
        B.waste_moe_step(uh, h_in, 1, idx, gate, logits, y, 0)
    uev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        h_in.copy_(pool[i % DECODE_POOL])
        flush.zero_()
        uev[i][0].record(stream)
        ug.replay()
        uev[i][1].record(stream)
    torch.cuda.synchronize()
    unfused_ms = sum(a.elapsed_time(b) for a, b in uev) / K
    del ug
    B.waste_moe_destroy(uh)

    # per-kernel device times: the same step launched directly with CUDA events between
    # its kernels, queued behind a short spin kernel so launches never starve the GPU
    B.waste_moe_set_profiling(layer.handle, True)
    prof = []
    n_prof = max(8, min(K, 200))
    t_start = time.time()
    for i in range(n_prof):
        h_in.copy_(pool[i % DECODE_POOL])
        flush.zero_()
        torch.cuda._sleep(100_000)
        step()
        prof.append(B.waste_moe_read_profile(layer.handle))
    torch.cuda.synchronize()
    args.sampler.mark(t_start, time.time())
    B.waste_moe_set_profiling(layer.handle, False)

    step_bytes, gu_bytes, dn_bytes = decode_algorithmic_bytes(w)
    kern = {k: statistics.mean(p[k] for p in prof) for k in prof[0] if prof[0][k] >= 0}
    ms_per_step = total_ms / K

    # the register-reconstruct form of the expert kernels (WASTE_FLAG_K2_RECONSTRUCT: each
    # 8-weight vector rebuilt from its 3 codebook rows in shared memory, then an 8-term dot
    # product) on the same weights, per-kernel times as above
    rcfg = B.make_config(w.d, w.f, w.n_experts, w.top_k, w.act_dtype, 1, 0, B.FLAG_K2_RECONSTRUCT, layer.layer)
    rh = B.waste_moe_create(rcfg, layer.router_w, layer.router_b, layer.records, layer.stride, layer.codebooks)
    B.waste_moe_set_profiling(rh, True)
    rprof = []
    for i in range(max(8, min(K, 40))):
        h_in.copy_(pool[i % DECODE_POOL])
        flush.zero_()
        torch.cuda._sleep(100_000)
        B.waste_moe_step(rh, h_in, 1, idx, gate, logits, y, 0)
        if i >= 3:
            rprof.append(B.waste_moe_read_profile(rh))
    torch.cuda.synchronize()
    B.waste_moe_destroy(rh)
    rk = {k: statistics.mean(p[k] for p in rprof) for k in rprof[0] if rprof[0][k] >= 0}
    peak_k2, _, _ = measured_peaks()
    k2a = dict(kernels_ms=rk, steps_profiled=len(rprof),
               gate_up_gbs=gu_bytes / (rk["gate_up"] * 1e-3) / 1e9,
               gate_up_frac=gu_bytes / (rk["gate_up"] * 1e-3) / 1e9 / peak_k2,
               down_frac=dn_bytes / (rk["down"] * 1e-3) / 1e9 / peak_k2,
               table_form_gate_up_ms=kern.get("gate_up"), table_form_down_ms=kern.get("down"),
               table_form_experts_ms=kern.get("experts"))
    out["decode"] = dict(step_ms=ms_per_step, kernels_ms=kern, stats=st, step_bytes=step_bytes,
                         gate_up_bytes=gu_bytes, down_bytes=dn_bytes,
                         hbm_gbs_step=step_bytes / (ms_per_step * 1e-3) / 1e9,
                         median_step_ms=statistics.median(step_ms),
                         launches_per_step=len(kern), profiled_steps=n_prof, unfused_ms=unfused_ms,
                         k2a_reconstruct=k2a)

    # ---- end to end through the C ABI with host buffers: h2d copy of the token from
    # pinned memory, then route + forward with the result written by the combine straight
    # into the caller's pinned host buffer (any device-accessible pointer is an output the
    # C ABI takes) -- one graph per step
    h_host = torch.empty(1, w.d, dtype=torch.float32).pin_memory()
    y_host = torch.empty(1, w.d, dtype=torch.float32).pin_memory()
    host_pool = [p.cpu() for p in pool[:8]]

    def step_to_host():
        layer.step(h_in, 1, idx, gate, y_host, 0, logits)

    with torch.cuda.stream(side):
        for i in range(3):
            h_in.copy_(h_host, non_blocking=True)
            step_to_host()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2):
        h_in.copy_(h_host, non_blocking=True)
        step_to_host()
    for i in range(args.warmup):
        h_host.copy_(host_pool[i % 8])
        g2.replay()
    torch.cuda.synchronize()
    ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t_start = time.time()
    for i in range(K):
        torch.cuda.current_stream().synchronize()  # the host buffer is free again
        h_host.copy_(host_pool[i % 8])
        flush.zero_()
        ev2[i][0].record(stream)
        g2.replay()
        ev2[i][1].record(stream)
    torch.cuda.synchronize()
    args.sampler.mark(t_start, time.time())
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev2), args.world, dev)
    # the same loop timed by the host's clock, one step at a time: the copy of the next token
    # into the pinned buffer, the launch, and the wait for the result in host memory are all
    # inside
    torch.cuda.synchronize()
    t_w = time.perf_counter()
    for i in range(K):
        h_host.copy_(host_pool[i % 8])
        g2.replay()
        torch.cuda.current_stream().synchronize()
    wall_s = time.perf_counter() - t_w
    # the last token's result in host memory equals the same step written to device memory
    step()
    torch.cuda.synchronize()
    same = bool(torch.equal(y.cpu(), y_host))
    out["e2e"] = dict(value=args.world * K / (e2e_ms * 1e-3), unit=UNIT,
                      h2d_bytes_per_step=w.d * 4, d2h_bytes_per_step=w.d * 4,
                      output_equals_device_path=same,
                      timing="CUDA events on the stream around each step's graph (H2D copy of the token "
                             "from pinned memory, route + experts, result written into pinned host memory); "
                             "host launch cost outside",
                      wall_clock_value=args.world * K / wall_s,
                      wall_clock_timing="host clock over the whole loop, each step: host copy of the "
                                        "token into the pinned buffer, graph launch, wait for the result "
                                        "(no L2 flush)")
    out["_layer"] = layer
    out["_pool"] = pool


def run_batched(args, dev, out, name, steps):
    """Batched decode (128 tokens, Zipf popularity) or a prefill chunk (512 tokens): route +
    grouped forward over all tokens per step, from a CUDA graph; the same call with every slot
    on the lookup path (WASTE_FLAG_FORCE_GEMV) for comparison."""
    from rvq_compressed_expert_gb300 import binding as B
    from rvq_compressed_expert_gb300 import synth
    from rvq_compressed_expert_gb300.layer import MoELayer

    w = synth.WORKLOADS[name]
    T = w.tokens
    layer = MoELayer(w, seed=0, layer=0, device=dev)
    h = synth.hidden(0, T, w.d, w.act_dtype, dev)
    idx, gate, logits, y = layer.alloc_outputs(T)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def timed(handle, K):
        def step():
            B.waste_moe_step(handle, h, T, idx, gate, logits, y, 0)
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(3):
                step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            flush.zero_()
            g.replay()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        t0 = time.time()
        for i in range(K):
            flush.zero_()
            ev[i][0].record(stream)
            g.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        args.sampler.mark(t0, time.time())
        del g
        return sum(a.elapsed_time(b) for a, b in ev) / K

    layer.reset_stats()
    ms = timed(layer.handle, steps)
    st = {k: v / (steps + 6) for k, v in layer.stats().items()}
    # per-kernel times, launched directly with events between the phases
    B.waste_moe_set_profiling(layer.handle, True)
    prof = []
    for _ in range(5):
        flush.zero_()
        torch.cuda._sleep(100_000)
        B.waste_moe_step(layer.handle, h, T, idx, gate, logits, y, 0)
        prof.append(B.waste_moe_read_profile(layer.handle))
    B.waste_moe_set_profiling(layer.handle, False)
    kern = {k: statistics.mean(p[k] for p in prof) for k in prof[0] if prof[0][k] >= 0}
    counts = torch.bincount(idx.flatten().long(), minlength=w.n_experts).cpu()
    n_distinct = int((counts > 0).sum())
    n_tc = int((counts >= 4).sum())
    # lookup-only comparison on a second handle over the same weights
    gcfg = B.make_config(w.d, w.f, w.n_experts, w.top_k, w.act_dtype, T, 0, B.FLAG_FORCE_GEMV, 0)
    gh = B.waste_moe_create(gcfg, layer.router_w, layer.router_b, layer.records, layer.stride,
                            layer.codebooks)
    ms_gemv = timed(gh, 3)
    B.waste_moe_destroy(gh)

    per_expert = expert_code_bytes(w.d, w.f) + 3 * 3 * 256 * 8 * 4
    alg_bytes = n_distinct * per_expert + w.n_experts * w.d * 4 + T * w.d * (2 + 4)
    flops = T * w.top_k * 3 * 2 * w.d * w.f
    peak_gbs, _, pk = measured_peaks()
    # fp16 operands run at the bf16 dense rate (nominal ratio 1:1).  A step lasts milliseconds
    # and is replayed back to back, so the sustained figure is its peak; the burst one is
    # reported beside it
    peak_tf = float(pk["bf16_tflops_sustained"]) if pk else 1700.0
    peak_tf_burst = float(pk["bf16_tflops"]) if pk else 1900.0
    out[name] = dict(
        workload=f"{name}: d={w.d} f={w.f} E={w.n_experts} top-{w.top_k}, T={T} tokens/step, "
                 f"{w.act_dtype} h, router bias {w.bias}",
        tok_s=T / (ms * 1e-3), ms_per_step=ms, steps=steps,
        kernels_ms=kern,
        distinct_experts=n_distinct, tensor_core_experts=n_tc,
        tokens_per_expert_max=int(counts.max()), tokens_per_expert_mean=float(counts[counts > 0].float().mean()),
        algorithmic_bytes_per_step=alg_bytes,
        hbm_frac_whole_step=alg_bytes / (ms * 1e-3) / 1e9 / peak_gbs,
        tflops_whole_step=flops / (ms * 1e-3) / 1e12,
        tensor_frac_whole_step=flops / (ms * 1e-3) / 1e12 / peak_tf,
        tensor_peak="bf16_tflops_sustained of MEASURED_PEAKS.json" if pk else "fallback 1.7 PFLOP/s sustained",
        tensor_frac_whole_step_of_burst=flops / (ms * 1e-3) / 1e12 / peak_tf_burst,
        lookup_only_ms_per_step=ms_gemv, speedup_over_lookup_only=ms_gemv / ms,
        demand_code_bytes_per_step=st["demand_code_bytes"],
    )
    layer.close()


def run_stack(args, dev, out, w=None, key="stack"):
    """92 layers x 64 experts, one token, h += combine per layer; lookahead 6 vs off.  With w and
    key: another stack workload reported under key."""
    from rvq_compressed_expert_gb300 import binding as B
    from rvq_compressed_expert_gb300 import synth
    from rvq_compressed_expert_gb300.layer import MoELayer
    from rvq_compressed_expert_gb300.stack import DecodeStack

    w = w or synth.WORKLOADS["stack"]
    free, _ = torch.cuda.mem_get_info()
    need = w.n_layers * w.n_experts * 12_390_400 * 1.05 + (4 << 30)
    if free < need:
        out[key] = {"skipped": f"needs {need / 1e9:.0f} GB free, {free / 1e9:.0f} GB available"}
        return
    layers = [MoELayer(w, seed=0, layer=L, device=dev, max_tokens=1) for L in range(w.n_layers)]
    h0 = synth.hidden(7, 1, w.d, "f32", dev)
    stack = DecodeStack(layers, 1, dev)
    main = torch.cuda.Stream(device=dev)
    side = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    res, final, errors = {}, {}, []
    for P in (0, w.lookahead):
        main.wait_stream(torch.cuda.current_stream())
        for _ in range(2):
            stack.run(h0, P, main, side)  # warm-up outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=main):
            last = stack.run(h0, P, main, side)
        torch.cuda.synchronize()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        for L in layers:
            L.reset_stats()
        n = max(5, min(args.steps, 50))
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        cs = torch.cuda.current_stream()
        t_start = time.time()
        for i in range(n):
            flush.zero_()
            evs[i][0].record(cs)
            g.replay()
            evs[i][1].record(cs)
        torch.cuda.synchronize()
        args.sampler.mark(t_start, time.time())
        ms = sum(a.elapsed_time(b) for a, b in evs) / n
        sts = []
        for i, L in enumerate(layers):
            try:
                sts.append(L.stats())
            except B.WasteError as e:
                errors.append(f"lookahead {P}, layer {i}: {e}")
                L.reset_stats()
                sts.append(L.stats())
        final[P] = last.clone()
        res[P] = dict(
            ms_per_token=ms, tok_s=1e3 / ms,
            demand_code_bytes_per_token=sum(s["demand_code_bytes"] for s in sts) / n,
            prefetch_bytes_per_token=sum(s["prefetch_issued_bytes"] for s in sts) / n,
            prediction_hits_per_token=sum(s["prediction_hits"] for s in sts) / n)
        del g
    on, off = res[w.lookahead], res[0]
    out[key] = dict(
        workload=f"{w.n_layers} layers x {w.n_experts} experts, d={w.d} f={w.f} top-{w.top_k}, T=1, fp32, "
                 f"router bias {w.bias}, h += combine per layer; CUDA graph per token; L2 flushed between tokens",
        lookahead_form="inside the step (waste_moe_set_lookahead): layer L+1's router rows on layer L's "
                       "router launch, its top-P selected and prefetched by layer L's expert kernel",
        tok_s_lookahead_off=off["tok_s"], tok_s_lookahead_on=on["tok_s"],
        lookahead_speedup=on["tok_s"] / off["tok_s"],
        outputs_bit_identical=bool(torch.equal(final[0], final[w.lookahead])),
        demand_code_bytes_equal=on["demand_code_bytes_per_token"] == off["demand_code_bytes_per_token"],
        demand_code_bytes_per_token=off["demand_code_bytes_per_token"],
        prefetch_bytes_per_token=on["prefetch_bytes_per_token"],
        prediction_accuracy=on["prediction_hits_per_token"] / ((w.n_layers - 1) * w.lookahead),
    )
    if errors:
        out[key]["device_errors"] = errors[:8]
    for L in layers:
        L.close()
    del layers
    torch.cuda.empty_cache()


def measured_link_gbs(ts) -> float:
    """The copy engines' host -> HBM rate over 64 records of the bank's pinned buffer."""
    n = min(64, ts.host.numel() // ts.stride)
    dst = torch.empty(n * ts.stride, dtype=torch.uint8, device="cuda")
    src = ts.host[:n * ts.stride]
    dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    ts_ = []
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        ts_.append(a.elapsed_time(b))
    del dst
    return n * ts.stride / (statistics.median(ts_) * 1e-3) / 1e9


def run_tiered(args, dev, out):
    """16 layers x 64 experts with their records in pinned host memory behind an HBM cache;
    one token at a time (eager: the fetch plan depends on the routing); cache sizes below,
    near and above one token's working set (16 layers x top-16 = 256 records); lookahead
    0, 6 and 16 experts into the next layer."""
    from rvq_compressed_expert_gb300 import binding as B
    from rvq_compressed_expert_gb300 import synth
    from rvq_compressed_expert_gb300.bank import TieredStack
    from rvq_compressed_expert_gb300.stack import DecodeStack

    w = synth.WORKLOADS["tiered"]
    stride = 12_390_400
    host_need = w.n_layers * w.n_experts * stride
    try:
        host_free = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError):
        host_free = None
    if host_free is not None and host_free < 2 * host_need:
        out["tiered"] = {"skipped": f"needs {2 * host_need / 1e9:.0f} GB free host memory"}
        return
    working_set = w.n_layers * w.top_k
    slot_sizes = (working_set // 2, working_set * 5 // 4, working_set * 5 // 2)
    ts = TieredStack(w, 0, w.n_layers, slot_sizes[0], dev, max_tokens=1)
    stack = DecodeStack(ts.layers, 1, dev, banked=True)
    n_warm, n_timed = 4, 16
    tokens = [synth.hidden(1000 + i, 1, w.d, "f32", dev) for i in range(n_warm + n_timed)]
    main = torch.cuda.Stream(device=dev)
    side = torch.cuda.Stream(device=dev)
    rows, finals, errors = [], {}, []
    modes = (("overlap", 0), ("serial", B.FLAG_BANK_SERIAL))
    for slots in slot_sizes:
        for P, (mode, flags) in [(p, m) for p in (0, w.lookahead, w.top_k) for m in modes]:
            ts.rebank(slots, flags)
            main.wait_stream(torch.cuda.current_stream())
            for i in range(n_warm):
                stack.run(tokens[i], P, main, side)
            torch.cuda.synchronize()
            s0 = ts.stats()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n_timed)]
            outs = []
            t_start = time.time()
            for i in range(n_timed):
                evs[i][0].record(main)
                o = stack.run(tokens[n_warm + i], P, main, side)
                evs[i][1].record(main)
                with torch.cuda.stream(main):
                    outs.append(o.clone())
            torch.cuda.synchronize()
            args.sampler.mark(t_start, time.time())
            s1 = ts.stats()
            for L, ml in enumerate(ts.layers):
                try:
                    ml.stats()
                except Exception as e:  # an expert without a slot: reported, not hidden
                    errors.append(f"slots {slots}, lookahead {P}, layer {L}: {e}")
                    ml.reset_stats()
            st = {k: s1[k] - s0[k] for k in s1}
            ms = sum(a.elapsed_time(b) for a, b in evs) / n_timed
            demand = st["demand_hits"] + st["demand_misses"]
            finals[(slots, P, mode)] = torch.stack(outs)
            rows.append(dict(
                slots=slots, cache_gb=slots * ts.stride / 1e9, lookahead=P, copy=mode,
                tok_s=1e3 / ms, ms_per_token=ms,
                demand_hit_rate=st["demand_hits"] / max(demand, 1),
                copied_gb_per_token=st["copied_bytes"] / n_timed / 1e9,
                demand_copies_per_token=st["demand_misses"] / n_timed,
                lookahead_copies_per_token=st["prefetch_copies"] / n_timed,
                link_gbs_lower_bound=st["copied_bytes"] / n_timed / (ms * 1e-3) / 1e9))
    ref = finals[(slot_sizes[0], 0, "serial")]
    link = measured_link_gbs(ts)
    for r in rows:
        r["link_bound_tok_s"] = link / r["copied_gb_per_token"] if r["copied_gb_per_token"] else None
        r["frac_of_link_bound"] = r["tok_s"] / r["link_bound_tok_s"] if r["link_bound_tok_s"] else None
    out["tiered"] = dict(
        workload=f"{w.n_layers} layers x {w.n_experts} experts (d={w.d} f={w.f} top-{w.top_k}, Zipf(1.1) "
                 f"router bias), records ({host_need / 1e9:.1f} GB) in pinned host memory, HBM cache of "
                 f"n slots; T=1, fp32, h += combine per layer; eager; {n_warm} warm-up then {n_timed} "
                 f"timed tokens per row from an empty cache; per-token working set {working_set} records "
                 f"({working_set * ts.stride / 1e9:.2f} GB), larger than L2",
        link_gbs=link,
        link_note="host->HBM copy rate of the copy engines (cudaMemcpyAsync of 64 records from the same "
                  "pinned buffer into HBM), measured here: the bound of every row",
        rows=rows,
        outputs_bit_identical=all(torch.equal(v, ref) for v in finals.values()),
    )
    if errors:
        out["tiered"]["device_errors"] = errors[:8]
    ts.close()
    del stack, finals, ref
    torch.cuda.empty_cache()


def run_encoder(args, dev, out):
    """RVQ encoder on one expert of the decode shape (gate and up 1536 x 7168, down 7168 x 1536),
    8 Lloyd rounds per stage; then the encoded expert through the expert kernels against the
    dense expert on one token."""
    from rvq_compressed_expert_gb300 import binding as B
    from rvq_compressed_expert_gb300 import synth
    from rvq_compressed_expert_gb300.layer import MoELayer

    d, f, iters = 7168, 1536, 8
    shapes = [(f, d), (f, d), (d, f)]
    Ws, codes, cbs, mats = [], [], [], []
    total_ms, pairs = 0.0, 0
    for k, (rows, cols) in enumerate(shapes):
        W = synth.dense_matrix(20, 0, 0, k, rows, cols, dev)
        n = rows * cols // 8
        init = synth.rvq_init(21 + k, n, dev)
        cb = torch.empty(3, 256, 8, device=dev)
        c = torch.empty(rows, 3, cols // 8, dtype=torch.uint8, device=dev)
        err = torch.empty(3, dtype=torch.float64, device=dev)
        B.waste_rvq_train(W, init, 1, cb, c, err)  # warm-up (allocation paths, module load)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_start = time.time()
        a.record()
        B.waste_rvq_train(W, init, iters, cb, c, err)
        b.record()
        torch.cuda.synchronize()
        args.sampler.mark(t_start, time.time())
        ms = a.elapsed_time(b)
        total_ms += ms
        pairs += n * 256 * 3 * (iters + 1)
        norm2 = float((W.double() ** 2).sum())
        mats.append(dict(shape=[rows, cols], ms=ms,
                         rel_rmse_after_stage=[math.sqrt(float(e) / norm2) for e in err.cpu().tolist()]))
        Ws.append(W)
        codes.append(c)
        cbs.append(cb)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    clock_hz = 2.07e9
    peak_ops = sms * 128 * clock_hz  # fp32 lane operations per second (adds and fused multiply-adds)
    ops = pairs * 16.0  # 8 subtractions + 8 fused multiply-adds per vector and centroid
    # the encoded expert through the expert kernels, one token, against the dense expert
    w = synth.Workload("encoded", d, f, 1, 1, 1, "f32", "none")
    li = synth.layer_inputs(w, 0, 0, dev, with_codes=False)
    li = synth.LayerInputs(li.router_w, li.router_b, torch.stack(cbs).unsqueeze(0).contiguous(), tuple(codes))
    layer = MoELayer(w, 0, 0, dev, inputs=li)
    x = synth.hidden(22, 1, d, "f32", dev)
    y = torch.empty(1, d, device=dev)
    layer.forward(x, 1, torch.zeros(1, 1, dtype=torch.int32, device=dev), torch.ones(1, 1, device=dev), y)
    torch.cuda.synchronize()
    xd = x[0].double()
    zg, zu = Ws[0].double() @ xd, Ws[1].double() @ xd
    yd = Ws[2].double() @ (zg / (1 + torch.exp(-zg)) * zu)
    rel = float(torch.linalg.norm(y[0].double() - yd) / torch.linalg.norm(yd))
    layer.close()
    out["encoder"] = dict(
        workload=f"one expert of the decode shape (gate, up {f}x{d}; down {d}x{f}), dense weights "
                 f"N(0, 0.02^2); greedy residual k-means, 3 stages x 256 centroids, {iters} Lloyd rounds "
                 f"per stage, centroids started on seeded vectors",
        ms_per_expert=total_ms, matrices=mats,
        vector_centroid_pairs_per_s=pairs / (total_ms * 1e-3),
        roofline={"bound": "alu", "achieved": ops / (total_ms * 1e-3) / 1e9, "peak": peak_ops / 1e9,
                  "unit": "Gop/s", "frac": ops / (total_ms * 1e-3) / peak_ops,
                  "note": "fp32 lane operations (8 adds + 8 fused multiply-adds per vector and centroid) against "
                          f"{sms} SMs x 128 fp32 lanes x 2.07 GHz"},
        encoded_expert_output_rel_err_vs_dense=rel,
    )
    del Ws, codes, cbs
    torch.cuda.empty_cache()


def cpu_baseline_decode(layer, pool, budget_s=12.0):
    """The oracle (single-threaded C, double) on a bounded sample of decode tokens."""
    import oracle
    w = layer.w
    Wr = layer.router_w.cpu()
    b = layer.router_b.cpu()
    cbs = layer.codebooks.cpu().numpy()
    done, spent = 0, 0.0
    while done < 1 or (spent < budget_s and done < len(pool)):
        h = pool[done].cpu()[0]
        logits = oracle.router(Wr, b, h)
        idx, _ = oracle.topk_softmax(logits, w.top_k)
        codes = {int(e): layer.expert_codes_host(int(e)) for e in idx}
        t0 = time.perf_counter()
        oracle.moe_token(h, Wr, b, cbs, lambda e: codes[int(e)], w.top_k)
        spent += time.perf_counter() - t0
        done += 1
    return dict(value=done / spent, unit=UNIT, cores=1, kind="oracle",
                sample=f"{done} decode tokens (full layer each: router over 384 experts, top-16, "
                       f"16 expert FFNs from codes, combine), single-threaded C oracle",
                host=host_description())


def _oracle_worker(job):
    """One process of the parallel CPU baseline: the single-threaded oracle on up to n decode
    tokens of a layer drawn on the CPU (the same shapes and distributions); only the oracle's
    own call is timed.  Returns (tokens, seconds)."""
    seed0, n = job
    import oracle
    from rvq_compressed_expert_gb300 import synth
    w = synth.WORKLOADS["decode"]
    li = synth.layer_inputs(w, 0, 0, "cpu", with_codes=False)
    cbs = li.codebooks.numpy()
    done, spent = 0, 0.0
    for i in range(n):
        h = synth.hidden(seed0 + i, 1, w.d, "f32", "cpu")[0]
        logits = oracle.router(li.router_w, li.router_b, h)
        idx, _ = oracle.topk_softmax(logits, w.top_k)
        codes = {int(e): synth.expert_codes(0, 0, int(e), w.d, w.f, "cpu") for e in idx}
        t0 = time.perf_counter()
        oracle.moe_token(h, li.router_w, li.router_b, cbs, lambda e: codes[int(e)], w.top_k)
        spent += time.perf_counter() - t0
        done += 1
    return done, spent


def cpu_baseline_parallel(tokens_per_proc=3):
    """The same oracle in one process per host core (spawned, so no GPU state is inherited),
    each timing its own tokens: the aggregate rate is the sum of the processes' rates."""
    import multiprocessing as mp
    n = os.cpu_count() or 1
    with mp.get_context("spawn").Pool(n) as pool:
        res = pool.map(_oracle_worker, [(5000 + 100 * i, tokens_per_proc) for i in range(n)])
    rate = sum(d / s for d, s in res if s > 0)
    return dict(value=rate, unit=UNIT, cores=n, kind="oracle",
                sample=f"{sum(d for d, _ in res)} decode tokens over {n} processes of the single-threaded "
                       f"C oracle ({tokens_per_proc} each, layer drawn on the CPU); sum of per-process rates",
                host=host_description())


def native(args):
    ws, rank, local = dist_env()
    args.world = ws
    if ws > 1:
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from rvq_compressed_expert_gb300 import _build
    from rvq_compressed_expert_gb300 import binding as B
    _build.build()
    B.load()
    args.sampler = ClockSampler(local) if rank == 0 else None
    if args.sampler is None:
        class _Null:
            def mark(self, *a):
                pass

            def stop(self):
                return {}
        args.sampler = _Null()
    res = {}
    run_decode(args, dev, res)
    # the extra legs are reported from rank 0 alone, so only rank 0 runs them (the tiered leg
    # alone pins 12.7 GB of host memory)
    if rank == 0 and not args.no_batched:
        run_batched(args, dev, res, "batched", 20)
        run_batched(args, dev, res, "prefill", 10)
    if rank == 0 and not args.no_stack:
        run_stack(args, dev, res)
        # a shorter stack whose router bias follows a weak Zipf law (s = 0.3), so the
        # lookahead's predictions miss some experts
        from rvq_compressed_expert_gb300 import synth as _s
        zw = _s.Workload("stack-zipf", 7168, 1536, 64, 16, 1, "f32", "zipf", n_layers=16, lookahead=6, zipf_s=0.3)
        run_stack(args, dev, res, zw, "stack_zipf")
    if rank == 0 and not args.no_tiered:
        run_tiered(args, dev, res)
    if rank == 0 and not args.no_encoder:
        run_encoder(args, dev, res)
    clocks = args.sampler.stop()
    cpu = cpu_par = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_decode(res["_layer"], res["_pool"])
        try:
            cpu_par = cpu_baseline_parallel()
        except Exception as e:  # the parallel line is optional; the single-core one stands
            cpu_par = {"unavailable": f"{type(e).__name__}: {e}"}
    if rank != 0:
        return
    from rvq_compressed_expert_gb300 import synth
    w = synth.WORKLOADS["decode"]
    d = res["decode"]
    peak, peak_kind, _ = measured_peaks()
    kern = d["kernels_ms"]
    if "step" in kern:  # one persistent kernel runs the whole step
        dominant, alg = "fused_step_kernel", d["step_bytes"]
        achieved = alg / (kern["step"] * 1e-3) / 1e9
        traffic = ncu_traffic("fused_step_decode")
    elif "experts" in kern:  # the gate/up and down units in one launch
        dominant, alg = "lut_experts_kernel", d["gate_up_bytes"] + d["down_bytes"]
        achieved = alg / (kern["experts"] * 1e-3) / 1e9
        traffic = ncu_traffic("lut_experts_decode")
    else:
        dominant = max(("gate_up", "down"), key=lambda k: kern[k])
        alg = d["gate_up_bytes"] if dominant == "gate_up" else d["down_bytes"]
        achieved = alg / (kern[dominant] * 1e-3) / 1e9
        traffic = ncu_traffic("lut_gate_up_decode" if dominant == "gate_up" else "lut_down_decode")
    value = ws / (d["step_ms"] * 1e-3)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": d["step_ms"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded RVQ codes, codebooks, router and tokens of the stated shapes)",
        "config": {
            "workload": "decode layer: d=7168 f=1536 E=384 experts top-16, T=1 token/step, fp32 h; "
                        "RVQ 3x256 codebooks per matrix, 8-weight vectors, 12.39 MB codes per expert",
            "step": "router GEMV + top-16 + softmax + RVQ gate/up table-lookup GEMV + SwiGLU + down "
                    "table-lookup GEMV + gate-weighted combine (waste_moe_step: "
                    f"{d['launches_per_step']} kernels: the router, its last CTA taking the top-k; "
                    + ("the gate/up and down units in one launch; " if "experts" in kern else
                       "gate/up; down; ") + "the combine) replayed from a CUDA graph",
            "l2": "flushed between steps (256 MiB write outside the per-step CUDA events); "
                  "each step also uses a different token (pool of 64)",
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
            "hbm_gbs_whole_step": d["hbm_gbs_step"],
            "hbm_frac_whole_step": d["hbm_gbs_step"] / peak,
            "hbm_frac_expert_kernels": (d["gate_up_bytes"] + d["down_bytes"])
            / ((kern["gate_up"] + kern["down"]) * 1e-3) / 1e9 / peak if "gate_up" in kern
            else (d["gate_up_bytes"] + d["down_bytes"]) / (kern["experts"] * 1e-3) / 1e9 / peak
            if "experts" in kern else None,
            "algorithmic_bytes_per_step": d["step_bytes"],
            "kernels_ms": kern,
            "ms_per_step_persistent_step_kernel": d["unfused_ms"],
            "k2a_register_reconstruct": d["k2a_reconstruct"],
        },
        "roofline": {
            "bound": "hbm",
            "kernel": dominant,
            "achieved": achieved,
            "peak": peak,
            "unit": "GB/s",
            "frac": achieved / peak,
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback 6.8 TB/s",
            "algorithmic_bytes_per_launch": alg,
            "traffic": traffic,
        },
        "e2e": res["e2e"],
        "gpu_launches": args.steps * d["launches_per_step"],
        "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples")},
        "cpu_baseline": cpu,
        "cpu_baseline_parallel": cpu_par,
        "stats_per_step": {k: v / args.steps for k, v in d["stats"].items()},
    }
    if "verify_crc" in res:
        line["config"]["create_with_crc_verify"] = res["verify_crc"]
    for extra in ("batched", "prefill", "stack", "stack_zipf", "tiered", "encoder"):
        if extra in res:
            line[extra] = res[extra]
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- reference arm (the oracle)

def reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import oracle
    from rvq_compressed_expert_gb300 import synth
    oracle.build()
    w = synth.WORKLOADS["decode"]
    li = synth.layer_inputs(w, 0, 0, "cpu", with_codes=False)
    cbs = li.codebooks.numpy()

    def one_token(i):
        h = synth.hidden(100 + i, 1, w.d, "f32", "cpu")[0]
        logits = oracle.router(li.router_w, li.router_b, h)
        idx, _ = oracle.topk_softmax(logits, w.top_k)
        codes = {int(e): synth.expert_codes(0, 0, int(e), w.d, w.f, "cpu") for e in idx}
        t0 = time.perf_counter()
        oracle.moe_token(h, li.router_w, li.router_b, cbs, lambda e: codes[int(e)], w.top_k)
        return time.perf_counter() - t0

    for i in range(min(args.warmup, 1)):
        one_token(i)
    K = args.steps if args.steps <= 20 else 20
    spent = sum(one_token(1000 + i) for i in range(K))
    value = K / spent
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": ws,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": spent / K * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "decode layer: d=7168 f=1536 E=384 experts top-16, T=1 token/step, fp32 h",
                   "parallelism": "host cores, single thread"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{K} decode tokens, one per step (capped at 20 steps)",
                         "host": host_description()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def profile_case(args):
    """Small case for ncu captures: the decode step at full d, f and top-16 over 32 resident
    experts (0.4 GB of records instead of 4.7 GB; the per-launch work is the same as the
    full decode layer).  Runs `--warmup` then `--steps` plain launches, no timing."""
    from rvq_compressed_expert_gb300 import _build
    from rvq_compressed_expert_gb300 import binding as B
    from rvq_compressed_expert_gb300 import synth
    from rvq_compressed_expert_gb300.layer import MoELayer
    _build.build()
    B.load()
    if args.prefill:
        # the grouped tensor-core path at full d and f: 64 bf16 tokens over 32 experts
        # (about 32 tokens per expert; 0.4 GB of records)
        w = synth.Workload("prefill-e32", 7168, 1536, 32, 16, 64, "bf16", "none")
    else:
        w = synth.Workload("decode-e32", 7168, 1536, 32, 16, 1, "f32", "offsets")
    flags = 0 if (args.phases or args.prefill) else B.FLAG_STEP_KERNEL
    if args.recon:
        flags = B.FLAG_K2_RECONSTRUCT
    layer = MoELayer(w, seed=0, layer=0, device="cuda", flags=flags)
    idx, gate, logits, y = layer.alloc_outputs(w.tokens)
    trace = None
    if args.trace:
        trace = torch.zeros(4096 * 4, dtype=torch.int64, device="cuda")
        B.waste_moe_set_trace(layer.handle, trace, 4096)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    for i in range(args.warmup + args.steps):
        h = synth.hidden(100 + i, w.tokens, w.d, w.act_dtype, "cuda")
        if trace is not None:
            flush.zero_()
            trace.zero_()
        layer.step(h, w.tokens, idx, gate, y, 0, logits)
        if trace is not None and i >= args.warmup:
            torch.cuda.synchronize()
            if args.phases:
                print_unit_trace(trace.view(-1, 4).cpu(), w)
            else:
                print_trace(trace.view(-1, 4).cpu(), w)
    torch.cuda.synchronize()
    layer.close()
    print("profile case done")


def profile_stack(args):
    """Small stack for ncu captures of the lookahead's DRAM bytes: 8 layers x 32 resident
    experts at d=7168, f=1536, top-16, one token per pass through the stack (eager launches),
    with the lookahead of --lookahead experts (0 = off).  The last --steps tokens are the ones
    to capture (each token: per layer rmsnorm, route, experts, combine, and with the lookahead
    the next layer's router, top-k and prefetch)."""
    from rvq_compressed_expert_gb300 import _build
    from rvq_compressed_expert_gb300 import binding as B
    from rvq_compressed_expert_gb300 import synth
    from rvq_compressed_expert_gb300.layer import MoELayer
    from rvq_compressed_expert_gb300.stack import DecodeStack
    _build.build()
    B.load()
    w = synth.Workload("stack-e32", 7168, 1536, 32, 16, 1, "f32", "offsets", n_layers=8, lookahead=6)
    layers = [MoELayer(w, seed=0, layer=L, device="cuda", max_tokens=1) for L in range(w.n_layers)]
    stack = DecodeStack(layers, 1)
    main = torch.cuda.Stream()
    side = torch.cuda.Stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    for i in range(args.warmup + args.steps):
        h = synth.hidden(200 + i, 1, w.d, "f32", "cuda")
        flush.zero_()
        main.wait_stream(torch.cuda.current_stream())
        stack.run(h, args.lookahead, main, side)
        torch.cuda.current_stream().wait_stream(main)
        torch.cuda.synchronize()
    for l in layers:
        l.stats()
        l.close()
    print("stack profile case done")


def profile_encoder():
    """One encoder training of a dense 1536 x 7168 matrix (the gate matrix of the decode shape),
    two Lloyd rounds per stage: a small case for ncu captures of the assignment kernels."""
    from rvq_compressed_expert_gb300 import _build
    from rvq_compressed_expert_gb300 import binding as B
    from rvq_compressed_expert_gb300 import synth
    _build.build()
    B.load()
    rows, cols = 1536, 7168
    W = synth.dense_matrix(20, 0, 0, 0, rows, cols, "cuda")
    init = synth.rvq_init(21, rows * cols // 8, "cuda")
    cb = torch.empty(3, 256, 8, device="cuda")
    codes = torch.empty(rows, 3, cols // 8, dtype=torch.uint8, device="cuda")
    err = torch.empty(3, dtype=torch.float64, device="cuda")
    B.waste_rvq_train(W, init, 2, cb, codes, err)
    torch.cuda.synchronize()
    print("encoder profile case: squared error after each stage", err.tolist())


def profile_route(args):
    """Small case for ncu captures of the one-token router: the decode layer's router (d=7168,
    E=384, top-16, fp32 h) over narrow experts (f=256, 0.8 GB of records), `--warmup` then
    `--steps` one-token routes, each a CUDA-graph replay after an L2 flush."""
    from rvq_compressed_expert_gb300 import _build
    from rvq_compressed_expert_gb300 import binding as B
    from rvq_compressed_expert_gb300 import synth
    from rvq_compressed_expert_gb300.layer import MoELayer
    _build.build()
    B.load()
    w = synth.Workload("route-e384", 7168, 256, 384, 16, 1, "f32", "offsets")
    layer = MoELayer(w, seed=0, layer=0, device="cuda")
    idx, gate, logits, _ = layer.alloc_outputs(1)
    h = synth.hidden(3, 1, w.d, "f32", "cuda")
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        layer.route(h, 1, idx, gate, logits)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.route(h, 1, idx, gate, logits)
    for _ in range(args.warmup + args.steps):
        flush.zero_()
        graph.replay()
    torch.cuda.synchronize()
    layer.stats()  # raises if a device wait gave up
    layer.close()
    print("route profile case done")


def print_unit_trace(tr, w):
    """Per-phase summary of the lookup kernels' unit trace: table build and row streaming."""
    import math as _m
    slots = w.tokens * w.top_k
    n_gu = slots * 2 * _m.ceil(_m.ceil(w.d / 8 / 32) / 2)  # (slot, segment pair, matrix) units
    rows = tr.tolist()
    out = []
    for name, a, b in (("gate_up", 0, n_gu), ("down", n_gu, len(rows))):
        its = [r for r in rows[a:b] if r[2] > 0]
        if not its:
            continue
        t0 = min(r[0] for r in its)
        tab = [(r[1] - r[0]) / 1e3 for r in its]
        run = [(r[2] - r[1]) / 1e3 for r in its]
        wait = [(r[3] >> 32) / 1e3 for r in its]
        span = (max(r[2] for r in its) - t0) / 1e3
        per_sm = {}
        for r in its:
            per_sm.setdefault(r[3] & 0xffffffff, []).append(r)
        busy = [sum((x[2] - x[0]) for x in v) / 1e3 for v in per_sm.values()]
        out.append(f"{name}: units={len(its)} span {span:.1f} us; to barrier mean {sum(wait)/len(wait):.2f}; "
                   f"tables mean {sum(tab)/len(tab):.2f} "
                   f"max {max(tab):.2f}; rows mean {sum(run)/len(run):.2f} max {max(run):.2f}; "
                   f"SM busy mean {sum(busy)/len(busy):.1f} max {max(busy):.1f} us over {len(per_sm)} SMs")
    live = [r for r in rows if r[2] > 0]
    if live:
        out.append(f"all units: span {(max(r[2] for r in live) - min(r[0] for r in live)) / 1e3:.1f} us")
    print(" | ".join(out))


def print_trace(tr, w):
    """Phase timeline of one step-kernel launch from its item trace."""
    import math as _m
    n_router = (w.n_experts + 3) // 4
    slots = w.tokens * w.top_k
    nseg = _m.ceil(w.d / 8 / 32)
    rows = [r for r in tr.tolist() if r[1] > 0]
    if not rows:
        print("no trace")
        return
    t0 = min(r[0] for r in rows)
    n_gu = slots * 2 * _m.ceil(nseg / 2)  # (slot, segment pair, matrix) units
    bounds = [("router", 0, n_router), ("topk", n_router, n_router + 1),
              ("gate_up", n_router + 1, n_router + 1 + n_gu)]
    dn0 = n_router + 1 + n_gu
    n_items = len(tr)
    used = [i for i in range(n_items) if tr[i][1] > 0]
    last = max(used)
    n_comb = _m.ceil(w.d / 512)
    bounds += [("down", dn0, last + 1 - n_comb), ("combine", last + 1 - n_comb, last + 1)]
    out = []
    for name, a, b in bounds:
        its = [tr[i].tolist() for i in range(a, b) if tr[i][1] > 0]
        if not its:
            continue
        st = [(x[0] - t0) / 1e3 for x in its]
        en = [(x[1] - t0) / 1e3 for x in its]
        du = [(x[1] - x[0]) / 1e3 for x in its]
        out.append(f"{name}: n={len(its)} start {min(st):.1f}-{max(st):.1f} end {min(en):.1f}-{max(en):.1f} "
                   f"dur mean {sum(du)/len(du):.2f} max {max(du):.2f} us")
    print(" | ".join(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-stack", action="store_true")
    ap.add_argument("--no-tiered", action="store_true")
    ap.add_argument("--no-encoder", action="store_true")
    ap.add_argument("--no-batched", action="store_true")
    ap.add_argument("--prefill", action="store_true",
                    help="with --profile-case: the grouped tensor-core path (64 bf16 tokens)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", action="store_true",
                    help="run a small decode case for ncu captures and exit")
    ap.add_argument("--phases", action="store_true",
                    help="with --profile-case: one kernel per phase instead of the step kernel")
    ap.add_argument("--recon", action="store_true",
                    help="with --profile-case: the register-reconstruct form of the expert kernels")
    ap.add_argument("--trace", action="store_true",
                    help="with --profile-case: print the step kernel's item timeline")
    ap.add_argument("--profile-encoder", action="store_true",
                    help="train one 1536 x 7168 matrix with the RVQ encoder (2 Lloyd rounds) for ncu and exit")
    ap.add_argument("--profile-stack", action="store_true",
                    help="pass tokens through an 8-layer stack (32 experts each) for ncu and exit")
    ap.add_argument("--lookahead", type=int, default=6, help="with --profile-stack: experts predicted per layer")
    ap.add_argument("--profile-route", action="store_true",
                    help="route one token through the decode layer's router (graph replays) for ncu and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile_case:
        profile_case(args)
        return
    if args.profile_encoder:
        profile_encoder()
        return
    if args.profile_route:
        profile_route(args)
        return
    if args.profile_stack:
        profile_stack(args)
        return
    if args.impl == "reference":
        reference(args)
    else:
        native(args)


if __name__ == "__main__":
    main()
