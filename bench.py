#!/usr/bin/env python
"""Benchmark of paged GQA split-KV decode attention on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
plan_update (host, once per step) and, for each of the workload's independent
layer pools, append_run(): the step's new tokens appended and attended in one
launch (split-KV partial kernel, + merge where a row is split; --append-mode
separate runs kv_append, then run()).  The per-layer calls are replayed from one
CUDA graph.  With 24 (or 28) independent pools the inputs of a step
are several times larger than L2, so every step reads K/V from HBM.

Default workload: 128 requests x (300 cached + 1 appended) tokens, page 16,
Hq 14 / Hkv 2 / head_dim 64, bf16, pool of 8192 pages per layer, 24 layers.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line on rank 0.  Multi-GPU runs are independent replicas (each
rank its own requests, no collective on the data path; weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "paged GQA decode: achieved HBM GB/s (% of peak); µs/layer call at 128x300 ctx"
LAYERS = {"qwen05_decode": 24, "qwen15_mixed": 28, "long_context_b1": 8, "long_context_b4": 3,
          "ragged": 4, "wide_group": 4, "prefill_chunk": 4, "tiny": 1}
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# distributed plumbing (also exercised by the gloo tests)
# ---------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank scalar (the slowest rank sets the job time)."""
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# peaks and clocks
# ---------------------------------------------------------------------------

DECODE_SOURCES = ("paged_kv_gqa_05_gb300/csrc/decode_tc.cuh", "paged_kv_gqa_05_gb300/csrc/common.cuh")
PREFILL_SOURCES = DECODE_SOURCES + ("paged_kv_gqa_05_gb300/csrc/tcgen05.cuh",
                                    "paged_kv_gqa_05_gb300/csrc/prefill_t5.cuh")
# workload -> (ncu summary under profiles/, the sources of the kernel it describes)
PROFILE_FILES = {"qwen05_decode": ("decode_tc_qwen05_decode_128x301.md", DECODE_SOURCES),
                 "long_context_b4": ("decode_tc_long_context_b4_32768.md", DECODE_SOURCES),
                 "prefill_chunk": ("prefill_t5_prefill_chunk_512x1536.md", PREFILL_SOURCES)}


def kernel_sources_hash(sources=DECODE_SOURCES) -> str:
    """Hash of a kernel's sources, with common.cuh's block of host-side launcher
    declarations left out (it does not change the compiled kernel)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, f), "rb") as fh:
            text = fh.read()
        if f.endswith("common.cuh"):
            text = re.sub(rb"// Launchers \(defined in the kernel translation units\)\..*?// Device helpers \(inline PTX\)",
                          b"", text, flags=re.S)
        h.update(text)
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None when there is
    none for this workload or the kernel source changed after it was taken."""
    if workload not in PROFILE_FILES:
        return None
    name, sources = PROFILE_FILES[workload]
    fields = {}
    try:
        with open(os.path.join(ROOT, "profiles", name)) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
    except OSError:
        return None
    if fields.get("kernel_sources_sha256_16") != kernel_sources_hash(sources):
        return None
    try:
        return int(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s"


def bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback 1.9 PFLOP/s"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed loops run
    (every GPU is queried; rows are kept for the device whose UUID torch reports)."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.proc = None
        self.path = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(device).uuid).lower().replace("gpu-", "")
        except Exception:
            self.uuid = ""

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        mine = [r for r in rows if self.uuid and self.uuid in r[0].lower()]
        if not mine and len({r[0] for r in rows}) == 1:
            mine = rows
        if not mine:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples for this GPU"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in mine if num(r[1]) is not None]
        mx = [num(r[2]) for r in mine if num(r[2]) is not None]
        reasons = set()
        for r in mine:
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                 r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(mine),
                "power_w_max": max((num(r[3]) or 0.0) for r in mine)}


# ---------------------------------------------------------------------------
# workload on the device
# ---------------------------------------------------------------------------

def build_layers(name: str, layers: int, seed: int, device: torch.device):
    """Layer 0 comes from the CPU generator (the oracle checks it in the tests);
    the other layers' pools and rows are drawn on the GPU with seeded generators."""
    from paged_kv_gqa_05_gb300 import workloads as W
    w = W.make(name, seed)
    dt = W.TORCH_DTYPES[w.dtype]
    P, ps, Hkv, D = w.k_pool.shape
    kp, vp = [w.k_pool.to(device)], [w.v_pool.to(device)]
    for l in range(1, layers):
        gen = torch.Generator(device=device).manual_seed(seed * 1000 + l)
        k, v = W.make_pools(P, ps, Hkv, D, w.dtype, w.kv_indptr, w.kv_indices, w.last_page_len, gen,
                            device=device)
        if w.slot_mapping is not None:
            s = torch.from_numpy(w.slot_mapping[w.slot_mapping >= 0]).to(device)
            k.view(-1, Hkv, D)[s] = float("nan")
            v.view(-1, Hkv, D)[s] = float("nan")
        kp.append(k)
        vp.append(v)
    rows, Hq = w.q.shape[0], w.q.shape[1]
    T = 0 if w.k_new is None else w.k_new.shape[0]
    # per-step inputs of all layers in one contiguous buffer (one H2D copy for the e2e leg)
    q_elems, kv_elems = rows * Hq * D, T * Hkv * D
    per_layer = q_elems + 2 * kv_elems
    inputs = torch.empty(layers * per_layer, dtype=dt, device=device)
    gen = torch.Generator(device=device).manual_seed(seed * 1000 + 999)
    inputs.copy_(torch.randn(inputs.shape, generator=gen, device=device).to(dt))
    def views(buf):
        """Per-layer q, k_new, v_new views of one step's input buffer."""
        q, kn, vn = [], [], []
        for l in range(layers):
            base = l * per_layer
            q.append(buf[base:base + q_elems].view(rows, Hq, D))
            kn.append(buf[base + q_elems:base + q_elems + kv_elems].view(T, Hkv, D))
            vn.append(buf[base + q_elems + kv_elems:base + per_layer].view(T, Hkv, D))
        return q, kn, vn

    q, kn, vn = views(inputs)
    q[0].copy_(w.q.to(device))
    if T:
        kn[0].copy_(w.k_new.to(device))
        vn[0].copy_(w.v_new.to(device))
    out = torch.empty(layers, rows, Hq, D, dtype=dt, device=device)
    return dict(w=w, k_pool=kp, v_pool=vp, q=q, k_new=kn, v_new=vn, inputs=inputs, out=out, views=views,
                kv_indices=torch.from_numpy(w.kv_indices).to(device),
                slots=None if w.slot_mapping is None else torch.from_numpy(w.slot_mapping).to(device))


def step_bytes(w, layers: int) -> dict:
    from paged_kv_gqa_05_gb300 import workloads as W
    a = W.algorithmic_bytes(w, out_elem_bytes=2)
    append = 0
    if w.k_new is not None:
        n = int((w.slot_mapping >= 0).sum())
        append = n * 2 * w.num_kv_heads * w.head_dim * 2 * 2 + 8 * len(w.slot_mapping)  # read rows + write slots
    return {"attention_per_layer": a["total"], "append_per_layer": append,
            "per_step": layers * (a["total"] + append), "kv_whole_pages_per_layer": a["kv_whole_pages"]}


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------

def run_ours(args, rank, world, local):
    import paged_kv_gqa_05_gb300 as pg
    from paged_kv_gqa_05_gb300 import workloads as W
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(world, "nccl")
    layers = LAYERS[args.workload]
    L = build_layers(args.workload, layers, seed=args.seed + rank, device=device)
    w = L["w"]
    dt = L["q"][0].dtype
    plan = pg.Plan(w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, dt, max_batch=w.batch,
                   max_q_rows=w.rows, max_splits=args.max_splits, split_tokens=args.split_tokens,
                   ctas_per_sm=args.ctas_per_sm, decode_kernel=args.decode_kernel,
                   pipeline_stages=args.stages,
                   rope_theta=args.rope_theta, rope_max_position=int(w.kv_lens.max()) if args.rope_theta > 0 else 0,
                   prefill_kernel=args.prefill_kernel, prefill_splits=args.prefill_splits)
    stream = torch.cuda.Stream(device)
    positions = (torch.from_numpy(W.row_positions(w)).to(device)
                 if args.rope_theta > 0 and L["slots"] is not None else None)
    launches_per_layer = {}

    def update_plan():
        plan.update(w.kv_indptr, w.last_page_len, L["kv_indices"], w.num_pages, qo_indptr=w.qo_indptr,
                    causal=w.causal, stream=stream)

    fused = args.append_mode == "fused" and L["slots"] is not None

    def layer_calls(with_append=True):
        for l in range(layers):
            if fused and with_append:
                # one launch: the step's new rows are appended and attended together; the
                # pool rows it reads were written by earlier steps (no in-flight writer)
                pg.append_run(plan.handle, L["k_new"][l], L["v_new"][l], L["q"][l], L["k_pool"][l],
                              L["v_pool"][l], out=L["out"][l], pool_stable=True, stream=stream)
                continue
            if with_append and L["slots"] is not None and positions is not None:
                plan.kv_append_rope(L["k_pool"][l], L["v_pool"][l], L["k_new"][l], L["v_new"][l], L["slots"],
                                    positions, stream=stream)
            elif with_append and L["slots"] is not None:
                pg.kv_append(L["k_pool"][l], L["v_pool"][l], L["k_new"][l], L["v_new"][l], L["slots"],
                             stream=stream)
            # a step without new rows: no kernel in flight writes the pool rows the call reads,
            # so its loads may begin before its dependency wait (the run-only graph keeps the
            # plain call)
            pg.run(plan.handle, L["q"][l], L["k_pool"][l], L["v_pool"][l], out=L["out"][l],
                   pool_stable=with_append and L["slots"] is None, stream=stream)

    with torch.cuda.stream(stream):
        update_plan()
        layer_calls()  # eager warm-up: loads modules, sets kernel attributes, builds TMA maps
    torch.cuda.synchronize()
    info = plan.info()
    per_layer_launches = ((1 if (L["slots"] is not None and not fused) else 0) + 1 +
                          (1 if info["num_merge_tasks"] else 0))

    graphs = {}
    if not args.no_graph:
        for key, with_append in (("step", True), ("run_only", False)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                layer_calls(with_append)
            graphs[key] = g
        torch.cuda.synchronize()

    def replay(key, with_append=True):
        if graphs:
            graphs[key].replay()
        else:
            layer_calls(with_append)

    def step():
        update_plan()
        replay("step")

    # e2e: pinned host copies of every step's inputs in and outputs out.  With graphs the
    # steps are double-buffered, as a serving loop runs them: while step s computes on one
    # set of device buffers, step s + 1's inputs go up into the other set on one copy stream
    # and step s - 1's outputs come down from it on another.  The timed region holds K steps
    # plus the first step's upload and the last step's download: K + 1 copies each way.
    host_in = torch.empty(L["inputs"].shape, dtype=dt, pin_memory=True)
    host_in.copy_(L["inputs"])
    host_out = torch.empty(L["out"].shape, dtype=dt, pin_memory=True)
    h2d, d2h = torch.cuda.Stream(device), torch.cuda.Stream(device)
    inputs2, out2 = torch.empty_like(L["inputs"]), torch.empty_like(L["out"])
    bufsets = [(L["inputs"], L["q"], L["k_new"], L["v_new"], L["out"]), (inputs2, *L["views"](inputs2), out2)]

    def layers_on(bs):
        _, qs, kns, vns, outs = bs
        for l in range(layers):
            if fused:
                pg.append_run(plan.handle, kns[l], vns[l], qs[l], L["k_pool"][l], L["v_pool"][l], out=outs[l],
                              pool_stable=True, stream=stream)
                continue
            if L["slots"] is not None and positions is not None:
                plan.kv_append_rope(L["k_pool"][l], L["v_pool"][l], kns[l], vns[l], L["slots"], positions,
                                    stream=stream)
            elif L["slots"] is not None:
                pg.kv_append(L["k_pool"][l], L["v_pool"][l], kns[l], vns[l], L["slots"], stream=stream)
            pg.run(plan.handle, qs[l], L["k_pool"][l], L["v_pool"][l], out=outs[l],
                   pool_stable=L["slots"] is None, stream=stream)

    def e2e_calls(b):
        fork = torch.cuda.Event()
        fork.record(stream)
        h2d.wait_event(fork)
        d2h.wait_event(fork)
        with torch.cuda.stream(h2d):
            bufsets[1 - b][0].copy_(host_in, non_blocking=True)   # the next step's inputs
        with torch.cuda.stream(d2h):
            host_out.copy_(bufsets[1 - b][4], non_blocking=True)  # the previous step's outputs
        layers_on(bufsets[b])
        for s in (h2d, d2h):
            join = torch.cuda.Event()
            join.record(s)
            stream.wait_event(join)

    if graphs:
        for b in (0, 1):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                e2e_calls(b)
            graphs[f"e2e{b}"] = g
        torch.cuda.synchronize()

    def e2e_run(steps):
        if graphs:
            L["inputs"].copy_(host_in, non_blocking=True)  # the first step's inputs
            for s in range(steps):
                update_plan()
                graphs[f"e2e{s % 2}"].replay()
            host_out.copy_(bufsets[(steps - 1) % 2][4], non_blocking=True)  # the last step's outputs
            return
        for _ in range(steps):
            L["inputs"].copy_(host_in, non_blocking=True)
            step()
            host_out.copy_(L["out"], non_blocking=True)

    def timed(fn, steps):
        barrier(world)
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            start.record(stream)
            for _ in range(steps):
                fn()
            end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return start.elapsed_time(end) / 1e3  # seconds

    # Untimed burn-in before the warm-up steps: ~0.3 s of steps brings a GPU that was idle
    # (a fresh box) to its working clocks; the first timed run on one was 11 % slow without it.
    burn_in, t_b = 0, time.perf_counter()
    with torch.cuda.stream(stream):
        while time.perf_counter() - t_b < 0.3:
            for _ in range(20):
                step()
            burn_in += 20
            torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    t_dev = max_over_ranks(timed(step, args.steps), world, device)
    run_reps = max(args.steps, 1)
    t_run = max_over_ranks(timed(lambda: replay("run_only", False), run_reps), world, device)
    with torch.cuda.stream(stream):
        e2e_run(max(2, min(args.warmup, 10)))
    e2e_steps = max(args.steps, 2)
    t_e2e = max_over_ranks(timed(lambda: e2e_run(e2e_steps), 1), world, device)
    clocks = sampler.stop()

    # host time of one plan update (validation, work list, one staged H2D copy), GPU idle
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        t0 = time.perf_counter()
        for _ in range(50):
            update_plan()
        plan_us = (time.perf_counter() - t0) / 50 * 1e6
    torch.cuda.synchronize()

    flags = pg.read_device_flags()
    if flags:
        raise RuntimeError(f"device-side check fired during the benchmark: flags={flags}")
    if torch.isnan(L["out"]).any():
        raise RuntimeError("NaN in outputs: an out-of-table read happened")

    b = step_bytes(w, layers)
    total_bytes = sum_over_ranks(b["per_step"] * args.steps, world, device)
    value = total_bytes / t_dev / 1e9
    peak, peak_src = hbm_peak()
    if per_layer_launches == 1 and not args.no_graph:
        # the decode kernel is the only launch of a layer: its average duration is the
        # timed step divided by the launches in it (append bytes are part of its work)
        per_launch_s = t_dev / (args.steps * layers)
        launch_bytes = b["attention_per_layer"] + b["append_per_layer"]
        timing_note = "timed step / launches (one decode_tc launch per layer), events on the launch stream"
    else:
        per_launch_s = t_run / (run_reps * layers)
        launch_bytes = b["attention_per_layer"]
        timing_note = "run()-only CUDA graph over the layer pools, events on the launch stream"
    achieved = launch_bytes / per_launch_s / 1e9
    # the committed counters describe the default launch of this workload only
    default_launch = (args.decode_kernel != "cuda_core" and not args.rope_theta and not args.split_tokens and
                      args.prefill_kernel == "auto" and not args.prefill_splits and
                      not args.max_splits and not args.stages and not args.ctas_per_sm)
    traffic = profiled_traffic(args.workload) if default_launch else None
    e2e_value = sum_over_ranks(b["per_step"] * e2e_steps, world, device) / t_e2e / 1e9
    if info["num_items"] == 0 and info["num_prefill_tiles"] > 0:
        # only multi-row requests: the prefill-segment kernel (a contraction) dominates
        flops = W.algorithmic_flops(w)
        tpeak, tpeak_src = bf16_peak()
        tf = flops / per_launch_s / 1e12
        roofline = {"bound": "tensor", "achieved": round(tf, 2), "peak": tpeak, "unit": "TFLOP/s",
                    "frac": round(tf / tpeak, 4), "traffic": traffic, "peak_source": tpeak_src,
                    "algorithmic_flops_per_launch": flops,
                    "kernel": ("prefill_tc_kernel" if args.prefill_kernel == "mma_sync" else "prefill_t5_kernel")
                              + (" (+ merge_kernel)" if info["num_merge_tasks"] else ""),
                    "timing": timing_note}
    else:
        roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                    "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": peak_src,
                    "algorithmic_bytes_per_launch": launch_bytes,
                    "kernel": ("decode_cuda_core" if args.decode_kernel == "cuda_core" else "decode_tc_kernel")
                              + (" (+ merge_kernel)" if info["num_merge_tasks"] else ""),
                    "timing": timing_note}

    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_dev / args.steps * 1e3, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "io_dtype": w.dtype,
        "data": "synthetic",
        "config": {
            "workload": w.name, "description": w.description, "layers": layers,
            "batch": w.batch, "q_rows": w.rows, "page_size": w.page_size,
            "num_qo_heads": w.num_qo_heads, "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "kv_tokens": int(w.kv_lens.sum()),
            "l2": f"inputs larger than L2: {layers} independent layer pools per step",
            "graph": not args.no_graph, "burn_in_steps": burn_in,
            "parallelism": "replicas" if world > 1 else "single",
            "decode_kernel": args.decode_kernel, "append_mode": args.append_mode if L["slots"] is not None else None,
            "rope_theta": args.rope_theta if args.rope_theta > 0 else None,
            "prefill_kernel": args.prefill_kernel if w.qo_indptr is not None else None,
            "plan": {k: info[k] for k in ("num_items", "num_merge_tasks", "split_tokens", "max_splits_used",
                                          "num_sms")},
        },
        "us_per_layer": round(t_dev / args.steps / layers * 1e6, 3),
        "us_per_run_call": round(t_run / (run_reps * layers) * 1e6, 3),
        "plan_update_host_us": round(plan_us, 2),
        "us_per_decode_launch": round(per_launch_s * 1e6, 3),
        "pct_of_peak": round(100.0 * value / peak, 2),
        "bytes": b,
        "roofline": roofline,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(L["inputs"].numel() * L["inputs"].element_size()),
                "d2h_bytes_per_step": int(L["out"].numel() * L["out"].element_size())},
        "gpu_launches": int(per_layer_launches * layers * args.steps),
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    plan.close()
    return result


# ---------------------------------------------------------------------------
# the CPU oracle (baseline leg and --impl reference)
# ---------------------------------------------------------------------------

def _oracle_layer(w, orc, nthreads, rows_subset=None):
    from paged_kv_gqa_05_gb300 import workloads as W
    if rows_subset is None:
        return orc.paged_attention(W.raw16(w.q), W.raw16(w.k_pool), W.raw16(w.v_pool), w.kv_indptr,
                                   w.kv_indices, w.last_page_len, w.dtype, qo_indptr=w.qo_indptr,
                                   causal=w.causal, nthreads=nthreads)
    sub = rows_subset
    return orc.paged_attention(W.raw16(w.q[sub.q_rows]), W.raw16(w.k_pool), W.raw16(w.v_pool),
                               sub.kv_indptr, sub.kv_indices, sub.last_page_len, w.dtype,
                               qo_indptr=sub.qo_indptr, causal=w.causal, nthreads=nthreads)


class _Subset:
    """The first n requests of a workload (their page table and query rows)."""

    def __init__(self, w, n):
        n = max(1, min(n, w.batch))
        self.n = n
        self.kv_indptr = w.kv_indptr[:n + 1].copy()
        self.kv_indices = w.kv_indices[:self.kv_indptr[-1]].copy()
        self.last_page_len = w.last_page_len[:n].copy()
        if w.qo_indptr is None:
            self.qo_indptr = None
            self.q_rows = slice(0, n)
        else:
            self.qo_indptr = w.qo_indptr[:n + 1].copy()
            self.q_rows = slice(0, int(self.qo_indptr[-1]))
        rows = n if w.qo_indptr is None else int(self.qo_indptr[-1])
        kv = int(w.kv_lens[:n].sum()) * 2 * w.num_kv_heads * w.head_dim * 2
        self.bytes = kv + 2 * rows * w.num_qo_heads * w.head_dim * 2 + 4 * (2 * n + 1 + len(self.kv_indices))


def cpu_baseline(w, seconds: float) -> dict:
    import oracle
    orc = oracle.get()
    cores = os.cpu_count() or 1
    sub = _Subset(w, w.batch)
    _oracle_layer(w, orc, cores, sub)  # warm
    reps, t0 = 0, time.perf_counter()
    while True:
        _oracle_layer(w, orc, cores, sub)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= 1000:
            break
    # the same oracle on one thread, over a quarter of the time
    reps1, t1 = 0, time.perf_counter()
    while True:
        _oracle_layer(w, orc, 1, sub)
        reps1 += 1
        el1 = time.perf_counter() - t1
        if el1 >= seconds / 4 or reps1 >= 1000:
            break
    return {"value": round(sub.bytes * reps / el / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"one layer of {w.name} ({sub.n} requests), fp64 oracle repeated {reps} times "
                      f"over {el:.1f} s on {cores} threads",
            "single_thread": {"value": round(sub.bytes * reps1 / el1 / 1e9, 4), "unit": "GB/s",
                              "sample": f"{reps1} repetitions over {el1:.1f} s on 1 thread"}}


def run_reference(args, rank, world):
    """--impl reference: the CPU oracle as it stands, on this arm's workload."""
    if rank != 0:
        return None
    import oracle
    from paged_kv_gqa_05_gb300 import workloads as W
    orc = oracle.get()
    w = W.make(args.workload, args.seed)
    cores = os.cpu_count() or 1
    budget = 120.0  # seconds for the whole warmup + timed run
    t0 = time.perf_counter()
    _oracle_layer(w, orc, cores, _Subset(w, 1))
    t1 = max(time.perf_counter() - t0, 1e-4)
    n = int(budget / (args.steps + args.warmup) / t1)
    sub = _Subset(w, max(1, min(w.batch, n)))
    for _ in range(args.warmup):
        _oracle_layer(w, orc, cores, sub)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_layer(w, orc, cores, sub)
    el = time.perf_counter() - t0
    value = sub.bytes * args.steps / el / 1e9
    sample = (f"{sub.n} of {w.batch} requests of one layer of {w.name} per step, fp64 oracle on "
              f"{cores} threads")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "description": w.description},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


SECONDARY_WORKLOADS = ("long_context_b1", "long_context_b4", "qwen15_mixed", "ragged", "prefill_chunk")
SECONDARY_KEYS = ("value", "unit", "ms_per_step", "us_per_layer", "us_per_run_call", "pct_of_peak", "roofline",
                  "e2e", "gpu_launches", "clocks", "steps", "warmup")


def secondary_lines(args, rank, world, local) -> dict:
    """The same measurement on the other workloads, each with its own timed region,
    roofline and clock record (the headline line stays on the 128 x 301 step)."""
    import copy
    out = {}
    for name in SECONDARY_WORKLOADS:
        a = copy.copy(args)
        a.workload = name
        a.steps = max(1, min(args.steps, 300))
        a.warmup = max(3, min(args.warmup, 10))
        a.no_cpu_baseline = True
        torch.cuda.empty_cache()
        r = run_ours(a, rank, world, local)
        line = {k: r[k] for k in SECONDARY_KEYS}
        line["config"] = {k: r["config"][k] for k in ("workload", "description", "layers", "plan")}
        out[name] = line
    torch.cuda.empty_cache()
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(LAYERS), default="qwen05_decode")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-graph", action="store_true", help="launch the layer calls eagerly")
    ap.add_argument("--split-tokens", type=int, default=0)
    ap.add_argument("--max-splits", type=int, default=0)
    ap.add_argument("--ctas-per-sm", type=int, default=0)
    ap.add_argument("--decode-kernel", choices=["auto", "tensor_core", "cuda_core"], default="auto")
    ap.add_argument("--stages", type=int, default=0, choices=[0, 1, 2, 3],
                    help="pipeline stages per warp (1: the wide form)")
    ap.add_argument("--append-mode", choices=["fused", "separate"], default="fused",
                    help="fused: pgqa_append_run per layer; separate: pgqa_kv_append then pgqa_run")
    ap.add_argument("--prefill-kernel", choices=["auto", "tcgen05", "mma_sync"], default="auto")
    ap.add_argument("--prefill-splits", type=int, default=0, help="key slices per prefill tile (0: automatic)")
    ap.add_argument("--rope-theta", type=float, default=0.0,
                    help="> 0: rotary embedding of q and the appended K rows with this base")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the per-workload lines of the other workloads (default run, N = 1 only)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local)
        if world == 1 and args.workload == "qwen05_decode" and not args.no_secondary:
            res["secondary"] = secondary_lines(args, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
