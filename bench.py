#!/usr/bin/env python3
"""Benchmark of the TokenSwift attention-side hot path on B300.

Default workload: one full speculative step of a Qwen2.5-14B-shaped model at
102400 tokens of context (48 layers, 40 query heads, 8 KV heads, head dim 128,
bf16 KV cache of 20.1 GB), every layer running the 120-row tree + n-gram
verify attention over the full cache (chunk importance fused), top-64 chunk
selection, then the gather into a 4096-token partial cache fused with the
4-row draft attention over it; then the vocabulary stage on 120 x 152064 fp32 logits (penalty 1.2
over a 1024-token window, min-p 0.1, greedy target, acceptance).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                    [--workload qwen14b-100k|qwen14b-<N>|llama8b-<N>|llama2-7b-100k] [--no-cpu-baseline]
                    [--one-stream] [--separate-select] [--separate-gather]

Prints one JSON line (rank 0).  Metric: verify-attention KV throughput
(prefix K+V bytes read by the verify pass, per second of the whole step).
Multi-GPU: N independent replicas (the step has no cross-GPU exchange);
value = total KV bytes of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tree-verify attn KV GB/s (% of HBM peak) at 100K ctx; µs/layer/spec step"
UNIT = "GB/s"


# DRAM traffic of the tcgen05 verify kernel, from one ncu capture of a
# full-size launch (dram__bytes_read.sum + dram__bytes_write.sum, one pass,
# Qwen2.5-14B shape at 102400 tokens: 751.82 + 3.73 MB for 419.43 MB of
# prefix K/V), expressed per prefix K/V byte.  It holds only for the kernel
# code it was taken on: the fingerprint below is of that code with comments and
# whitespace removed; for any other code the traffic is unknown (null).
VERIFY_TRAFFIC_PER_KV_BYTE = (751.376128 + 3.720704) / 419.430400
VERIFY_TRAFFIC_CODE_SHA1 = "f38d9cdabd162bcf6b6fcd83f711e5d624ea67f7"


def _code_fingerprint(paths) -> str:
    import hashlib
    import re
    h = hashlib.sha1()
    for p in paths:
        with open(p) as fh:
            t = fh.read()
        t = re.sub(r"/\*.*?\*/", " ", t, flags=re.S)
        t = re.sub(r"//[^\n]*", " ", t)
        h.update(" ".join(t.split()).encode())
    return h.hexdigest()


def verify_traffic(kv_bytes: float):
    csrc = os.path.join(ROOT, "long_context_attention_tree_b300", "csrc")
    if _code_fingerprint([os.path.join(csrc, "attn_tc.cu"), os.path.join(csrc, "tc_ptx.cuh")]) != VERIFY_TRAFFIC_CODE_SHA1:
        return None
    return kv_bytes * VERIFY_TRAFFIC_PER_KV_BYTE


def time_commit(step, s, reps: int = 20) -> dict:
    """ts_commit_path on layer 0 with the step's device-side result and path."""
    import long_context_attention_tree_b300 as ts
    L0 = step.layers[0]
    cfg = step.cfg
    evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(reps + 1)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(reps):
            evs[i].record(s)
            ts.ts_commit_path(L0.k, L0.v, cfg.N, step.result, step.path, stream=s)
        evs[reps].record(s)
    with torch.cuda.stream(s):
        g.replay()
        g.replay()
    s.synchronize()
    us = statistics.mean(evs[i].elapsed_time(evs[i + 1]) for i in range(reps)) * 1e3
    Lacc = int(step.result[0].item())
    nbytes = 2 * 2 * cfg.Hkv * Lacc * cfg.d * 2  # K and V rows of the path, read then written
    return {"us": us, "accepted": Lacc, "bytes": nbytes, "gbs": nbytes / us / 1e3}


def time_sampled_vocab(step, s, reps: int = 5) -> dict:
    """The vocab stage with min-p sampled targets (seeded Philox stream), one
    CUDA graph of event-separated calls on the step's inputs."""
    import long_context_attention_tree_b300 as ts
    cfg, vi = step.cfg, step.vocab_inputs
    evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(reps + 1)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(reps):
            evs[i].record(s)
            ts.ts_penalty_minp_sample_verify(vi.logits, vi.history, cfg.theta, cfg.min_p, cfg.temperature, 2024, i,
                                             vi.draft, vi.parent, vi.anchor, step.target, step.kept, step.result,
                                             step.path, stream=s)
        evs[reps].record(s)
    with torch.cuda.stream(s):
        g.replay()
        g.replay()
    s.synchronize()
    us = statistics.mean(evs[i].elapsed_time(evs[i + 1]) for i in range(reps)) * 1e3
    nbytes = vi.logits.numel() * 4
    return {"us": us, "gbs": nbytes / us / 1e3, "bytes": nbytes}


def time_verify_configs(peaks, s, reps: int = 12) -> dict:
    """The verify call on every other workload of the pages' evaluation, each on
    enough layers that consecutive calls read cold HBM: the LLaMA2-7B MHA layer
    at 102400 tokens (HBM-bound) and the LLaMA3.1-8B layer at 20K-100K
    (tensor-bound).  One CUDA graph of event-separated calls per workload,
    rotating over the layers; the first replay uploads the graph, the second is
    timed."""
    import long_context_attention_tree_b300 as ts
    from long_context_attention_tree_b300 import workloads as W
    out = {}
    l2 = 126e6
    todo = [("llama2-7b-100k", W.WORKLOADS["llama2-7b-100k"])]
    todo += [(f"llama8b-{n // 1024}k", W.WORKLOADS["llama8b-sweep"].with_N(n)) for n in W.SWEEP_N]
    for name, cfg in todo:
        n_layers = max(2, math.ceil(3 * l2 / cfg.kv_bytes_per_layer()))
        layers = [W.make_layer_inputs(cfg, i, device="cuda") for i in range(n_layers)]
        mask = torch.from_numpy(ts.ts_tree_mask_from_parents(cfg.parents).view(np.int64)).cuda()
        ws = torch.empty(max(16, ts.ts_tree_attn_workspace_bytes(cfg.T, cfg.Hq, cfg.Hkv, cfg.d, cfg.N)),
                         dtype=torch.uint8, device="cuda")
        o = torch.empty((cfg.T, cfg.Hq, cfg.d), dtype=torch.bfloat16, device="cuda")
        sc = torch.empty((cfg.Hkv, cfg.n_chunks), dtype=torch.float32, device="cuda")
        evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(reps + 1)]
        with torch.cuda.stream(s):
            for x in layers:  # warm-up outside the graph (kernel attributes)
                ts.ts_tree_attn(x.q, x.k, x.v, cfg.N, mask, o, chunk_scores=sc, workspace=ws,
                                scale=cfg.scale, stream=s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(reps):
                x = layers[i % n_layers]
                evs[i].record(s)
                ts.ts_tree_attn(x.q, x.k, x.v, cfg.N, mask, o, chunk_scores=sc, workspace=ws,
                                scale=cfg.scale, stream=s)
            evs[reps].record(s)
        with torch.cuda.stream(s):
            g.replay()
            g.replay()
        s.synchronize()
        us = statistics.mean(evs[i].elapsed_time(evs[i + 1]) for i in range(reps)) * 1e3
        kv = cfg.kv_bytes_per_layer()
        flops = 4.0 * cfg.T * cfg.Hq * cfg.N * cfg.d
        gbs = kv / us / 1e3
        tf = flops / us / 1e6
        t_hbm = kv / (peaks["hbm"] * 1e9)
        t_tc = flops / (peaks["bf16"] * 1e12)
        bound = "hbm" if t_hbm >= t_tc else "tensor"
        out[name] = {"N": cfg.N, "Hq": cfg.Hq, "Hkv": cfg.Hkv, "T": cfg.T, "layers_rotated": n_layers,
                     "us_per_call": us, "kv_gbs": gbs, "kv_frac_of_hbm": gbs / peaks["hbm"], "tflops": tf,
                     "bound": bound,
                     "roofline_frac": (t_hbm if bound == "hbm" else t_tc) / (us * 1e-6),
                     "tensor_frac_of_burst": tf / peaks["bf16"]}
        del layers, g
        torch.cuda.empty_cache()
    return out


def workload_config(name: str):
    from long_context_attention_tree_b300 import workloads as W
    if name == "qwen14b-100k":
        return W.WORKLOADS["qwen14b-100k"]
    if name == "llama2-7b-100k":
        return W.WORKLOADS["llama2-7b-100k"]
    if name.startswith("qwen14b-"):  # the Qwen2.5-14B shape at another context length (profiling)
        N = int(name.split("-")[1].lower().replace("k", "")) * 1024 if name.lower().endswith("k") else int(name.split("-")[1])
        return W.WORKLOADS["qwen14b-100k"].with_N(N)
    if name.startswith("llama8b-"):
        N = int(name.split("-")[1].lower().replace("k", "")) * 1024 if name.lower().endswith("k") else int(name.split("-")[1])
        return W.WORKLOADS["llama8b-sweep"].with_N(N)
    raise SystemExit(f"unknown workload {name}")


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    sm_max=d.get("sm_max_mhz", 2032.0), source="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, sm_max=2032.0, source="fallback")


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [line.strip().split(", ") for line in self.f if line.strip()]
        self.f.close()
        os.unlink(self.f.name)
        return rows

    @staticmethod
    def summarize(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        reasons = set()
        for r in rows:
            if len(r) < 9:
                continue
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                 r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        pw = [float(r[3]) for r in rows if len(r) >= 9 and r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------- distributed helpers
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: float, seconds_per_rank: float, ws: int):
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    t = max_over_ranks(seconds_per_rank, ws)
    return units_per_rank * ws / t, t


# ---------------------------------------------------------------------------- CPU oracle baseline
def cpu_oracle_sample(cfg, layer_fraction_rows: float = 1.0, seed_layer: int = 0):
    """Time the fp64 oracle on one layer of the workload (host cores).

    Returns (seconds, kv_bytes_equivalent, description, threads)."""
    import oracle
    from long_context_attention_tree_b300 import workloads as W
    oracle.build()
    x = W.make_layer_inputs(cfg, seed_layer, device="cpu")
    T, Hq = cfg.T, cfg.Hq
    n_rows = T * Hq
    rows = np.arange(n_rows, dtype=np.int32)
    if layer_fraction_rows < 1.0:
        step = max(1, int(round(1 / layer_fraction_rows)))
        rows = rows[::step]
    t0 = time.perf_counter()
    oracle.tree_attn(x.q, x.k, x.v, cfg.N, cfg.parents, cfg.scale, rows=rows)
    sc = oracle.score_chunks(x.q[0], x.k, cfg.N).astype(np.float32)
    sel = oracle.select(sc, cfg.k_sel)
    B = cfg.k_sel * cfg.chunk
    kp = oracle.gather(sel, x.k, cfg.N, cfg.chunk, B + cfg.draft_rows)
    vp = oracle.gather(sel, x.v, cfg.N, cfg.chunk, B + cfg.draft_rows)
    kp[:, B:] = x.k_draft_tail
    vp[:, B:] = x.v_draft_tail
    oracle.tree_attn(x.q_draft, kp, vp, B, [-1] + list(range(cfg.draft_rows - 1)), cfg.scale)
    t_layer = time.perf_counter() - t0
    frac = rows.size / n_rows
    t_vocab = 0.0
    if cfg.vocab:
        vi = W.make_vocab_inputs(cfg.parents, cfg.vocab, cfg.window, seed=1000 * cfg.cid + 999, device="cpu")
        t1 = time.perf_counter()
        tgt, _ = oracle.penalty_minp(vi.logits.numpy(), vi.history.numpy(), cfg.theta, cfg.min_p, cfg.temperature)
        oracle.accept(vi.draft.numpy(), cfg.parents, tgt, vi.anchor)
        t_vocab = time.perf_counter() - t1
    # per-layer share of the vocab stage; verify rows scale the KV bytes
    seconds = t_layer + t_vocab / max(cfg.layers, 1)
    kv = cfg.kv_bytes_per_layer() * frac
    desc = (f"layer {seed_layer} of {cfg.layers}: verify attention on {rows.size}/{n_rows} rows, chunk scores, "
            f"top-{cfg.k_sel} selection, gather, {cfg.draft_rows}-row draft attention"
            + (f"; vocab stage ({T}x{cfg.vocab}) counted as 1/{cfg.layers} of a step" if cfg.vocab else "")
            + "; KV bytes scaled by the verify row fraction")
    return seconds, kv, desc, oracle.num_threads()


# ---------------------------------------------------------------------------- reference arm (the oracle)
def run_reference(args, ws, rank):
    if rank != 0:
        return
    cfg = workload_config(args.workload)
    import oracle
    oracle.build()
    frac = args.ref_row_fraction
    vals = []
    desc = threads = None
    for i in range(args.warmup + args.steps):
        s, kv, desc, threads = cpu_oracle_sample(cfg, frac, seed_layer=i % cfg.layers)
        if i >= args.warmup:
            vals.append((s, kv))
    secs = sum(s for s, _ in vals)
    kv = sum(k for _, k in vals)
    value = kv / secs / 1e9
    ms_per_step = secs / len(vals) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload + " (one layer per step, oracle)", "layers": cfg.layers, "N": cfg.N,
                   "Hq": cfg.Hq, "Hkv": cfg.Hkv, "d": cfg.d, "T": cfg.T},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- native arm
def run_native(args, ws, rank, local):
    import long_context_attention_tree_b300 as ts
    from long_context_attention_tree_b300.step import SpecStep
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the product path has no CPU fallback)")
    ts.lib()
    cfg = workload_config(args.workload)
    peaks = read_peaks()
    # the step computes what the method consumes: O (and the chunk scores), no log-sum-exp
    step = SpecStep(cfg, layers=args.layers, want_lse=False, fuse_gather=not args.separate_gather,
                    overlap_select=not args.one_stream, fuse_select=not args.separate_select)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()

    # warm-up
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            step.run(s)
    s.synchronize()

    # ---- timed region: one CUDA graph per timed step (the whole step: every
    # layer's verify, refresh and draft calls, then the vocab stage), replayed
    # back to back between two events on the launching stream.  The calls of a
    # layer are chained as programmatic dependent launches, so no event sits
    # between them here; the per-call times come from a separate graph below.
    nL = step.n_layers

    def ev():
        return torch.cuda.Event(enable_timing=True, external=True)

    graphs = []
    launches0 = ts.ts_launch_count()
    for k in range(args.steps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step.run(s)
        graphs.append(g)
    launches = ts.ts_launch_count() - launches0  # kernels per replay x steps (counted at capture)
    with torch.cuda.stream(s):
        graphs[0].replay()  # first replay uploads the graph
    s.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        ev0.record(s)
        for g in graphs:
            g.replay()
        ev1.record(s)
    s.synchronize()
    dev_status = ts.ts_device_error(True)
    torch.cuda.synchronize()
    barrier(ws)
    time.sleep(0.2)
    clk = ClockSampler.summarize(clocks.stop())
    t_total = ev0.elapsed_time(ev1) / 1e3
    kv_step = step.kv_bytes_per_step()
    value_bps, t_max = aggregate(kv_step * args.steps, t_total, ws)
    ms_per_step = t_max / args.steps * 1e3

    # ---- per-call times: one more step captured with event-record nodes
    # around every call (each call timed on the stream it runs on); an event
    # node between two calls ends their programmatic overlap, so this graph
    # runs a little slower than the timed ones
    mk = {"layer": [], "vocab": None}
    gb = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gb, stream=s):
        for i in range(nL):
            e = (ev(), ev(), ev(), ev())
            e[0].record(s)
            step.run_verify(i, s)
            e[1].record(s)
            step.run_refresh(i, s)
            e[2].record(s)
            step.run_draft(i, s)
            e[3].record(s)
            mk["layer"].append(e)
        if step.vocab:
            e = (ev(), ev())
            e[0].record(s)
            step.run_vocab(s)
            e[1].record(s)
            mk["vocab"] = e
    with torch.cuda.stream(s):
        gb.replay()
        gb.replay()
    s.synchronize()
    marks = [mk]
    verify_ms = [e[0].elapsed_time(e[1]) for mk in marks for e in mk["layer"]]
    refresh_ms = [e[1].elapsed_time(e[2]) for mk in marks for e in mk["layer"]]
    draft_ms = [e[2].elapsed_time(e[3]) for mk in marks for e in mk["layer"]]
    vocab_ms = [mk["vocab"][0].elapsed_time(mk["vocab"][1]) for mk in marks if mk["vocab"] is not None]
    verify_avg_s = statistics.mean(verify_ms) / 1e3

    # ---- dominant kernel roofline: the verify attention call
    T, Hq, d, N = cfg.T, cfg.Hq, cfg.d, cfg.N
    flops = 4.0 * T * Hq * N * d
    kv_layer = cfg.kv_bytes_per_layer()
    tensor_path = ts.ts_tree_attn_uses_tensor_cores(T, Hq, cfg.Hkv, d, N)
    if tensor_path:
        # The verify kernel runs at the full SM clock (about 600 W, far below the
        # power cap) inside a timed region well under a second, so the burst
        # cuBLAS peak is its denominator; the sustained figure (measured at a
        # power-capped ~1155 MHz) is reported beside it.
        achieved = flops / verify_avg_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16"],
                "unit": "TFLOP/s", "peak_source": f"bf16 burst, {peaks['source']}",
                "peak_sustained": peaks["bf16_sus"], "frac_of_sustained": achieved / peaks["bf16_sus"]}
    else:
        # CUDA-core fp32 FMA path: 148 SMs x 128 lanes x 2 flop x max SM clock
        alu_peak = 148 * 128 * 2 * peaks["sm_max"] * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": flops / verify_avg_s / 1e12, "peak": alu_peak, "unit": "TFLOP/s",
                "peak_source": "fp32 FMA: 148 SMs x 128 lanes x 2 flop x 2032 MHz"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = verify_traffic(kv_layer) if tensor_path else None
    roof["kernel"] = "ts_tree_attn (verify, T=%d)" % T
    roof["algorithmic_per_launch"] = {"kv_bytes": kv_layer, "flops": flops}
    roof["verify_us_per_layer"] = verify_avg_s * 1e6
    roof["verify_kv_gbs"] = kv_layer / verify_avg_s / 1e9
    roof["verify_kv_frac_of_hbm"] = kv_layer / verify_avg_s / 1e9 / peaks["hbm"]

    # ---- every row of the step, timed the same way (algorithmic bytes per call)
    B, Td = step.B, step.Td
    refresh_s = statistics.mean(refresh_ms) / 1e3
    draft_s = statistics.mean(draft_ms) / 1e3
    gather_bytes = 4 * cfg.Hkv * B * d * 2           # selected K and V chunks read, then written
    draft_bytes = 2 * cfg.Hkv * (B + Td) * d * 2     # partial-cache K and V
    draft_flops = 4.0 * Td * Hq * (B + Td) * d
    kernels = {
        "verify": {"us": verify_avg_s * 1e6, "kv_gbs": kv_layer / verify_avg_s / 1e9,
                   "tflops": flops / verify_avg_s / 1e12},
    }
    if step.fuse_select:
        # selection, gather and drafting pass in one kernel (the selected K/V
        # read once, written once into the compact cache)
        fused_bytes = gather_bytes + 2 * cfg.Hkv * Td * d * 2
        t = refresh_s + draft_s
        kernels["select_gather_draft_attention"] = {"us": t * 1e6, "gbs": fused_bytes / t / 1e9,
                                                    "bytes": fused_bytes, "tflops": draft_flops / t / 1e12}
    elif step.fuse_gather:
        # selection alone, then the gather fused with the drafting pass (the
        # selected K/V read once, written once into the compact cache)
        fused_bytes = gather_bytes + 2 * cfg.Hkv * Td * d * 2
        kernels["select"] = {"us": refresh_s * 1e6}
        kernels["gather_draft_attention"] = {"us": draft_s * 1e6, "gbs": fused_bytes / draft_s / 1e9,
                                             "bytes": fused_bytes, "tflops": draft_flops / draft_s / 1e12}
    else:
        kernels["select_gather"] = {"us": refresh_s * 1e6, "gbs": gather_bytes / refresh_s / 1e9,
                                    "bytes": gather_bytes}
        kernels["draft_attention"] = {"us": draft_s * 1e6, "gbs": draft_bytes / draft_s / 1e9, "bytes": draft_bytes,
                                      "tflops": draft_flops / draft_s / 1e12}
    if vocab_ms:
        vocab_s = statistics.mean(vocab_ms) / 1e3
        vbytes = T * cfg.vocab * 4
        kernels["penalty_minp_verify"] = {"us": vocab_s * 1e6, "gbs": vbytes / vocab_s / 1e9, "bytes": vbytes}

    # ---- next row: commit of the accepted path into layer 0's cache (after the
    # timed region; moves the rows the last vocab stage accepted), one CUDA graph
    # of event-separated calls
    if step.vocab:
        kernels["commit_path"] = time_commit(step, s)
        kernels["penalty_minp_sample_verify"] = time_sampled_vocab(step, s)

    # ---- end to end through the public API with host buffers
    e2e = run_e2e(step, s, args, ws)

    # ---- the verify call on the other workloads (MHA 100K, LLaMA3.1-8B sweep)
    configs = None
    if rank == 0 and not args.no_configs:
        configs = time_verify_configs(peaks, s)

    # ---- CPU oracle baseline (rank 0, one GPU only)
    cpu = None
    if ws == 1 and rank == 0 and not args.no_cpu_baseline:
        secs, kv, desc, threads = cpu_oracle_sample(cfg, args.cpu_row_fraction)
        cpu = {"value": kv / secs / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc,
               "seconds": secs}

    if rank == 0:
        value = value_bps / 1e9
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "model_shape": cfg.name, "layers": step.n_layers, "N": N,
                       "Hq": Hq, "Hkv": cfg.Hkv, "d": d, "T_verify": T, "tree": list(cfg.branching),
                       "ngram_chains": cfg.n_chains, "budget": cfg.budget, "draft_rows": cfg.draft_rows,
                       "vocab": cfg.vocab, "parallelism": f"replicas{ws}",
                       "l2": f"inputs larger than L2 ({kv_step / 1e9:.1f} GB of KV per step)"},
            "us_per_layer_step": ms_per_step * 1e3 / step.n_layers,
            "kv_frac_of_hbm_peak": value / ws / peaks["hbm"],
            "kv_frac_of_hbm_nominal_8tbs": value / ws / 8000.0,
            "roofline": roof,
            "kernels": kernels,
            "configs": configs,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "timing": "each timed step is one CUDA graph replay between two events; the per-call times in "
                      "'kernels' come from one more replay with event nodes between the calls",
            "device_status": dev_status,
            "clocks": clk,
            "peaks": peaks,
        }
        print(json.dumps(line), flush=True)


def copy_rows_h2d(dst, src, stream) -> None:
    """dst: a CUDA view [H][rows][d] whose rows are contiguous within each H
    (as the batch's own rows of a [Hkv][ld][d] cache are); src: the same
    shape, contiguous, in pinned host memory.  One 2-D DMA copy, no kernel."""
    from cuda.bindings import runtime as rt
    width = dst.shape[1] * dst.shape[2] * dst.element_size()
    err, = rt.cudaMemcpy2DAsync(dst.data_ptr(), dst.stride(0) * dst.element_size(), src.data_ptr(), width, width,
                                dst.shape[0], rt.cudaMemcpyKind.cudaMemcpyHostToDevice, stream.cuda_stream)
    if err != rt.cudaError_t.cudaSuccess:
        raise RuntimeError(f"cudaMemcpy2DAsync: {err}")


def run_e2e(step, s, args, ws):
    """Same metric through the public API with host buffers: every step copies
    that step's inputs (per-layer Q, the batch's own K/V rows, draft Q and the
    draft rows' own K/V; logits, history, drafts, parents) from pinned host
    memory and reads the result back, all inside the timed region (the copies
    of later layers overlap earlier layers' compute).  Warmed up eagerly, then
    timed as one CUDA graph per step."""
    cfg = step.cfg
    N, T, B = cfg.N, cfg.T, step.B
    host = []
    h2d = 0
    for L in step.layers:
        hq = L.q.cpu().pin_memory()
        hkt = L.k[:, N:N + T].contiguous().cpu().pin_memory()
        hvt = L.v[:, N:N + T].contiguous().cpu().pin_memory()
        hqd = L.q_draft.cpu().pin_memory()
        hkd = L.k_part[:, B:].contiguous().cpu().pin_memory()
        hvd = L.v_part[:, B:].contiguous().cpu().pin_memory()
        host.append((hq, hkt, hvt, hqd, hkd, hvd))
        h2d += sum(t.numel() * t.element_size() for t in (hq, hkt, hvt, hqd, hkd, hvd))
    hv = None
    if step.vocab:
        vi = step.vocab_inputs
        hv = (vi.logits.cpu().pin_memory(), vi.history.cpu().pin_memory(), vi.draft.cpu().pin_memory(),
              vi.parent.cpu().pin_memory())
        h2d += sum(t.numel() * t.element_size() for t in hv)
        out_h = torch.empty(4 + T, dtype=torch.int32).pin_memory()
    else:
        out_h = torch.empty(step.layers[-1].out.numel(), dtype=torch.bfloat16).pin_memory()
    d2h = out_h.numel() * out_h.element_size()

    # Copies run on their own stream, one layer ahead of the compute that needs
    # them: layer i's inputs land while layer i-1 computes.  A buffer is
    # refilled only after the previous step's use of it (event per layer).
    cs = torch.cuda.Stream()
    nL = len(step.layers)
    ready = [torch.cuda.Event() for _ in range(nL + 1)]  # inputs of layer i (i = nL: vocab) copied
    done = [torch.cuda.Event() for _ in range(nL + 1)]   # layer i (vocab) of the previous step finished

    def one_step(start=None):
        with torch.cuda.stream(cs):
            if start is not None:
                cs.wait_event(start)  # nothing of the timed region starts before its first event
            for i, L in enumerate(step.layers):
                hq, hkt, hvt, hqd, hkd, hvd = host[i]
                cs.wait_event(done[i])
                L.q.copy_(hq, non_blocking=True)
                copy_rows_h2d(L.k[:, N:N + T], hkt, cs)
                copy_rows_h2d(L.v[:, N:N + T], hvt, cs)
                L.q_draft.copy_(hqd, non_blocking=True)
                copy_rows_h2d(L.k_part[:, B:], hkd, cs)
                copy_rows_h2d(L.v_part[:, B:], hvd, cs)
                ready[i].record(cs)
            if step.vocab:
                vi = step.vocab_inputs
                cs.wait_event(done[nL])
                vi.logits.copy_(hv[0], non_blocking=True)
                vi.history.copy_(hv[1], non_blocking=True)
                vi.draft.copy_(hv[2], non_blocking=True)
                vi.parent.copy_(hv[3], non_blocking=True)
                ready[nL].record(cs)
        for i in range(nL):
            s.wait_event(ready[i])
            step.run_layer(i, s)
            done[i].record(s)
        if step.vocab:
            s.wait_event(ready[nL])
            step.run_vocab(s)
            out_h[:4].copy_(step.result, non_blocking=True)
            out_h[4:].copy_(step.path, non_blocking=True)
            done[nL].record(s)
        else:
            out_h.copy_(step.layers[-1].out.reshape(-1), non_blocking=True)

    with torch.cuda.stream(s):
        for _ in range(max(1, min(args.warmup, 2))):
            one_step()
    s.synchronize()
    cs.synchronize()

    # The same step captured as one CUDA graph: its memcpy nodes copy from the
    # same pinned host buffers every replay, the copy stream forking from the
    # compute stream at the start of the step and joined by the compute
    # stream's waits on the copies.  A replay starts when the previous one has
    # ended, so only the first layer's copies are not hidden.
    fork = torch.cuda.Event()

    def one_step_graphed():
        fork.record(s)
        cs.wait_event(fork)
        with torch.cuda.stream(cs):
            for i, L in enumerate(step.layers):
                hq, hkt, hvt, hqd, hkd, hvd = host[i]
                L.q.copy_(hq, non_blocking=True)
                copy_rows_h2d(L.k[:, N:N + T], hkt, cs)
                copy_rows_h2d(L.v[:, N:N + T], hvt, cs)
                L.q_draft.copy_(hqd, non_blocking=True)
                copy_rows_h2d(L.k_part[:, B:], hkd, cs)
                copy_rows_h2d(L.v_part[:, B:], hvd, cs)
                ready[i].record(cs)
            if step.vocab:
                vi = step.vocab_inputs
                vi.logits.copy_(hv[0], non_blocking=True)
                vi.history.copy_(hv[1], non_blocking=True)
                vi.draft.copy_(hv[2], non_blocking=True)
                vi.parent.copy_(hv[3], non_blocking=True)
                ready[nL].record(cs)
        for i in range(nL):
            s.wait_event(ready[i])
            step.run_layer(i, s)
        if step.vocab:
            s.wait_event(ready[nL])
            step.run_vocab(s)
            out_h[:4].copy_(step.result, non_blocking=True)
            out_h[4:].copy_(step.path, non_blocking=True)
        else:
            out_h.copy_(step.layers[-1].out.reshape(-1), non_blocking=True)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        one_step_graphed()
    with torch.cuda.stream(s):
        g.replay()
    s.synchronize()
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        for k in range(args.steps):
            g.replay()
        e1.record(s)
    s.synchronize()
    t = e0.elapsed_time(e1) / 1e3
    val, _ = aggregate(step.kv_bytes_per_step() * args.steps, t, ws)
    return {"value": val / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": t / args.steps * 1e3,
            "timing": "each step one CUDA graph replay: host->device copies of the step's inputs from pinned "
                      "memory, the step, the device->host read of its result"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="qwen14b-100k")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip timing the verify call on the other workloads")
    ap.add_argument("--layers", type=int, default=None, help="run only this many layers (profiling)")
    ap.add_argument("--one-stream", action="store_true",
                    help="run each layer's calls in order on one stream (no selection beside the verify merge)")
    ap.add_argument("--separate-select", action="store_true",
                    help="the selection as its own call before the gather-and-draft call")
    ap.add_argument("--separate-gather", action="store_true",
                    help="gather with the selection call, then the drafting attention over the compact cache")
    ap.add_argument("--cpu-row-fraction", type=float, default=1.0,
                    help="fraction of verify rows the CPU oracle baseline computes")
    ap.add_argument("--ref-row-fraction", type=float, default=1.0 / 32,
                    help="fraction of verify rows per reference-arm step")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    ws, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, ws, rank)
        else:
            run_native(args, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
