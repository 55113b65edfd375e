#!/usr/bin/env python3
"""Benchmark of the Qwen3-style Q8_0 decoder on one GB300 (or N replicas).

Default workload: the Qwen3-0.6B geometry (seed 1, tied lm_head, Q8_0
weights, f32 KV cache), a 512-token seeded prompt prefilled untimed, then K
greedy decode steps at batch 1 (K = 256 covers positions 512..767). One
step is one token through the whole path: embedding, 28 layers, final norm,
lm_head with fused argmax. The timed region is a single qw3_generate_greedy
call of K steps, timed with CUDA events on the model's stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload qwen3-0.6b-decode|qwen3-0.6b-batch64|qwen3-8b|qwen3-0.6b-prefill4096]

Prints one JSON line. `--impl reference` times the CPU oracle on the host
cores on the same workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

from quantized_transformer_decode_gb300 import inputs  # noqa: E402

METRIC = "Qwen3-0.6B-shape Q8_0 decode tok/s @B=1; achieved HBM GB/s vs peak"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ------------------------------------------------------------ byte counts

def q8_0_bytes(rows: int, cols: int) -> int:
    return rows * (cols // 32) * 34


def weight_bytes_per_step(s: inputs.Qwen3Shape) -> int:
    """Q8_0 bytes every decode step streams: all layer linears plus lm_head."""
    layer = (q8_0_bytes(s.q_width + 2 * s.kv_width, s.hidden) + q8_0_bytes(s.hidden, s.q_width)
             + q8_0_bytes(2 * s.intermediate, s.hidden) + q8_0_bytes(s.hidden, s.intermediate))
    return s.n_layers * layer + q8_0_bytes(s.vocab, s.hidden)


def kv_bytes_per_position(s: inputs.Qwen3Shape) -> int:
    """f32 K and V read per cached position, all layers."""
    return s.n_layers * 2 * s.kv_width * 4


def decode_bytes(s: inputs.Qwen3Shape, B: int, positions: list[list[int]]) -> int:
    """Algorithmic bytes of the decode steps: positions[step][b] is the
    position of the new token of sequence b; it attends over pos+1 rows."""
    w = weight_bytes_per_step(s) * len(positions)
    kv = sum((p + 1) for step in positions for p in step) * kv_bytes_per_position(s)
    return w + kv


def decode_launches_per_step(s: inputs.Qwen3Shape, B: int) -> int:
    """Kernels of one decode step (the library's own launch plan): B <= 4 rows
    with B * max(K) <= 16384 use the GEMV path (embed, 5 per layer, lm_head);
    larger batches the tiled path (embed, 7 per layer, norm + lm_head + argmax)."""
    kmax = max(s.hidden, s.intermediate, s.q_width)
    if B <= 4 and B * kmax <= 16384:
        return 2 + 5 * s.n_layers
    return 4 + 7 * s.n_layers


def prefill_flops(s: inputs.Qwen3Shape, S: int) -> float:
    lin = s.n_layers * s.hidden * (s.q_width + 2 * s.kv_width + s.q_width + 3 * s.intermediate)
    attn = 4.0 * s.head_dim * s.n_heads * s.n_layers * S * (S + 1) / 2
    return 2.0 * S * lin + attn + 2.0 * s.vocab * s.hidden


def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def profiled_traffic(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it still
    describes the current kernel (profiles/traffic.json-like line in the
    summary: `traffic <key> <bytes> <source-hash>`)."""
    f = ROOT / "profiles" / "traffic.txt"
    if not f.exists():
        return None
    import hashlib
    src = ROOT / "quantized_transformer_decode_gb300" / "csrc"
    h = hashlib.sha256()
    for cu in sorted(src.glob("*.cu*")):
        h.update(cu.read_bytes())
    digest = h.hexdigest()[:16]
    for ln in f.read_text().splitlines():
        parts = ln.split()
        if len(parts) == 4 and parts[0] == "traffic" and parts[1] == kernel_key and parts[3] == digest:
            return float(parts[2])
    return None


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in out.splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------- distributed glue

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate_max(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_sum(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------- CPU oracle

def oracle_cores():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_decode(w: inputs.Workload, n_warm: int, n_steps: int, prompt_len: int | None = None):
    """Build the oracle for the workload, prefill untimed, run n_warm untimed
    and then n_steps timed greedy decode steps; return (seconds, steps)."""
    from oracle import qw3_oracle as orc
    s = w.shape
    P = w.prompt_len if prompt_len is None else prompt_len
    om = orc.OracleModel.from_f32(s, dict((n, a) for n, _, a in inputs.iter_weights(s, w.seed)))
    cache = om.new_cache(P + n_warm + n_steps + 1)
    prompt = inputs.prompt_tokens(s, w.seed, P) if w.batch == 1 else inputs.batch_prefix_tokens(s, w.seed, 0, P)
    tok = orc.argmax_lowest(om.forward(cache, prompt, 0))
    for _ in range(n_warm):
        tok = orc.argmax_lowest(om.forward(cache, [tok], cache.len))
    t0 = time.perf_counter()
    for _ in range(n_steps):
        tok = orc.argmax_lowest(om.forward(cache, [tok], cache.len))
    return time.perf_counter() - t0, n_steps


def run_reference(a, w: inputs.Workload):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    if w.decode_steps == 0:
        print(json.dumps({"impl": "reference", "unavailable": "prefill workload has no oracle decode arm"}))
        return 0
    s = w.shape
    if s.n_layers * (s.hidden * (2 * s.q_width + 2 * s.kv_width) + 3 * s.hidden * s.intermediate) > 1e9:
        print(json.dumps({"impl": "reference", "unavailable": "the f64 oracle of a model past 1e9 weights takes "
                                                               "~10 min to build on the host; not a bounded run"}))
        return 0
    steps, warm = a.steps, a.warmup
    # Batched workloads: one sequence of the batch stands for the step's cost per token.
    P = min(w.prompt_len, 512) if w.batch > 1 else w.prompt_len
    secs, n = oracle_decode(w, warm, steps, P)
    tok_s = n / secs
    cores = oracle_cores()
    sample = (f"oracle (f64 numpy) greedy decode at B=1: prefill {P} seeded tokens untimed, {warm} untimed "
              f"steps, then {n} timed steps at positions {P + warm}..{P + warm + n - 1}")
    if w.batch > 1:
        sample += f"; one sequence of the batch-{w.batch} workload with a {P}-token prefix"
    line = {
        "impl": "reference", "metric": METRIC if w.name == "qwen3-0.6b-decode" else f"{w.name} decode tok/s",
        "value": tok_s, "unit": "tok/s", "n_gpus": a.gpus, "steps": steps, "warmup": warm,
        "ms_per_step": 1e3 * secs / n, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded random weights and prompt)",
        "config": workload_config(w, steps),
        "cpu_baseline": {"value": tok_s, "unit": "tok/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": tok_s, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def workload_config(w: inputs.Workload, steps: int) -> dict:
    s = w.shape
    cfg = {"workload": f"{w.name}: Qwen3 dense, vocab {s.vocab}, hidden {s.hidden}, {s.n_layers} layers, "
                       f"{s.n_heads}/{s.n_kv_heads} heads, head_dim {s.head_dim}, intermediate {s.intermediate}, "
                       f"{'tied' if s.tied else 'untied'} lm_head, seed {w.seed}; "
                       f"prefill {w.prompt_len} tokens untimed, then greedy decode at B={w.batch}",
           "batch": w.batch, "prompt_len": w.prompt_len, "timed_positions": [w.prompt_len, w.prompt_len + steps - 1],
           "weights": f"Q8_0, {weight_bytes_per_step(s) / 1e6:.1f} MB streamed per step", "kv_cache": "f32",
           "l2": ("inputs larger than L2 (the Q8_0 weights streamed every step exceed the 129 MB L2)"
                  if weight_bytes_per_step(s) > 129e6 else
                  "inputs smaller than L2: the weights stay L2-resident between steps (a small test case)")}
    return cfg


# ------------------------------------------------------------ GPU decode

def run_decode(a, w: inputs.Workload):
    import torch
    from quantized_transformer_decode_gb300 import build as qbuild
    from quantized_transformer_decode_gb300 import qw3

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the CPU oracle runs with --impl reference)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        qbuild.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()

    s, B, P = w.shape, w.batch, w.prompt_len
    K, W = a.steps, a.warmup
    cap = P + max(K, 1) + W + 2
    flags = qw3.QW3_FLAG_PER_KERNEL if a.per_kernel else 0
    model = qw3.Qw3Model.from_f32(s, inputs.iter_weights(s, w.seed), max_seqs=B, max_seq_len=cap,
                                  max_prefill=min(P, 4096), flags=flags)
    persistent, launches_per_step = model.decode_plan(B)
    stream = model.stream
    firsts = []
    for b in range(B):
        toks = inputs.prompt_tokens(s, w.seed, P) if B == 1 else inputs.batch_prefix_tokens(s, w.seed, b, P)
        _, am = model.prefill(b, torch.from_numpy(toks).to(dev))
        firsts.append(am)
    first = torch.cat(firsts)
    model.sync()

    # warm-up: W untimed steps (also captures the graph), then rewind
    if W > 0:
        model.generate_greedy(first, W)
        model.sync()
        for b in range(B):
            model.truncate(b, P)
    out = torch.empty((K, B), dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    clocks = ClockSampler(local).start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        qw3.qw3_generate_greedy(model.h, B, None, K, first.data_ptr(), out.data_ptr())
        ev1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    model.sync()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    ms = ev0.elapsed_time(ev1)
    ms_max = aggregate_max(ms, world, dev)
    tokens_all = aggregate_sum(float(K * B), world, dev)
    value = tokens_all / (ms_max / 1e3)

    # per-kernel durations of the last timed step from the device trace
    kernel_stats = None
    if not persistent and B == 1:
        tr = model.read_trace(4096).astype(np.int64)
        n_k = decode_launches_per_step(s, B)
        if tr.shape[0] >= 2 * n_k:
            first_rec, last_rec = tr[0:2 * n_k:2], tr[1:2 * n_k:2]
            start = first_rec[:, 1]
            end = np.maximum(first_rec[:, 4], np.where(last_rec[:, 4] > 0, last_rec[:, 4], 0))
            dur = (end - start).astype(np.float64)
            kernel_stats = dur

    positions = [[P + i] * B for i in range(K)]
    if B > 1:
        positions = [[P + i for _ in range(B)] for i in range(K)]
    alg_bytes = decode_bytes(s, B, positions)
    hbm_peak, _, peak_kind = peaks()
    achieved = alg_bytes / (ms / 1e3) / 1e9

    # e2e: host token in, host token out, one qw3_decode per step
    for b in range(B):
        model.truncate(b, P)
    h_tok = torch.empty(B, dtype=torch.int32, pin_memory=True)
    h_out = torch.empty(B, dtype=torch.int32, pin_memory=True)
    d_tok = torch.empty(B, dtype=torch.int32, device=dev)
    d_am = torch.empty(B, dtype=torch.int32, device=dev)
    h_tok.copy_(first.cpu())
    seqs = list(range(B))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(K):
            d_tok.copy_(h_tok, non_blocking=True)
            qw3.qw3_decode(model.h, B, seqs, d_tok.data_ptr(), [P + i] * B, 0, d_am.data_ptr())
            h_out.copy_(d_am, non_blocking=True)
            stream.synchronize()
            h_tok.copy_(h_out)
    e2e_s = time.perf_counter() - t0
    e2e_s = aggregate_max(e2e_s, world, dev)
    e2e_val = tokens_all / e2e_s
    e2e_ids_match = bool(torch.equal(h_out.to(dev), out[K - 1]))
    model.sync()
    del h_tok, h_out
    torch.cuda.synchronize()

    gpu_launches = launches_per_step * K
    kernel_desc = ("k_step: one persistent launch per decode step (embedding, every layer's projections, "
                   "attention, FFN, lm_head and argmax)" if persistent else
                   "decode step (per-kernel path: Q8_0 GEMVs, attention, embedding, lm_head + argmax)")
    line = {
        "metric": METRIC if w.name == "qwen3-0.6b-decode" else f"{w.name} decode tok/s",
        "value": value, "unit": "tok/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_max / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded random-init weights quantised to Q8_0, seeded prompt)",
        "config": dict(workload_config(w, K), parallelism="replicas" if world > 1 else "single GPU",
                       timing="CUDA events on the model stream around one qw3_generate_greedy call of K steps"),
        "roofline": {"bound": "hbm", "kernel": kernel_desc,
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_step": alg_bytes / K,
                     "traffic": profiled_traffic("k_step" if persistent else "decode_step")},
        "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "e2e": {"value": e2e_val, "unit": "tok/s", "h2d_bytes_per_step": 4 * B, "d2h_bytes_per_step": 4 * B,
                "how": "per step: pinned host token -> device, qw3_decode, argmax -> pinned host, stream sync",
                "ids_match_timed_run": e2e_ids_match},
        "gpu_launches": gpu_launches,
    }
    if kernel_stats is not None and B == 1:
        n_l = s.n_layers
        idx = {"embed": [0], "qkv_gemv": [1 + 5 * l for l in range(n_l)], "attention": [2 + 5 * l for l in range(n_l)],
               "o_gemv": [3 + 5 * l for l in range(n_l)], "gate_up_gemv": [4 + 5 * l for l in range(n_l)],
               "down_gemv": [5 + 5 * l for l in range(n_l)], "lm_head_argmax": [1 + 5 * n_l]}
        wb = {"qkv_gemv": q8_0_bytes(s.q_width + 2 * s.kv_width, s.hidden), "o_gemv": q8_0_bytes(s.hidden, s.q_width),
              "gate_up_gemv": q8_0_bytes(2 * s.intermediate, s.hidden), "down_gemv": q8_0_bytes(s.hidden, s.intermediate),
              "lm_head_argmax": q8_0_bytes(s.vocab, s.hidden)}
        ks = {}
        tot = float(np.sum(kernel_stats))
        for name, ii in idx.items():
            d = kernel_stats[ii]
            ent = {"launches": len(ii), "mean_us": float(np.mean(d)) / 1e3, "share": float(np.sum(d)) / tot}
            if name in wb:
                ent["gbs"] = wb[name] / (float(np.mean(d)) / 1e9) / 1e9
            ks[name] = ent
        line["kernels_last_step"] = {"source": "device %globaltimer trace of the last timed step "
                                               "(first CTA after its dependency wait to last CTA exit)",
                                     "step_us": tot / 1e3, "kernels": ks}
    if rank == 0:
        cb = None
        big = s.n_layers * (s.hidden * (2 * s.q_width + 2 * s.kv_width) + 3 * s.hidden * s.intermediate) > 1e9
        if big and not a.no_cpu_baseline:
            # not a bounded sample: building the f64 oracle of this model takes ~10 minutes on the host
            line["cpu_baseline_note"] = ("skipped for models past 1e9 weights (the oracle alone takes ~10 min to "
                                         "build); the 0.6B line carries the CPU baseline")
        elif not a.no_cpu_baseline and world >= 1:
            n_cpu = a.cpu_steps
            pre = P if B == 1 else min(P, 512)
            secs, n = oracle_decode(w, 0, n_cpu, pre)
            cb = {"value": n / secs, "unit": "tok/s", "cores": oracle_cores(), "kind": "oracle",
                  "sample": f"oracle (f64 numpy) greedy decode at B=1 after an untimed {pre}-token prefill: {n} timed "
                            f"steps"}
        line["cpu_baseline"] = cb
        print(json.dumps(line), flush=True)
    model.close()
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------- GPU prefill

def run_prefill(a, w: inputs.Workload):
    import torch
    from quantized_transformer_decode_gb300 import build as qbuild
    from quantized_transformer_decode_gb300 import qw3

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        qbuild.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    s, S = w.shape, w.prompt_len
    model = qw3.Qw3Model.from_f32(s, inputs.iter_weights(s, w.seed), max_seqs=1, max_seq_len=S + 1, max_prefill=S)
    toks = torch.from_numpy(inputs.prompt_tokens(s, w.seed, S)).to(dev)
    am = torch.empty(1, dtype=torch.int32, device=dev)
    for _ in range(a.warmup):
        model.reset(0)
        qw3.qw3_prefill(model.h, 0, toks.data_ptr(), S, 0, am.data_ptr())
    model.sync()
    clocks = ClockSampler(local).start()
    stream = model.stream
    evs = []
    for _ in range(a.steps):
        model.reset(0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        qw3.qw3_prefill(model.h, 0, toks.data_ptr(), S, 0, am.data_ptr())
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    clk = clocks.stop()
    model.sync()
    ms = sum(e0.elapsed_time(e1) for e0, e1 in evs)
    ms_max = aggregate_max(ms, world, dev)
    value = aggregate_sum(float(S * a.steps), world, dev) / (ms_max / 1e3)
    flops = prefill_flops(s, S)
    _, tf_peak, peak_kind = peaks()
    achieved = flops / (ms / a.steps / 1e3) / 1e12
    # kernels of one prefill (the library's plan): embedding, per layer 2 norms,
    # 4 activation packs + 4 tensor-core GEMMs, Q/K norm + RoPE + append,
    # causal attention; final norm + lm_head GEMV on the last row
    launches_per_step = 1 + 12 * s.n_layers + 1
    line = {"metric": f"{w.name} prefill tok/s", "value": value, "unit": "tok/s", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms_max / a.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded random-init weights quantised to Q8_0, seeded prompt)",
            "config": {"workload": f"{w.name}: one {S}-token prefill per step", "prompt_len": S,
                       "l2": "inputs larger than L2"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": tf_peak, "unit": "TFLOP/s",
                         "frac": achieved / tf_peak,
                         "peak_source": f"{peak_kind} bf16 sustained (MEASURED_PEAKS.json bf16_tflops_sustained)",
                         "note": "achieved counts the model's FLOPs (linear + causal attention + last-row lm_head); "
                                 "the GEMMs and the causal attention (chunks of 128+ rows) run as three bf16 MMAs "
                                 "per product (hi/lo split for f32 accuracy)",
                         "algorithmic_flops_per_step": flops, "traffic": None},
            "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
            "gpu_launches": launches_per_step * a.steps, "cpu_baseline": None,
            "e2e": None}
    if rank == 0:
        print(json.dumps(line), flush=True)
    model.close()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="qwen3-0.6b-decode", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--cpu-steps", type=int, default=8, help="oracle decode steps timed for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--per-kernel", action="store_true",
                    help="batch-1 decode through the per-kernel chain instead of the persistent step kernel")
    a = ap.parse_args(argv)
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = inputs.WORKLOADS[a.workload]
    if a.impl == "reference":
        return run_reference(a, w)
    if w.decode_steps == 0:
        return run_prefill(a, w)
    return run_decode(a, w)


if __name__ == "__main__":
    sys.exit(main())
