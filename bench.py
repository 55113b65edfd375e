#!/usr/bin/env python3
"""Benchmark of the Qwen3-style Q8_0 decoder on one GB300 (or N replicas).

Headline (`value`): the Qwen3-0.6B geometry (seed 1, tied lm_head, Q8_0
weights, f32 KV cache), a 512-token seeded prompt prefilled untimed, then K
greedy decode steps at batch 1 (positions 512..512+K-1; K = 256 by default).
One step is one token through the whole path: embedding, 28 layers, final
norm, lm_head with fused argmax. A timed run is one qw3_generate_greedy
call of K steps, timed with CUDA events on the model's stream; the line
reports the median of three runs (the cache is rewound between runs).

The same line carries `workloads`: the other configurations of the
benchmark, each timed the same way with its own roofline -- a 4096-token
prefill (tensor roofline), batch-64 decode over 2048-token prefixes and the
Qwen3-8B geometry at batch 1 after an 8192-token prompt (HBM roofline).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload qwen3-0.6b-decode|qwen3-0.6b-batch64|qwen3-8b|qwen3-0.6b-prefill4096]
                    [--no-workloads] [--no-cpu-baseline]

Prints one JSON line. `--impl reference` times the CPU oracle on the host
cores on the same workload and positions instead (rank 0 only).
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


def weight_bytes_per_step(s: inputs.Qwen3Shape, wtype: str = "q8_0") -> int:
    """Weight bytes every decode step streams (all layer linears plus the
    lm_head): Q8_0 34 bytes per 32 weights, Q4_K 144 per 256."""
    layer = (q8_0_bytes(s.q_width + 2 * s.kv_width, s.hidden) + q8_0_bytes(s.hidden, s.q_width)
             + q8_0_bytes(2 * s.intermediate, s.hidden) + q8_0_bytes(s.hidden, s.intermediate))
    total = s.n_layers * layer + q8_0_bytes(s.vocab, s.hidden)
    return total if wtype == "q8_0" else total // 34 * 32 // 256 * 144


def kv_bytes_per_position(s: inputs.Qwen3Shape) -> int:
    """f32 K and V read per cached position, all layers."""
    return s.n_layers * 2 * s.kv_width * 4


# bytes of a cached value relative to f32, per cache type: f32, IEEE half,
# q8_0 (34 bytes per 32 values)
KV_SCALE = {"f32": 1.0, "f16": 0.5, "q8_0": 34.0 / 128.0}


def decode_bytes(s: inputs.Qwen3Shape, B: int, positions: list[list[int]], kv: str = "f32",
                 wtype: str = "q8_0") -> int:
    """Algorithmic bytes of the decode steps: positions[step][b] is the
    position of the new token of sequence b; it attends over pos+1 rows."""
    w = weight_bytes_per_step(s, wtype) * len(positions)
    kvb = sum((p + 1) for step in positions for p in step) * kv_bytes_per_position(s) * KV_SCALE[kv]
    return int(w + kvb)


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


def _oracle_model(w: inputs.Workload, shape=None):
    from oracle import qw3_oracle as orc
    s = w.shape if shape is None else shape
    return orc.OracleModel.from_f32(s, dict((n, a) for n, _, a in inputs.iter_weights(s, w.seed)))


def oracle_decode(w: inputs.Workload, n_warm: int, n_steps: int, prompt_len: int | None = None):
    """Build the oracle for the workload, prefill untimed, run n_warm untimed
    greedy steps, rewind the cache to the prompt, then time n_steps steps
    (positions P..P+n_steps-1, the GPU arm's); return (seconds, steps)."""
    from oracle import qw3_oracle as orc
    s = w.shape
    P = w.prompt_len if prompt_len is None else prompt_len
    om = _oracle_model(w)
    cache = om.new_cache(P + max(n_warm, n_steps) + 1)
    prompt = inputs.prompt_tokens(s, w.seed, P) if w.batch == 1 else inputs.batch_prefix_tokens(s, w.seed, 0, P)
    first = orc.argmax_lowest(om.forward(cache, prompt, 0))
    tok = first
    for _ in range(n_warm):
        tok = orc.argmax_lowest(om.forward(cache, [tok], cache.len))
    cache.truncate(P)
    tok = first
    t0 = time.perf_counter()
    for _ in range(n_steps):
        tok = orc.argmax_lowest(om.forward(cache, [tok], cache.len))
    return time.perf_counter() - t0, n_steps


def oracle_prefill_rate(w: inputs.Workload, n_tokens: int):
    """Time the oracle's prefill of the first n_tokens of the workload's
    prompt; return tokens per second."""
    om = _oracle_model(w)
    prompt = inputs.prompt_tokens(w.shape, w.seed, w.prompt_len)[:n_tokens]
    cache = om.new_cache(n_tokens + 1)
    t0 = time.perf_counter()
    om.forward(cache, prompt, 0)
    return n_tokens / (time.perf_counter() - t0)


def oracle_decode_extrapolated(w: inputs.Workload, n_layers_built: int = 1):
    """Decode-step time of a model too large to build on the host: a
    1-layer model of the same geometry is built, one decode step is timed
    whole (embedding, layer, final norm, lm_head) and its layer alone, and
    the step is extrapolated to all layers: t = t_step + (L - 1) * t_layer.
    Returns (seconds per step, description)."""
    from oracle import qw3_oracle as orc
    s = w.shape
    s1 = s.with_layers(n_layers_built)
    om = _oracle_model(w, s1)
    P = 16
    prompt = inputs.prompt_tokens(s1, w.seed, P)
    cache = om.new_cache(P + 4)
    tok = orc.argmax_lowest(om.forward(cache, prompt, 0))
    t0 = time.perf_counter()
    tok = orc.argmax_lowest(om.forward(cache, [tok], cache.len))
    t_step = time.perf_counter() - t0
    x = om.tok_embd.row(np.asarray([tok]))
    lw = om.layers[0]
    t1 = time.perf_counter()
    x = om._attention_block(0, lw, x, np.asarray([cache.len]), cache)
    x = om._ffn_block(lw, x)
    t_layer = time.perf_counter() - t1
    secs = t_step + (s.n_layers - n_layers_built) * t_layer
    return secs, (f"oracle (f64 numpy) decode step of a {n_layers_built}-layer model of this geometry after a "
                  f"{P}-token prompt, timed whole and per layer, extrapolated to {s.n_layers} layers")


def run_reference(a, w: inputs.Workload):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    cores = oracle_cores()
    s = w.shape
    if w.decode_steps == 0:
        n = min(256, w.prompt_len)
        rate = oracle_prefill_rate(w, n)
        line = {"impl": "reference", "metric": f"{w.name} prefill tok/s", "value": rate, "unit": "tok/s",
                "n_gpus": a.gpus, "steps": 1, "warmup": 0, "ms_per_step": 1e3 * w.prompt_len / rate,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded random weights and prompt)",
                "config": {"workload": f"{w.name}: one {w.prompt_len}-token prefill per step"},
                "cpu_baseline": {"value": rate, "unit": "tok/s", "cores": cores, "kind": "oracle",
                                 "sample": f"oracle (f64 numpy) prefill of the first {n} tokens of the prompt; "
                                           f"the rate of the whole {w.prompt_len}-token prompt is lower "
                                           f"(attention grows with length)"},
                "e2e": {"value": rate, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0
    steps, warm = a.steps, a.warmup
    big = s.n_layers * (s.hidden * (2 * s.q_width + 2 * s.kv_width) + 3 * s.hidden * s.intermediate) > 1e9
    if big:
        secs_per, sample = oracle_decode_extrapolated(w)
        tok_s, n, secs = 1.0 / secs_per, steps, secs_per * steps
    else:
        # Batched workloads: one sequence of the batch stands for the step's cost per token.
        P = min(w.prompt_len, 512) if w.batch > 1 else w.prompt_len
        secs, n = oracle_decode(w, warm, steps, P)
        tok_s = n / secs
        sample = (f"oracle (f64 numpy) greedy decode at B=1: prefill {P} seeded tokens untimed, {warm} untimed "
                  f"steps, rewind, then {n} timed steps at positions {P}..{P + n - 1}")
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


def workload_config(w: inputs.Workload, steps: int, kv: str = "f32", wtype: str = "q8_0") -> dict:
    s = w.shape
    cfg = {"workload": f"{w.name}: Qwen3 dense, vocab {s.vocab}, hidden {s.hidden}, {s.n_layers} layers, "
                       f"{s.n_heads}/{s.n_kv_heads} heads, head_dim {s.head_dim}, intermediate {s.intermediate}, "
                       f"{'tied' if s.tied else 'untied'} lm_head, seed {w.seed}; "
                       f"prefill {w.prompt_len} tokens untimed, then greedy decode at B={w.batch}",
           "batch": w.batch, "prompt_len": w.prompt_len, "timed_positions": [w.prompt_len, w.prompt_len + steps - 1],
           "weights": f"{wtype.upper()}, {weight_bytes_per_step(s, wtype) / 1e6:.1f} MB streamed per step",
           "kv_cache": kv,
           "l2": ("inputs larger than L2 (the Q8_0 weights streamed every step exceed the 129 MB L2)"
                  if weight_bytes_per_step(s) > 129e6 else
                  "inputs smaller than L2: the weights stay L2-resident between steps (a small test case)")}
    return cfg


# ------------------------------------------------------------- GPU arms

def _gpu_setup():
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
    return torch, qw3, world, rank, local, dev


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _decode_model(qw3, w: inputs.Workload, cap: int, flags: int = 0):
    s = w.shape
    return qw3.Qw3Model.from_f32(s, inputs.iter_weights(s, w.seed), max_seqs=w.batch, max_seq_len=cap,
                                 max_prefill=min(w.prompt_len, 4096), flags=flags)


def _prefill_batch(torch, model, w: inputs.Workload, dev):
    firsts = []
    for b in range(w.batch):
        toks = (inputs.prompt_tokens(w.shape, w.seed, w.prompt_len) if w.batch == 1 else
                inputs.batch_prefix_tokens(w.shape, w.seed, b, w.prompt_len))
        _, am = model.prefill(b, torch.from_numpy(toks).to(dev), want_logits=False)
        firsts.append(am)
    first = torch.cat(firsts)
    model.sync()
    return first


def time_decode(torch, qw3, model, w: inputs.Workload, K: int, W: int, runs: int, world: int, local: int, dev):
    """W untimed warm-up steps, then `runs` timed qw3_generate_greedy calls of
    K steps each, every one from the same cache state (positions P..P+K-1).
    Returns (ms per run, tokens of the last run, first tokens, clocks)."""
    B, P = w.batch, w.prompt_len
    first = _prefill_batch(torch, model, w, dev)
    if W > 0:
        model.generate_greedy(first, W)
        model.sync()
    out = torch.empty((K, B), dtype=torch.int32, device=dev)
    stream = model.stream
    clocks = ClockSampler(local).start()
    ms = []
    for _ in range(runs):
        for b in range(B):
            model.truncate(b, P)
        torch.cuda.synchronize()
        _barrier(world)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            qw3.qw3_generate_greedy(model.h, B, None, K, first.data_ptr(), out.data_ptr())
            ev1.record(stream)
        torch.cuda.synchronize()
        ms.append(ev0.elapsed_time(ev1))
    clk = clocks.stop()
    model.sync()
    _barrier(world)
    return ms, out, first, clk


def decode_roofline(w: inputs.Workload, K: int, ms_step: float, key: str, kv: str = "f32",
                    wtype: str = "q8_0") -> dict:
    s, B, P = w.shape, w.batch, w.prompt_len
    positions = [[P + i] * B for i in range(K)]
    alg = decode_bytes(s, B, positions, kv, wtype) / K
    hbm_peak, _, kind = peaks()
    achieved = alg / (ms_step / 1e3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
            "peak_source": (f"{kind} (MEASURED_PEAKS.json hbm_gbs)" if kind == "measured" else "fallback 6.8 TB/s"),
            "algorithmic_bytes_per_step": alg, "traffic": profiled_traffic(key)}


def step_phase_table(torch, qw3, w: inputs.Workload, dev, sm_mhz):
    """Per-phase times of one decode step of the persistent step kernel,
    from a separately built traced model (untimed): mean over layers of the
    last CTA's phases, from its SM cycle counter."""
    s = w.shape
    model = _decode_model(qw3, w, w.prompt_len + 16, flags=qw3.QW3_FLAG_TRACE)
    try:
        first = _prefill_batch(torch, model, w, dev)
        model.generate_greedy(first, 4)
        model.sync()
        if not model.decode_plan(1)[0]:
            return None
        tr = model.read_trace(1 << 20).astype(np.int64).reshape(-1)
    finally:
        model.close()
    L = s.n_layers
    nph = 6 * L + 2
    per = nph * 4 + 64
    a = tr[per: per + nph * 4].reshape(nph, 4)        # the last CTA
    clk = (sm_mhz or 2070.0)                          # cycles per microsecond
    names = ("qkv", "attention", "combine", "o_proj", "gate_up", "down")
    phases = {}
    for q in range(1, 7):
        d = [(a[6 * l + q, 3] - a[6 * l + q - 1, 3]) / clk for l in range(1, L) if a[6 * l + q, 3] and a[6 * l + q - 1, 3]]
        if d:
            phases[names[q - 1]] = {"mean_us": float(np.mean(d)), "share_of_layer": None}
    layer_us = float(np.mean(np.diff([a[6 * l + 6, 3] for l in range(L)]))) / clk
    for v in phases.values():
        v["share_of_layer"] = v["mean_us"] / layer_us
    lm_us = float(a[nph - 1, 3] - a[nph - 1, 0]) / clk
    return {"source": "SM cycle counter of the last CTA of the persistent step kernel, a separate traced run "
                      "(untimed); phase time = its output published minus the previous phase's",
            "layer_us": layer_us, "lm_head_us": lm_us, "phases": phases}


def run_decode_line(a, torch, qw3, world, rank, local, dev, w: inputs.Workload, K: int, W: int, headline: bool,
                    kv: str = "f32", wtype: str = "q8_0"):
    s, B, P = w.shape, w.batch, w.prompt_len
    runs = max(1, a.runs)
    cap = P + max(K, 1) + W + 2
    flags = qw3.QW3_FLAG_PER_KERNEL if a.per_kernel else 0
    flags |= {"f32": 0, "f16": qw3.QW3_FLAG_KV_F16, "q8_0": qw3.QW3_FLAG_KV_Q8}[kv]
    if wtype == "q4_k":
        flags |= qw3.QW3_FLAG_WEIGHTS_Q4_K
    model = _decode_model(qw3, w, cap, flags)
    persistent, launches_per_step = model.decode_plan(B)
    ms_runs, out, first, clk = time_decode(torch, qw3, model, w, K, W, runs, world, local, dev)
    ms = statistics.median(ms_runs)
    ms_max = aggregate_max(ms, world, dev)
    tokens_all = aggregate_sum(float(K * B), world, dev)
    value = tokens_all / (ms_max / 1e3)
    roof = decode_roofline(w, K, ms / K, "k_step" if persistent else "decode_step", kv, wtype)
    roof["kernel"] = ("k_step: one persistent launch per decode step (embedding, every layer's projections, "
                      "attention, FFN, lm_head and argmax)" if persistent else
                      "decode step (per-kernel path: Q8_0 GEMVs or GEMMs, attention, embedding, lm_head + argmax)")
    line = {
        "metric": (METRIC if headline and w.name == "qwen3-0.6b-decode" else
                   f"{w.name} decode tok/s" + ("" if kv == "f32" else f" ({kv} KV cache)")
                   + ("" if wtype == "q8_0" else f" ({wtype} weights)")),
        "value": value, "unit": "tok/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_max / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": f"synthetic (seeded random-init weights quantised to {wtype.upper()}, seeded prompt)",
        "config": dict(workload_config(w, K, kv, wtype), parallelism="replicas" if world > 1 else "single GPU",
                       timing=f"CUDA events on the model stream around one qw3_generate_greedy call of K steps; "
                              f"median of {runs} runs from the same cache state (ms per run: "
                              f"{', '.join(f'{x:.3f}' for x in ms_runs)})"),
        "roofline": roof,
        "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "gpu_launches": launches_per_step * K,
    }
    if headline:
        # e2e: host token in, host token out, one qw3_decode per step
        for b in range(B):
            model.truncate(b, P)
        stream = model.stream
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
        e2e_s = aggregate_max(time.perf_counter() - t0, world, dev)
        line["e2e"] = {"value": tokens_all / e2e_s, "unit": "tok/s", "h2d_bytes_per_step": 4 * B,
                       "d2h_bytes_per_step": 4 * B,
                       "how": "per step: pinned host token -> device, qw3_decode, argmax -> pinned host, stream sync",
                       "ids_match_timed_run": bool(torch.equal(h_out.to(dev), out[K - 1]))}
        model.sync()
    model.close()
    torch.cuda.synchronize()
    if headline and persistent and B == 1 and rank == 0 and not a.no_trace:
        line["phases_last_step"] = step_phase_table(torch, qw3, w, dev, clk["sm_mhz"])
    return line


def run_prefill_line(a, torch, qw3, world, rank, local, dev, w: inputs.Workload, runs: int):
    s, S = w.shape, w.prompt_len
    model = qw3.Qw3Model.from_f32(s, inputs.iter_weights(s, w.seed), max_seqs=1, max_seq_len=S + 1, max_prefill=S)
    toks_h = torch.from_numpy(inputs.prompt_tokens(s, w.seed, S)).pin_memory()
    toks = toks_h.to(dev)
    am = torch.empty(1, dtype=torch.int32, device=dev)
    for _ in range(max(1, a.warmup)):
        model.reset(0)
        qw3.qw3_prefill(model.h, 0, toks.data_ptr(), S, 0, am.data_ptr())
    model.sync()
    clocks = ClockSampler(local).start()
    stream = model.stream
    ms_runs = []
    for _ in range(runs):
        model.reset(0)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        qw3.qw3_prefill(model.h, 0, toks.data_ptr(), S, 0, am.data_ptr())
        e1.record(stream)
        torch.cuda.synchronize()
        ms_runs.append(e0.elapsed_time(e1))
    clk = clocks.stop()
    model.sync()
    ms = statistics.median(ms_runs)
    # e2e: the prompt from pinned host memory, prefill, the argmax back to the host
    h_am = torch.empty(1, dtype=torch.int32, pin_memory=True)
    d_toks = torch.empty(S, dtype=torch.int32, device=dev)
    e2e_ms = []
    for _ in range(runs):
        model.reset(0)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            d_toks.copy_(toks_h, non_blocking=True)
            qw3.qw3_prefill(model.h, 0, d_toks.data_ptr(), S, 0, am.data_ptr())
            h_am.copy_(am, non_blocking=True)
            stream.synchronize()
        e2e_ms.append(1e3 * (time.perf_counter() - t0))
    model.sync()
    model.close()
    ms_max = aggregate_max(ms, world, dev)
    value = aggregate_sum(float(S), world, dev) / (ms_max / 1e3)
    flops = prefill_flops(s, S)
    _, tf_peak, peak_kind = peaks()
    achieved = flops / (ms / 1e3) / 1e12
    launches = 1 + 12 * s.n_layers + 1
    return {"metric": f"{w.name} prefill tok/s", "value": value, "unit": "tok/s", "n_gpus": world,
            "steps": runs, "warmup": max(1, a.warmup), "ms_per_step": ms_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded random-init weights quantised to Q8_0, seeded prompt)",
            "config": {"workload": f"{w.name}: one {S}-token prefill per step (Qwen3-0.6B geometry, seed {w.seed})",
                       "prompt_len": S, "l2": "inputs larger than L2",
                       "timing": f"CUDA events around one qw3_prefill call; median of {runs} "
                                 f"(ms: {', '.join(f'{x:.3f}' for x in ms_runs)})"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": tf_peak, "unit": "TFLOP/s",
                         "frac": achieved / tf_peak,
                         "peak_source": f"{peak_kind} bf16 sustained (MEASURED_PEAKS.json bf16_tflops_sustained; "
                                        "the dense fp16 rate is nominally the bf16 rate)",
                         "note": "achieved counts the model's FLOPs (linear + causal attention + last-row lm_head); "
                                 "the GEMMs and the causal attention run as three fp16 MMAs per product (hi/lo "
                                 "split of power-of-two-scaled rows, for f32 accuracy) in short accumulation "
                                 "chains promoted into f32",
                         "algorithmic_flops_per_step": flops, "traffic": None},
            "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
            "gpu_launches": launches * runs,
            "e2e": {"value": S / (statistics.median(e2e_ms) / 1e3), "unit": "tok/s", "h2d_bytes_per_step": 4 * S,
                    "d2h_bytes_per_step": 4,
                    "how": "per step: pinned host prompt -> device, qw3_prefill, argmax -> pinned host, sync"}}


def cpu_baseline_for(w: inputs.Workload, headline_steps: int = 8):
    """The CPU oracle on this host, a bounded sample of the workload."""
    cores = oracle_cores()
    s = w.shape
    if w.decode_steps == 0:
        n = min(256, w.prompt_len)
        rate = oracle_prefill_rate(w, n)
        return {"value": rate, "unit": "tok/s", "cores": cores, "kind": "oracle",
                "sample": f"oracle (f64 numpy) prefill of the first {n} tokens of the prompt; the rate of the whole "
                          f"{w.prompt_len}-token prompt is lower (attention grows with length)"}
    big = s.n_layers * (s.hidden * (2 * s.q_width + 2 * s.kv_width) + 3 * s.hidden * s.intermediate) > 1e9
    if big:
        secs, sample = oracle_decode_extrapolated(w)
        return {"value": 1.0 / secs, "unit": "tok/s", "cores": cores, "kind": "oracle", "sample": sample}
    P = w.prompt_len if w.batch == 1 else min(w.prompt_len, 512)
    secs, n = oracle_decode(w, 0, headline_steps, P)
    sample = f"oracle (f64 numpy) greedy decode at B=1 after an untimed {P}-token prefill: {n} timed steps"
    if w.batch > 1:
        sample += f" (one sequence of the batch-{w.batch} workload, prefix cut to {P} tokens; per-sequence rate)"
    return {"value": n / secs, "unit": "tok/s", "cores": cores, "kind": "oracle", "sample": sample}


def run_ours(a, w: inputs.Workload):
    torch, qw3, world, rank, local, dev = _gpu_setup()
    K, W = a.steps, a.warmup
    if w.decode_steps == 0:
        line = run_prefill_line(a, torch, qw3, world, rank, local, dev, w, max(K, 3) if K < 50 else 5)
    else:
        line = run_decode_line(a, torch, qw3, world, rank, local, dev, w, K, W, headline=True)
    if world == 1 and not a.no_workloads and w.name == "qwen3-0.6b-decode":
        extra = {}
        wp = inputs.WORKLOADS["qwen3-0.6b-prefill4096"]
        extra["prefill4096"] = run_prefill_line(a, torch, qw3, world, rank, local, dev, wp, 5)
        for key, name in (("batch64", "qwen3-0.6b-batch64"), ("qwen3_8b", "qwen3-8b")):
            wd = inputs.WORKLOADS[name]
            extra[key] = run_decode_line(a, torch, qw3, world, rank, local, dev, wd, wd.decode_steps, W,
                                         headline=False)
        # the batch-64 workload with the pages' smaller cache types (modes,
        # not the workload's f32 cache): the K/V stream is 98 % of its bytes
        wb = inputs.WORKLOADS["qwen3-0.6b-batch64"]
        for kv in ("f16", "q8_0"):
            extra[f"batch64_kv_{kv}"] = run_decode_line(a, torch, qw3, world, rank, local, dev, wb, wb.decode_steps,
                                                        W, headline=False, kv=kv)
        # batch-1 decode of the 0.6B shape with Q4_K weights (4.5 bits per weight)
        extra["decode_q4_k"] = run_decode_line(a, torch, qw3, world, rank, local, dev, w, K, W, headline=False,
                                               wtype="q4_k")
        if rank == 0 and not a.no_cpu_baseline:
            for key, name in (("prefill4096", "qwen3-0.6b-prefill4096"), ("batch64", "qwen3-0.6b-batch64"),
                              ("qwen3_8b", "qwen3-8b")):
                extra[key]["cpu_baseline"] = cpu_baseline_for(inputs.WORKLOADS[name])
        line["workloads"] = extra
    if rank == 0:
        line["cpu_baseline"] = None if a.no_cpu_baseline else cpu_baseline_for(w, a.cpu_steps)
        print(json.dumps(line), flush=True)
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--runs", type=int, default=3, help="timed runs per line (the median is reported)")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="qwen3-0.6b-decode", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--cpu-steps", type=int, default=8, help="oracle decode steps timed for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="time the headline workload only")
    ap.add_argument("--no-trace", action="store_true", help="skip the untimed traced run of the phase table")
    ap.add_argument("--per-kernel", action="store_true",
                    help="batch-1 decode through the per-kernel chain instead of the persistent step kernel")
    a = ap.parse_args(argv)
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = inputs.WORKLOADS[a.workload]
    if a.impl == "reference":
        return run_reference(a, w)
    return run_ours(a, w)


if __name__ == "__main__":
    sys.exit(main())
