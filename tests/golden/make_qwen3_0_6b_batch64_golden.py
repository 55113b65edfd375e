#!/usr/bin/env python3
"""Write the oracle's reference outputs for the batched-decode workload.

The workload: the Qwen3-0.6B geometry (seed 1), 64 sequences, each with its
own 2048-token seeded prefix (default_rng([seed, 2, b])) prefilled, then
greedy decode; sequences are independent ("A transformer from scratch",
12.5: a batch step is B single-sequence steps sharing one weight pass), so
the oracle runs the sampled sequences one at a time. Only the CPU oracle
(oracle/) and the seeded input generators run here.

Output, tests/golden/qwen3_0_6b_batch64_greedy.npz:
  seqs     int32 [8]:      the sampled sequence slots b;
  ids      int32 [8][65]:  per sequence the prefill's argmax, then 64 step argmaxes;
  margins  f32 [8][65]:    the oracle's top-2 logit gap of each of those rows;
  rows     int32 [R][2]:   (sequence index into seqs, step) of the stored logits;
  logits   f32 [R][V]:     those rows (teacher-forced: the GPU is fed the oracle's ids).

Run (a few minutes on 8 host cores, ~6 GB of memory):
    python tests/golden/make_qwen3_0_6b_batch64_golden.py
"""
from __future__ import annotations

import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

from oracle import qw3_oracle as orc  # noqa: E402
from quantized_transformer_decode_gb300 import inputs  # noqa: E402

SEQS = (0, 9, 18, 27, 36, 45, 54, 63)
N_STEPS = 64
STORED = ((0, 64), (7, 1))


def top2_gap(lg) -> float:
    t = np.sort(np.asarray(lg, np.float64))[-2:]
    return float(t[1] - t[0])


def main() -> int:
    w = inputs.WORKLOADS["qwen3-0.6b-batch64"]
    s, P = w.shape, w.prompt_len
    t0 = time.time()
    om = orc.OracleModel.from_f32(s, inputs.generate_weights(s, w.seed))
    print(f"model built in {time.time() - t0:.0f} s", flush=True)
    ids_all, margins, rows = [], [], []
    for i, b in enumerate(SEQS):
        t1 = time.time()
        prefix = inputs.batch_prefix_tokens(s, w.seed, b, P)
        ids, logits = om.generate_greedy(om.new_cache(P + N_STEPS + 1), prefix, N_STEPS)
        ids_all.append(ids)
        margins.append([top2_gap(lg) for lg in logits])
        for (si, step) in STORED:
            if si == i:
                rows.append(np.asarray(logits[step], np.float32))
        print(f"sequence {b}: {time.time() - t1:.0f} s, ids {ids[:6]}...", flush=True)
    out = os.path.join(HERE, "qwen3_0_6b_batch64_greedy.npz")
    np.savez_compressed(out, seqs=np.asarray(SEQS, np.int32), ids=np.asarray(ids_all, np.int32),
                        margins=np.asarray(margins, np.float32), rows=np.asarray(STORED, np.int32),
                        logits=np.stack(rows), prompt_len=np.int32(P), n_steps=np.int32(N_STEPS),
                        seed=np.int32(w.seed))
    print(f"wrote {out}", flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
