#!/usr/bin/env python3
"""Write the oracle's reference outputs for the Qwen3-8B-shape workload.

The workload: the 8B geometry (seed 2, hidden 4096, 36 layers, 32/8 heads,
head_dim 128, intermediate 12288, untied lm_head) with Q8_0 weights, an
8192-token seeded prompt, then 64 greedy decode steps at batch 1 ("A
transformer from scratch", 12.5-12.6). Only the CPU oracle (oracle/) and the
seeded input generators run here; nothing comes from the CUDA path.

Output, tests/golden/qwen3_8b_greedy.npz:
  ids     int32 [65]: the prefill's argmax, then each step's argmax;
  margins f32 [65]:   the oracle's top-2 logit gap of each of those rows;
  steps   int32 [R]:  which rows of the greedy run the stored logits are
                      (0 = the prefill's last row, s = decode step s);
  logits  f32 [R][V]: those rows (the row each id was taken from; the GPU
                      is fed the oracle's ids, so these are teacher-forced);
  prompt_len, n_steps, seed.

Run (about two hours on 8 host cores, ~12 GB of memory):
    python tests/golden/make_qwen3_8b_golden.py
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

STORED_STEPS = (0, 1, 32, 64)


def main() -> int:
    w = inputs.WORKLOADS["qwen3-8b"]
    s, P, n_steps = w.shape, w.prompt_len, 64
    t0 = time.time()
    om = orc.OracleModel.from_f32_stream(s, ((name, a) for name, _, a in inputs.iter_weights(s, w.seed)))
    print(f"model built in {time.time() - t0:.0f} s", flush=True)
    prompt = inputs.prompt_tokens(s, w.seed, P)
    cache = om.new_cache(P + n_steps + 1)
    t1 = time.time()
    ids, logits = om.generate_greedy(cache, prompt, n_steps)
    print(f"prefill + {n_steps} steps in {time.time() - t1:.0f} s", flush=True)
    rows = np.stack([np.asarray(logits[k], np.float32) for k in STORED_STEPS])
    margins = np.asarray([np.diff(np.sort(np.asarray(lg, np.float64))[-2:])[0] for lg in logits], np.float32)
    out = os.path.join(HERE, "qwen3_8b_greedy.npz")
    np.savez_compressed(out, ids=np.asarray(ids, np.int32), margins=margins,
                        steps=np.asarray(STORED_STEPS, np.int32), logits=rows,
                        prompt_len=np.int32(P), n_steps=np.int32(n_steps), seed=np.int32(w.seed))
    print(f"wrote {out}: ids {ids[:8]}...", flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
