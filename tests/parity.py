"""Shared helpers of the GPU parity tests: build the oracle and the CUDA
model from the same seeded f32 tensors, and compare logits rows.

Tolerances (the stated parity bar): every logits row within max-abs 2e-3 and
relative L2 1e-4 of the oracle's; greedy ids and codec bytes bit-exact.
"""
from __future__ import annotations

import numpy as np

from oracle import qw3_oracle as orc
from quantized_transformer_decode_gb300 import inputs

MAX_ABS = 2e-3
REL_L2 = 1e-4


def row_errors(g, o):
    g = np.asarray(g, np.float64).reshape(-1)
    o = np.asarray(o, np.float64).reshape(-1)
    max_abs = float(np.max(np.abs(g - o))) if g.size else 0.0
    rel = float(np.linalg.norm(g - o) / max(np.linalg.norm(o), 1e-30))
    return max_abs, rel


def assert_logits_close(g, o, what="logits", max_abs=MAX_ABS, rel_l2=REL_L2):
    ma, rel = row_errors(g, o)
    assert ma <= max_abs and rel <= rel_l2, f"{what}: max-abs {ma:.3e} (<= {max_abs}), rel-L2 {rel:.3e} (<= {rel_l2})"
    return ma, rel


def build_pair(shape, seed, *, max_seqs=1, max_seq_len=256, max_prefill=64, flags=0):
    """(oracle model, CUDA model) over identical seeded f32 weights; each side
    quantises with its own Q8_0 encoder."""
    from quantized_transformer_decode_gb300.qw3 import Qw3Model
    w = inputs.generate_weights(shape, seed)
    om = orc.OracleModel.from_f32(shape, w)
    gm = Qw3Model.from_f32(shape, inputs.iter_weights(shape, seed), max_seqs=max_seqs, max_seq_len=max_seq_len,
                           max_prefill=max_prefill, flags=flags)
    return om, gm


def cuda_ints(vals):
    import torch
    return torch.tensor(np.asarray(vals, dtype=np.int32), device="cuda")
