"""Shared helpers of the GPU parity tests: build the oracle and the CUDA
model from the same seeded f32 tensors, and compare logits rows.

Tolerances (the stated parity bar): every logits row within max-abs 2e-3 and
relative L2 1e-4 of the oracle's; greedy ids and codec bytes bit-exact.

Near ties. The oracle sums in f64, the CUDA path in f32 and in another
order; reassociating a reduction changes the last bits of its result ("A
transformer from scratch", 12.5). Where the oracle's own two largest logits
of a row lie closer than TIE_MARGIN, both tokens are the greedy choice at f32
precision. One rule, applied by every test that compares greedy ids:
a teacher-forced step accepts either token of such a row (assert_argmax);
a free-running id sequence is compared bit-exactly up to the first such row
(tie_free_prefix), since after it the two runs may follow different, equally
valid continuations.
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


TIE_MARGIN = 1e-4


def top2_margin(row) -> float:
    r = np.sort(np.asarray(row, np.float64).reshape(-1))
    return float(r[-1] - r[-2]) if r.size > 1 else float("inf")


def tie_free_prefix(rows) -> int:
    """Number of leading logits rows whose top-2 margin is at least TIE_MARGIN."""
    for i, r in enumerate(rows):
        if top2_margin(r) < TIE_MARGIN:
            return i
    return len(rows)


def assert_argmax(got: int, want: int, row, what="argmax"):
    """got is the oracle's greedy token, or the row is a near tie between the
    two (row = the oracle's logits)."""
    row = np.asarray(row, np.float64).reshape(-1)
    assert got == want or row[want] - row[got] < TIE_MARGIN, \
        f"{what}: {got} != {want} (oracle margin {row[want] - row[got]:.3e})"


def assert_ids_prefix(got, want, rows, what="greedy ids"):
    """Free-running ids bit-exact up to the first near tie of the oracle's
    rows (rows[i] produced want[i])."""
    n = tie_free_prefix(rows)
    assert list(got)[:n] == list(want)[:n], f"{what}: differ before the first near tie (row {n})"


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
