"""Seeded synthetic workloads for the Qwen3-style dense decoder.

This module is the one piece shared by the CPU oracle and the CUDA path. It
holds shapes, seeds and value distributions only -- none of the model's
arithmetic (no quantisation, no norm, no matmul). Each side turns the f32
tensors drawn here into Q8_0 blocks with its own codec.

Shapes follow the Qwen3 tensor inventory of the minfer page ("Qwen3 Support
Plan (dense)", section 1) and the course config of "A transformer from
scratch" (section 12.1): linear weights are [out][in] row-major.

Distributions (no trained weights exist here, so seeded random ones stand in):
  * every linear weight, the token embedding included: N(0, 0.02), f32;
  * every norm weight (attn, ffn, q, k, output): 1 + N(0, 0.1), f32;
  * prompt tokens: uniform on [0, vocab).
Draw order: one numpy PCG64 stream per model seed, tensor by tensor in GGUF
order (token_embd, then per layer attn_norm, attn_q, attn_k, attn_v,
attn_q_norm, attn_k_norm, attn_output, ffn_norm, ffn_gate, ffn_up, ffn_down,
then output_norm, then output when the lm_head is untied).
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Iterator

import numpy as np

__all__ = [
    "Qwen3Shape", "TINY", "QWEN3_0_6B", "QWEN3_8B", "Workload", "WORKLOADS",
    "tensor_specs", "iter_weights", "generate_weights", "prompt_tokens",
    "batch_prefix_tokens", "uniform_block_values",
]


@dataclass(frozen=True)
class Qwen3Shape:
    """The nine integers of a Qwen3 dense config plus the lm_head tying."""
    vocab: int
    hidden: int
    n_layers: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    tied: bool = True

    @property
    def q_width(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_width(self) -> int:
        return self.n_kv_heads * self.head_dim

    def with_layers(self, n_layers: int) -> "Qwen3Shape":
        return replace(self, n_layers=n_layers)


# tiny parity model: 2 layers, hidden 256, 4/2 heads, head_dim 64
TINY = Qwen3Shape(vocab=4096, hidden=256, n_layers=2, n_heads=4, n_kv_heads=2,
                  head_dim=64, intermediate=768, tied=True)
# Qwen3-0.6B geometry ("A transformer from scratch", section 12.1)
QWEN3_0_6B = Qwen3Shape(vocab=151936, hidden=1024, n_layers=28, n_heads=16,
                        n_kv_heads=8, head_dim=128, intermediate=3072, tied=True)
# Qwen3-8B geometry, untied lm_head
QWEN3_8B = Qwen3Shape(vocab=151936, hidden=4096, n_layers=36, n_heads=32,
                      n_kv_heads=8, head_dim=128, intermediate=12288, tied=False)


@dataclass(frozen=True)
class Workload:
    """One seeded job: a model shape, a seed, a prompt length and decode steps."""
    name: str
    shape: Qwen3Shape
    seed: int
    prompt_len: int
    decode_steps: int
    batch: int = 1


WORKLOADS = {
    "tiny": Workload("tiny", TINY, seed=0, prompt_len=32, decode_steps=16),
    "qwen3-0.6b-decode": Workload("qwen3-0.6b-decode", QWEN3_0_6B, seed=1,
                                  prompt_len=512, decode_steps=256),
    "qwen3-0.6b-prefill4096": Workload("qwen3-0.6b-prefill4096", QWEN3_0_6B, seed=1,
                                       prompt_len=4096, decode_steps=0),
    "qwen3-0.6b-batch64": Workload("qwen3-0.6b-batch64", QWEN3_0_6B, seed=1,
                                   prompt_len=2048, decode_steps=128, batch=64),
    "qwen3-8b": Workload("qwen3-8b", QWEN3_8B, seed=2, prompt_len=8192, decode_steps=128),
}


def tensor_specs(shape: Qwen3Shape) -> list[tuple[str, str, tuple[int, ...]]]:
    """(name, kind, dims) in GGUF order; kind is 'linear' or 'norm'."""
    s = shape
    specs: list[tuple[str, str, tuple[int, ...]]] = [
        ("token_embd", "linear", (s.vocab, s.hidden))]
    for i in range(s.n_layers):
        p = f"blk.{i}."
        specs += [
            (p + "attn_norm", "norm", (s.hidden,)),
            (p + "attn_q", "linear", (s.q_width, s.hidden)),
            (p + "attn_k", "linear", (s.kv_width, s.hidden)),
            (p + "attn_v", "linear", (s.kv_width, s.hidden)),
            (p + "attn_q_norm", "norm", (s.head_dim,)),
            (p + "attn_k_norm", "norm", (s.head_dim,)),
            (p + "attn_output", "linear", (s.hidden, s.q_width)),
            (p + "ffn_norm", "norm", (s.hidden,)),
            (p + "ffn_gate", "linear", (s.intermediate, s.hidden)),
            (p + "ffn_up", "linear", (s.intermediate, s.hidden)),
            (p + "ffn_down", "linear", (s.hidden, s.intermediate)),
        ]
    specs.append(("output_norm", "norm", (s.hidden,)))
    if not s.tied:
        specs.append(("output", "linear", (s.vocab, s.hidden)))
    return specs


LINEAR_STD = np.float32(0.02)
NORM_STD = np.float32(0.1)


def iter_weights(shape: Qwen3Shape, seed: int) -> Iterator[tuple[str, str, np.ndarray]]:
    """Yield (name, kind, f32 array) one tensor at a time, in GGUF order."""
    rng = np.random.default_rng(seed)
    for name, kind, dims in tensor_specs(shape):
        z = rng.standard_normal(dims, dtype=np.float32)
        if kind == "linear":
            z *= LINEAR_STD
        else:
            z *= NORM_STD
            z += np.float32(1.0)
        yield name, kind, z


def generate_weights(shape: Qwen3Shape, seed: int) -> dict[str, np.ndarray]:
    """All f32 tensors of a model at once (small models only)."""
    return {name: arr for name, _, arr in iter_weights(shape, seed)}


def prompt_tokens(shape: Qwen3Shape, seed: int, n: int) -> np.ndarray:
    """The seeded prompt: n uniform token ids in [0, vocab), int32."""
    rng = np.random.default_rng([seed, 1])
    return rng.integers(0, shape.vocab, size=n, dtype=np.int64).astype(np.int32)


def batch_prefix_tokens(shape: Qwen3Shape, seed: int, b: int, n: int) -> np.ndarray:
    """Sequence b's seeded prefix for the batched-decode workload, int32."""
    rng = np.random.default_rng([seed, 2, b])
    return rng.integers(0, shape.vocab, size=n, dtype=np.int64).astype(np.int32)


def uniform_block_values(seed: int, n: int, lo: float = -2.0, hi: float = 2.0) -> np.ndarray:
    """n f32 values uniform on [lo, hi): the codec round-trip workload."""
    rng = np.random.default_rng([seed, 3])
    return (rng.random(n, dtype=np.float32) * np.float32(hi - lo) + np.float32(lo)).astype(np.float32)
