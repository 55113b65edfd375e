"""CPU oracle for the Qwen3-style dense decoder over GGUF Q8_0 weights.

TEST INFRASTRUCTURE. This module is the slow, plain statement of what the
model computes, written from the source pages, and nothing else. Only the test
suite, the smoke check and the benchmark's CPU-baseline leg may import it; the
product path (the CUDA library and its Python binding) never does. It shares no
code, tables or constants with the CUDA path: the only common module is the
seeded input generator, which holds none of the model's arithmetic.

Numerics. Weights are Q8_0 blocks dequantised exactly (d*q has at most 18
significant bits, so it is exact in f32 and f64). Every tensor handed from one
step to the next -- the residual stream, normalised activations, projections,
the KV cache, logits -- is stored in f32, as the pages store activations and
as the f32 KV cache of the workloads fixes. Inside each step the arithmetic is
f64: dot products (a library matmul on f64 operands), norms, RoPE angles,
softmax. The Q8_0 encoder itself is specified in f32 by the pages and is done
in f32 here.

Sources (page title, section):
  * "A transformer from scratch" (Fucina course ch. 12): sections 12.1 (config),
    12.3 (forward pass), 12.3.2 (RMSNorm), 12.3.3 (QKV), 12.3.4 (RoPE),
    12.3.5 (GQA, causal attention, scale), 12.3.6 (SwiGLU), 12.3.7 (residual,
    final norm, last-row lm_head; the all-rows form for verification),
    12.4 (KV cache and its contracts, the f16 cache), 12.6 (greedy loop).
  * "Model files and quantization" (Fucina course ch. 11): section 11.7
    (Q8_0 block, encoder, decoder, round-trip bound), 11.8 (the Q4_K block
    and its decode), 11.9 (the quantized matmul on Q8_0-encoded activations:
    per-block integer dots times d_w * d_a), 11.10 (finite-input guard).
  * "The LLM stack (fucina_llm)" (Fucina reference section 13): 13.4 (KV cache
    contract and its worked test; the q8_0 cache with integer-score decode
    attention), 13.6 (greedy argmax example).
  * minfer "Qwen3 Support Plan (dense)": section 1 (tensor inventory),
    section 2.1 (head_dim 128, scale 1/sqrt(128), full-head NeoX RoPE,
    theta 1e6), section 2.2 (per-head Q/K RMSNorm before RoPE).

Parity status: every function here is pinned by tests/test_oracle.py against
closed forms, invariants, the pages' worked examples and an independent f64
cacheless brute force; nothing here is "parity unpinned".
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Sequence

import numpy as np

QK8_0 = 32          # values per Q8_0 block
Q8_0_BYTES = 34     # f16 scale + 32 int8 quants


class OracleError(ValueError):
    """Base of the oracle's typed errors (the pages' error names)."""


class NonFiniteValue(OracleError):
    """Encoder input held NaN or +-inf (course 11.10, the allFinite guard)."""


class InvalidShape(OracleError):
    """A length or shape the format or model cannot take."""


class InvalidSequenceLength(OracleError):
    """forward called with pos0 != cache length (course 12.4, contract 2)."""


class KvCacheOverflow(OracleError):
    """The cache has no room for the new rows (course 12.4, contract 2)."""


# ---------------------------------------------------------------------------
# Q8_0 codec -- "Model files and quantization", section 11.7
# ---------------------------------------------------------------------------

def _round_half_away(v32: np.ndarray) -> np.ndarray:
    """Round f32 values to integers, halves away from zero.

    Reading of the pages: the course encoder rounds with Zig's @round, which
    the text says rounds halves away from zero (section 11.10 contrasts it with
    ggml's round-to-nearest-even). Done in f64, where |v| + 0.5 is exact for
    every f32 v below 2**29, so no double rounding can occur.
    """
    v = v32.astype(np.float64)
    return np.sign(v) * np.floor(np.abs(v) + 0.5)


def q8_0_quantize_parts(x: np.ndarray):
    """Encode f32 values in blocks of 32; return (d32, q, d16).

    Per block (section 11.7): amax = max|v|; d = amax / 127 in f32;
    inv_d = 0 if d == 0 else 1 / d in f32; q = clamp(round(v * inv_d), -127, 127)
    with the product v * inv_d rounded once to f32; the stored scale is d as
    an IEEE f16 (round to nearest even). d32 is the f32 scale used to encode,
    d16 the stored one.

    Edge readings (not covered by the pages): when d is so small that 1/d
    overflows to +inf, a nonzero v saturates to +-127 and a zero v (0 * inf is
    NaN) encodes as 0.
    """
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    if x.size % QK8_0:
        raise InvalidShape(f"length {x.size} is not a multiple of {QK8_0}")
    if not np.all(np.isfinite(x)):
        raise NonFiniteValue("Q8_0 encoder input holds NaN or inf")
    v = x.reshape(-1, QK8_0)
    amax = np.max(np.abs(v), axis=1)
    d = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        inv_d = np.where(d == 0, np.float32(0.0), np.float32(1.0) / d).astype(np.float32)
        prod = (v * inv_d[:, None]).astype(np.float32)
    nan = np.isnan(prod)
    prod = np.where(nan, np.float32(0.0), prod)
    r = np.clip(_round_half_away(prod), -127.0, 127.0)
    q = r.astype(np.int8)
    with np.errstate(over="ignore"):
        d16 = d.astype(np.float16)   # |d| above the f16 range stores as inf
    return d, q, d16


def q8_0_quantize(x: np.ndarray) -> np.ndarray:
    """Encode to the GGUF wire format: per block 2 bytes f16 d (little endian)
    then 32 int8 quants, 34 bytes in all (section 11.7, BlockQ8_0)."""
    _, q, d16 = q8_0_quantize_parts(x)
    nb = q.shape[0]
    out = np.empty((nb, Q8_0_BYTES), dtype=np.uint8)
    out[:, 0:2] = d16.astype("<f2").view(np.uint8).reshape(nb, 2)
    out[:, 2:] = q.view(np.uint8)
    return out.reshape(-1)


def q8_0_unpack(blocks: np.ndarray, n: int):
    """Split wire bytes into (d16 [nb] float16, q [nb, 32] int8)."""
    if n % QK8_0:
        raise InvalidShape(f"length {n} is not a multiple of {QK8_0}")
    nb = n // QK8_0
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1)
    if b.size != nb * Q8_0_BYTES:
        raise InvalidShape(f"{b.size} bytes do not hold {nb} Q8_0 blocks")
    b = b.reshape(nb, Q8_0_BYTES)
    d16 = np.ascontiguousarray(b[:, 0:2]).view("<f2").reshape(nb)
    q = np.ascontiguousarray(b[:, 2:]).view(np.int8)
    return d16, q


def q8_0_dequantize(blocks: np.ndarray, n: int) -> np.ndarray:
    """Decode: x = f32(d) * q per element (section 11.7). Exact in f32."""
    d16, q = q8_0_unpack(blocks, n)
    d = d16.astype(np.float32)
    return (d[:, None] * q.astype(np.float32)).astype(np.float32).reshape(-1)


# ---------------------------------------------------------------------------
# Q4_K codec -- "Model files and quantization", section 11.8
# ---------------------------------------------------------------------------

QK_K = 256          # values per Q4_K super-block
Q4_K_BYTES = 144    # f16 d, f16 dmin, 12 bytes of packed 6-bit scales/mins, 128 bytes of 4-bit codes


def q4k_pack_scales(sc: np.ndarray, m: np.ndarray) -> np.ndarray:
    """Eight 6-bit sub-scales and eight 6-bit sub-mins per super-block into
    the 12 bytes of the GGUF block (its published byte layout): bytes 0-3
    hold sub-scales 0-3 in their low six bits, bytes 4-7 sub-mins 0-3; the
    low nibbles of bytes 8-11 hold the low four bits of sub-scales 4-7, their
    high nibbles those of sub-mins 4-7; the top two bits of sub-scales 4-7
    sit in the top two bits of bytes 0-3, those of sub-mins 4-7 in bytes 4-7.
    sc, m: [nb, 8] integers in [0, 63]."""
    sc = sc.astype(np.uint16)
    m = m.astype(np.uint16)
    out = np.zeros((sc.shape[0], 12), np.uint16)
    out[:, 0:4] = sc[:, 0:4] | ((sc[:, 4:8] >> 4) << 6)
    out[:, 4:8] = m[:, 0:4] | ((m[:, 4:8] >> 4) << 6)
    out[:, 8:12] = (sc[:, 4:8] & 0xF) | ((m[:, 4:8] & 0xF) << 4)
    return out.astype(np.uint8)


def q4k_unpack_scales(scales: np.ndarray):
    """The inverse of the packing above: scales [nb, 12] bytes -> (sc, m),
    each [nb, 8] in [0, 63]."""
    b = scales.astype(np.uint16)
    sc = np.empty((b.shape[0], 8), np.uint16)
    m = np.empty((b.shape[0], 8), np.uint16)
    sc[:, 0:4] = b[:, 0:4] & 63
    m[:, 0:4] = b[:, 4:8] & 63
    sc[:, 4:8] = (b[:, 8:12] & 0xF) | ((b[:, 0:4] >> 6) << 4)
    m[:, 4:8] = (b[:, 8:12] >> 4) | ((b[:, 4:8] >> 6) << 4)
    return sc, m


def q4_k_quantize(x: np.ndarray) -> np.ndarray:
    """Encode f32 values in super-blocks of 256 to Q4_K wire bytes.

    The pages fix the block (f16 d and dmin, eight 6-bit sub-scales and
    sub-mins, 4-bit codes; x ~ d*sc*q - dmin*m per 32-value sub-block) but
    give no encoding algorithm; this is the plainest one, in f32:
    per sub-block lo = min(0, min x), S = (max x - lo) / 15, O = -lo; d =
    max S / 63 and dmin = max O / 63, stored as f16 (nearest even); sc =
    round(S / d16), m = round(O / dmin16), clamped to [0, 63] (0 when the
    stored scale is 0); per value q = round((x + dmin16*m) / (d16*sc)),
    clamped to [0, 15] (0 when d16*sc is 0). Rounding halves away from zero.
    Non-finite input is an error.
    """
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    if x.size % QK_K:
        raise InvalidShape(f"length {x.size} is not a multiple of {QK_K}")
    if not np.all(np.isfinite(x)):
        raise NonFiniteValue("Q4_K encoder input holds NaN or inf")
    nb = x.size // QK_K
    v = x.reshape(nb, 8, 32)
    lo = np.minimum(np.float32(0.0), v.min(axis=2)).astype(np.float32)
    S = ((v.max(axis=2) - lo).astype(np.float32) / np.float32(15.0)).astype(np.float32)
    O = (np.float32(0.0) - lo).astype(np.float32)            # +0, never -0, for an all-positive sub-block
    d = (S.max(axis=1) / np.float32(63.0)).astype(np.float32)
    dm = (O.max(axis=1) / np.float32(63.0)).astype(np.float32)
    with np.errstate(over="ignore"):
        d16 = d.astype(np.float16)
        dm16 = dm.astype(np.float16)
    d32 = d16.astype(np.float32)
    dm32 = dm16.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        sc = np.where(d32[:, None] > 0, np.clip(_round_half_away((S / d32[:, None]).astype(np.float32)), 0, 63), 0)
        m = np.where(dm32[:, None] > 0, np.clip(_round_half_away((O / dm32[:, None]).astype(np.float32)), 0, 63), 0)
    Se = (d32[:, None] * sc.astype(np.float32)).astype(np.float32)            # exact
    Oe = (dm32[:, None] * m.astype(np.float32)).astype(np.float32)            # exact
    with np.errstate(divide="ignore", invalid="ignore"):
        t = ((v + Oe[:, :, None]).astype(np.float32) / Se[:, :, None]).astype(np.float32)
        q = np.where(Se[:, :, None] > 0, np.clip(_round_half_away(np.nan_to_num(t)), 0, 15), 0).astype(np.uint8)
    q = q.reshape(nb, 4, 2, 32)                       # chunk c holds sub-blocks 2c (low nibble), 2c+1 (high)
    qs = (q[:, :, 0, :] | (q[:, :, 1, :] << 4)).reshape(nb, 128)
    out = np.empty((nb, Q4_K_BYTES), np.uint8)
    out[:, 0:2] = d16.astype("<f2").view(np.uint8).reshape(nb, 2)
    out[:, 2:4] = dm16.astype("<f2").view(np.uint8).reshape(nb, 2)
    out[:, 4:16] = q4k_pack_scales(sc.astype(np.uint16), m.astype(np.uint16))
    out[:, 16:] = qs
    return out.reshape(-1)


def q4_k_unpack(blocks: np.ndarray, n: int):
    """Wire bytes -> (d16 [nb], dmin16 [nb], sc [nb, 8], m [nb, 8], q [nb, 256] in value order)."""
    if n % QK_K:
        raise InvalidShape(f"length {n} is not a multiple of {QK_K}")
    nb = n // QK_K
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1)
    if b.size != nb * Q4_K_BYTES:
        raise InvalidShape(f"{b.size} bytes do not hold {nb} Q4_K blocks")
    b = b.reshape(nb, Q4_K_BYTES)
    d16 = np.ascontiguousarray(b[:, 0:2]).view("<f2").reshape(nb)
    dm16 = np.ascontiguousarray(b[:, 2:4]).view("<f2").reshape(nb)
    sc, m = q4k_unpack_scales(b[:, 4:16])
    qs = b[:, 16:].reshape(nb, 4, 32)
    q = np.stack([qs & 0xF, qs >> 4], axis=2).reshape(nb, 256)    # [chunk][low 32 | high 32]
    return d16, dm16, sc, m, q


def q4_k_dequantize(blocks: np.ndarray, n: int) -> np.ndarray:
    """Decode: per 32-value sub-block j, x = (d * sc_j) * q - (dmin * m_j),
    in f32 (the two products are exact; the difference rounds once)."""
    d16, dm16, sc, m, q = q4_k_unpack(blocks, n)
    nb = d16.size
    d1 = (d16.astype(np.float32)[:, None] * sc.astype(np.float32)).astype(np.float32)     # [nb, 8]
    m1 = (dm16.astype(np.float32)[:, None] * m.astype(np.float32)).astype(np.float32)
    qv = q.reshape(nb, 8, 32).astype(np.float32)
    return ((d1[:, :, None] * qv).astype(np.float32) - m1[:, :, None]).astype(np.float32).reshape(-1)


def matrix_from_blocks(blocks: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Dequantise a Q8_0 matrix stored [rows][cols/32 blocks] to f32 [rows, cols]."""
    return q8_0_dequantize(blocks, rows * cols).reshape(rows, cols)


# ---------------------------------------------------------------------------
# Elementwise and reduction steps -- "A transformer from scratch", 12.3
# ---------------------------------------------------------------------------

def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """y_i = x_i / sqrt(mean(x^2) + eps) * w_i over the last axis (12.3.2).

    The same function serves the per-head Q/K norm (minfer section 2.2): the
    last axis is then the head's head_dim values and w has length head_dim.
    """
    x64 = np.asarray(x, dtype=np.float32).astype(np.float64)
    ms = np.mean(x64 * x64, axis=-1, keepdims=True)
    y = x64 / np.sqrt(ms + float(eps)) * np.asarray(w, np.float32).astype(np.float64)
    return y.astype(np.float32)


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """f_i = theta^(-2i/d) for i < d/2 (12.3.4): pair i turns p*f_i radians."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / float(head_dim))


def rope_neox(x: np.ndarray, positions: Sequence[int], theta: float) -> np.ndarray:
    """NeoX "half" RoPE on x [M, heads, d] at positions [M] (12.3.4).

    Channel i pairs with channel i + d/2; the pair (a, b) at position p turns
    by angle p * f_i to (a cos - b sin, a sin + b cos), the course's rotate().
    Angles and rotation in f64, the result rounded to f32.
    """
    x64 = np.asarray(x, dtype=np.float32).astype(np.float64)
    d = x64.shape[-1]
    half = d // 2
    pos = np.asarray(positions, dtype=np.float64)
    ang = pos[:, None] * rope_inv_freq(d, theta)[None, :]          # [M, d/2]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a = x64[..., :half]
    b = x64[..., half:]
    out = np.concatenate([a * c - b * s, a * s + b * c], axis=-1)
    return out.astype(np.float32)


def kv_head_map(n_heads: int, n_kv_heads: int) -> list[int]:
    """Query head h reads KV head h / (n_heads / n_kv_heads) (12.3.5)."""
    if n_kv_heads <= 0 or n_heads % n_kv_heads:
        raise InvalidShape("n_heads must be a positive multiple of n_kv_heads")
    per = n_heads // n_kv_heads
    return [h // per for h in range(n_heads)]


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_positions: Sequence[int],
              scale: float, kv_head_for_head: Sequence[int]) -> np.ndarray:
    """Causal grouped-query attention (12.3.5).

    q [M, nh, d] at absolute positions q_positions; k, v [T, nkv, d] hold cache
    rows 0..T-1. The query at position p attends keys 0..p with weights
    softmax_j(q . k_j * scale) (max subtracted before exp) and returns the
    weighted sum of v_j. Returns [M, nh, d] f32.
    """
    q64 = np.asarray(q, np.float32).astype(np.float64)
    k64 = np.asarray(k, np.float32).astype(np.float64)
    v64 = np.asarray(v, np.float32).astype(np.float64)
    M, nh, d = q64.shape
    T = k64.shape[0]
    pos = np.asarray(q_positions, dtype=np.int64)
    masked = np.arange(T)[None, :] > pos[:, None]                   # [M, T]
    out = np.empty((M, nh, d), dtype=np.float64)
    for h in range(nh):
        g = kv_head_for_head[h]
        s = (q64[:, h, :] @ k64[:, g, :].T) * float(scale)
        s[masked] = -np.inf
        s -= np.max(s, axis=1, keepdims=True)
        p = np.exp(s)
        p /= np.sum(p, axis=1, keepdims=True)
        out[:, h, :] = p @ v64[:, g, :]
    return out.astype(np.float32)


def q8_scores(q: np.ndarray, kq: np.ndarray, kd: np.ndarray, kv_head_for_head: Sequence[int]) -> np.ndarray:
    """Raw attention scores of one query row over a q8_0 K cache ("The LLM
    stack", 13.4: the query row is quantised once per head to q8_0 and the
    scores are q8 x q8 dots straight on the cached K blocks).

    q [nh, d] f32 (after the Q norm and RoPE); kq [T, nkv, d] int8 codes and
    kd [T, nkv, d/32] f16 scales of the cached keys. Each head's query is
    encoded by the 11.7 encoder; a (key block, query block) pair contributes
    (k.d * q.d) * f32(i32 dot) in f32, the dotBlocks form of "Model files and
    quantization", 11.9; the blocks of a row sum in f64. Returns [nh, T] f64,
    before the 1/sqrt(d) scale.
    """
    q32 = np.asarray(q, np.float32)
    nh, d = q32.shape
    T = kq.shape[0]
    nb = d // QK8_0
    _, qa, qd16 = q8_0_quantize_parts(q32.reshape(-1))
    qa = qa.reshape(nh, nb, QK8_0).astype(np.float64)
    qd = qd16.astype(np.float32).reshape(nh, nb)
    out = np.zeros((nh, T), dtype=np.float64)
    for h in range(nh):
        g = kv_head_for_head[h]
        codes = kq[:, g, :].reshape(T, nb, QK8_0).astype(np.float64)
        scales = kd[:, g, :].astype(np.float32)
        for b in range(nb):
            acc = codes[:, b, :] @ qa[h, b]                                   # exact integer dots
            term = (scales[:, b] * qd[h, b]).astype(np.float32) * acc.astype(np.float32)
            out[h] += term.astype(np.float32)
    return out


def attention_q8_decode(q: np.ndarray, cache, layer: int, n: int, scale: float,
                        kv_head_for_head: Sequence[int]) -> np.ndarray:
    """Decode attention of one new row over a q8_0 cache holding n rows
    (13.4's integer score path): q8_scores, the 1/sqrt(d) scale and a
    max-subtracted softmax in f64, then the weighted sum of the dequantised
    V rows. Returns [1, nh, d] f32."""
    s = q8_scores(np.asarray(q, np.float32)[0], cache.kq[layer, :n], cache.kd[layer, :n], kv_head_for_head)
    s = s * float(scale)
    s -= np.max(s, axis=1, keepdims=True)
    p = np.exp(s)
    p /= np.sum(p, axis=1, keepdims=True)
    v64 = cache.v[layer, :n].astype(np.float64)                                # [n, nkv, d]
    nh, d = p.shape[0], v64.shape[2]
    out = np.empty((1, nh, d), dtype=np.float64)
    for h in range(nh):
        out[0, h] = p[h] @ v64[:, kv_head_for_head[h], :]
    return out.astype(np.float32)


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z * sigmoid(z) = z / (1 + e^-z), f64 (12.3.6)."""
    z64 = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z64 / (1.0 + np.exp(-z64))


def swiglu(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """silu(gate) * up, elementwise, rounded to f32 (12.3.6)."""
    return (silu(gate) * np.asarray(up, np.float32).astype(np.float64)).astype(np.float32)


def add_f32(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Residual add of two f32 tensors (12.3.7)."""
    return (np.asarray(a, np.float32).astype(np.float64)
            + np.asarray(b, np.float32).astype(np.float64)).astype(np.float32)


def argmax_lowest(logits: np.ndarray) -> int:
    """Greedy pick: the largest logit, the lowest index among equals (12.6).

    NaN logits are an error.
    """
    lg = np.asarray(logits)
    if np.isnan(lg).any():
        raise NonFiniteValue("NaN logit")
    return int(np.argmax(lg))


# ---------------------------------------------------------------------------
# Linear layers over dequantised Q8_0 weights
# ---------------------------------------------------------------------------

class QLinear:
    """A Q8_0 weight [out][in] for f64 matmuls.

    Storage only, never arithmetic: keep_f64 holds the dequantised matrix in
    f64, otherwise in f32, and lazy holds the Q8_0 blocks themselves and
    dequantises a chunk of rows per call (for models whose dequantised
    weights do not fit in host memory). d * q is exact in f32, so the three
    give identical results.
    """

    def __init__(self, blocks: np.ndarray, rows: int, cols: int, keep_f64: bool, lazy: bool = False,
                 wtype: str = "q8_0"):
        if wtype not in ("q8_0", "q4_k"):
            raise InvalidShape(f"weight type {wtype!r}")
        qk, nbytes = (QK8_0, Q8_0_BYTES) if wtype == "q8_0" else (QK_K, Q4_K_BYTES)
        if cols % qk:
            raise InvalidShape(f"in-dimension {cols} is not a multiple of {qk}")
        self.rows, self.cols = rows, cols
        self.lazy = lazy
        self.wtype = wtype
        # the wire blocks themselves, [rows][blocks of the row] (the q8act
        # path reads codes and scales)
        self.blocks = np.asarray(blocks, dtype=np.uint8).reshape(rows, (cols // qk) * nbytes)
        if lazy:
            self.w = None
        else:
            w32 = self._decode(self.blocks.reshape(-1), rows)
            self.w = w32.astype(np.float64) if keep_f64 else w32

    def _decode(self, blocks: np.ndarray, rows: int) -> np.ndarray:
        if self.wtype == "q4_k":
            return q4_k_dequantize(blocks, rows * self.cols).reshape(rows, self.cols)
        return matrix_from_blocks(blocks, rows, self.cols)

    def _rows32(self, r0: int, r1: int) -> np.ndarray:
        if self.lazy:
            return self._decode(self.blocks[r0:r1].reshape(-1), r1 - r0)
        return self.w[r0:r1]

    def __call__(self, x: np.ndarray) -> np.ndarray:
        """y[m, n] = sum_k W[n, k] x[m, k] in f64 (a library matmul), f32 out."""
        x64 = np.asarray(x, np.float32).astype(np.float64)
        if self.w is not None and self.w.dtype == np.float64:
            return (x64 @ self.w.T).astype(np.float32)
        out = np.empty((x64.shape[0], self.rows), dtype=np.float32)
        step = 8192
        for r0 in range(0, self.rows, step):
            r1 = min(self.rows, r0 + step)
            wc = self._rows32(r0, r1).astype(np.float64)
            out[:, r0:r1] = (x64 @ wc.T).astype(np.float32)
        return out

    def q8act(self, x: np.ndarray) -> np.ndarray:
        """The pages' quantized matmul ("Model files and quantization", 11.9,
        dotBlocks): each f32 input row is encoded to Q8_0 blocks by the 11.7
        encoder; each (weight block, activation block) pair contributes the
        i32 dot of their codes times w.d * a.d, evaluated in f32 as the page's
        dotBlocks writes it ((w.d * a.d) * f32(acc)); the per-block results of
        a row sum in f64. f32 out.

        Reading of the pages: dotBlocks fixes the per-block arithmetic; the
        sum over a row's blocks is not shown, and is done in f64 like every
        other reduction here.
        """
        if self.wtype != "q8_0":
            raise InvalidShape("the q8_0-activation path takes Q8_0 weights")
        x32 = np.asarray(x, np.float32)
        if x32.ndim != 2 or x32.shape[1] != self.cols:
            raise InvalidShape(f"q8act input {x32.shape} for a [{self.rows}, {self.cols}] weight")
        M, nb = x32.shape[0], self.cols // QK8_0
        _, qa, da16 = q8_0_quantize_parts(x32.reshape(-1))
        qa = qa.reshape(M, nb, QK8_0).astype(np.float64)         # codes, exact in f64
        da = da16.astype(np.float32).reshape(M, nb)
        out = np.empty((M, self.rows), dtype=np.float32)
        step = 8192
        for r0 in range(0, self.rows, step):
            r1 = min(self.rows, r0 + step)
            wd16, wq = q8_0_unpack(self.blocks[r0:r1].reshape(-1), (r1 - r0) * self.cols)
            wd = wd16.astype(np.float32).reshape(r1 - r0, nb)
            wq = wq.reshape(r1 - r0, nb, QK8_0).astype(np.float64)
            acc_sum = np.zeros((M, r1 - r0), dtype=np.float64)
            for b in range(nb):
                acc = qa[:, b, :] @ wq[:, b, :].T                    # integer dots (|acc| < 2^19: exact)
                scale = (wd[None, :, b] * da[:, b, None]).astype(np.float32)   # w.d * a.d in f32
                acc_sum += (scale * acc.astype(np.float32)).astype(np.float32)
            out[:, r0:r1] = acc_sum.astype(np.float32)
        return out

    def row(self, r: np.ndarray) -> np.ndarray:
        """Rows of the dequantised matrix as f32 (the embedding gather)."""
        if self.lazy:
            rr = np.asarray(r, dtype=np.int64).reshape(-1)
            return np.stack([self._rows32(int(i), int(i) + 1)[0] for i in rr]).astype(np.float32)
        return np.asarray(self.w[r], dtype=np.float32)


# ---------------------------------------------------------------------------
# KV cache -- course 12.4 and reference 13.4
# ---------------------------------------------------------------------------

class KvCache:
    """Per-layer K and V, each [capacity, kv_heads, head_dim].

    K is stored after the Q/K norm and RoPE, V as projected. append_layer
    writes at rows len.. without moving len; advance(m) moves it once per
    forward; truncate(keep) rewinds by a single store.

    dtype "f32" (the workloads' cache) or "f16", the course's default cache
    type ("A transformer from scratch", 12.4): appended rows are rounded to
    IEEE half (nearest even) and read back exactly as f32; or "q8_0" ("The
    LLM stack", 13.4; 12.4): each (position, kv head) row is stored as
    head_dim/32 Q8_0 blocks by the 11.7 encoder (codes in kq/vq, f16 scales
    in kd/vd; k and v hold the dequantised rows f32(d) * q that every reader
    sees). head_dim must be a multiple of 32.
    """

    def __init__(self, n_layers: int, n_kv_heads: int, head_dim: int, capacity: int, dtype: str = "f32"):
        if dtype not in ("f32", "f16", "q8_0"):
            raise InvalidShape(f"KV cache dtype {dtype!r}")
        if dtype == "q8_0" and head_dim % QK8_0:
            raise InvalidShape(f"a q8_0 KV cache needs head_dim % {QK8_0} == 0, got {head_dim}")
        self.capacity = capacity
        self.dtype = dtype
        np_t = np.float16 if dtype == "f16" else np.float32
        self.k = np.zeros((n_layers, capacity, n_kv_heads, head_dim), np_t)
        self.v = np.zeros((n_layers, capacity, n_kv_heads, head_dim), np_t)
        if dtype == "q8_0":
            nb = head_dim // QK8_0
            self.kq = np.zeros((n_layers, capacity, n_kv_heads, head_dim), np.int8)
            self.vq = np.zeros((n_layers, capacity, n_kv_heads, head_dim), np.int8)
            self.kd = np.zeros((n_layers, capacity, n_kv_heads, nb), np.float16)
            self.vd = np.zeros((n_layers, capacity, n_kv_heads, nb), np.float16)
        self.len = 0

    def _store_q8(self, codes, scales, deq, layer: int, rows: np.ndarray) -> None:
        m, nkv, d = rows.shape
        _, q, d16 = q8_0_quantize_parts(np.asarray(rows, np.float32).reshape(-1))
        q = q.reshape(m, nkv, d)
        d16 = d16.reshape(m, nkv, d // QK8_0)
        codes[layer, self.len:self.len + m] = q
        scales[layer, self.len:self.len + m] = d16
        deq[layer, self.len:self.len + m] = (np.repeat(d16.astype(np.float32), QK8_0, axis=2)
                                             * q.astype(np.float32)).astype(np.float32)

    def append_layer(self, layer: int, k_rows: np.ndarray, v_rows: np.ndarray) -> None:
        m = k_rows.shape[0]
        if self.len + m > self.capacity:
            raise KvCacheOverflow(f"len {self.len} + {m} > capacity {self.capacity}")
        if self.dtype == "q8_0":
            self._store_q8(self.kq, self.kd, self.k, layer, k_rows)
            self._store_q8(self.vq, self.vd, self.v, layer, v_rows)
            return
        # numpy's f32 -> f16 conversion rounds to nearest even
        self.k[layer, self.len:self.len + m] = np.asarray(k_rows, np.float32).astype(self.k.dtype)
        self.v[layer, self.len:self.len + m] = np.asarray(v_rows, np.float32).astype(self.v.dtype)

    def advance(self, m: int) -> None:
        if self.len + m > self.capacity:
            raise KvCacheOverflow(f"len {self.len} + {m} > capacity {self.capacity}")
        self.len += m

    def truncate(self, keep_len: int) -> None:
        if keep_len < self.len:
            self.len = keep_len

    def reset(self) -> None:
        self.len = 0

    def layer_rows(self, layer: int, n: int):
        return self.k[layer, :n].astype(np.float32), self.v[layer, :n].astype(np.float32)


# ---------------------------------------------------------------------------
# The model
# ---------------------------------------------------------------------------

@dataclass
class _Layer:
    attn_norm: np.ndarray
    wq: QLinear
    wk: QLinear
    wv: QLinear
    q_norm: np.ndarray
    k_norm: np.ndarray
    wo: QLinear
    ffn_norm: np.ndarray
    wg: QLinear
    wu: QLinear
    wd: QLinear


class OracleModel:
    """The dense Qwen3 decoder over Q8_0 weights (course 12.3, minfer 1-2).

    `shape` carries vocab, hidden, n_layers, n_heads, n_kv_heads, head_dim,
    intermediate, rms_eps, rope_theta and tied. `tensors` maps GGUF names to
    Q8_0 wire bytes (linear weights) or f32 arrays (norm weights).
    """

    F64_BUDGET_BYTES = 12 << 30

    def __init__(self, shape, tensors: dict, keep_f64: bool | None = None, lazy: bool = False,
                 wtype: str = "q8_0"):
        s = shape
        self.shape = s
        if s.head_dim % 2:
            raise InvalidShape("head_dim must be even for the half-layout RoPE")
        self.kv_head_for_head = kv_head_map(s.n_heads, s.n_kv_heads)
        n_params = s.vocab * s.hidden * (1 if s.tied else 2) + s.n_layers * (
            s.hidden * (2 * s.q_width + 2 * s.kv_width) + 3 * s.hidden * s.intermediate)
        if keep_f64 is None:
            keep_f64 = n_params * 8 <= self.F64_BUDGET_BYTES

        def lin(name, rows, cols):
            return QLinear(tensors[name], rows, cols, keep_f64, lazy, wtype)

        def norm(name, n):
            w = np.asarray(tensors[name], np.float32)
            if w.shape != (n,):
                raise InvalidShape(f"{name}: expected [{n}], got {list(w.shape)}")
            return w

        self.tok_embd = lin("token_embd", s.vocab, s.hidden)
        self.layers = []
        for i in range(s.n_layers):
            p = f"blk.{i}."
            self.layers.append(_Layer(
                attn_norm=norm(p + "attn_norm", s.hidden),
                wq=lin(p + "attn_q", s.q_width, s.hidden),
                wk=lin(p + "attn_k", s.kv_width, s.hidden),
                wv=lin(p + "attn_v", s.kv_width, s.hidden),
                q_norm=norm(p + "attn_q_norm", s.head_dim),
                k_norm=norm(p + "attn_k_norm", s.head_dim),
                wo=lin(p + "attn_output", s.hidden, s.q_width),
                ffn_norm=norm(p + "ffn_norm", s.hidden),
                wg=lin(p + "ffn_gate", s.intermediate, s.hidden),
                wu=lin(p + "ffn_up", s.intermediate, s.hidden),
                wd=lin(p + "ffn_down", s.hidden, s.intermediate),
            ))
        self.output_norm = norm("output_norm", s.hidden)
        # tied lm_head: no output.weight means the embedding table is reused
        self.output = self.tok_embd if s.tied else lin("output", s.vocab, s.hidden)
        self.act = "f32"

    def set_activations(self, kind: str) -> "OracleModel":
        """How the linear layers take their inputs: "f32" (the workloads'
        path, f64 dots over f32 activations) or "q8_0" (the pages' CPU path,
        "Model files and quantization" 11.9: activations re-quantized to Q8_0
        per row per call, integer block dots; QLinear.q8act). The embedding
        gather is a dequantising row lookup either way."""
        if kind not in ("f32", "q8_0"):
            raise InvalidShape(f"activation kind {kind!r}")
        self.act = kind
        return self

    def _lin(self, W: QLinear, x: np.ndarray) -> np.ndarray:
        return W.q8act(x) if self.act == "q8_0" else W(x)

    @classmethod
    def from_f32(cls, shape, weights: dict, keep_f64: bool | None = None, wtype: str = "q8_0") -> "OracleModel":
        """Quantise f32 linear weights (the embedding included) with this
        module's Q8_0 or Q4_K encoder."""
        from quantized_transformer_decode_gb300.inputs import tensor_specs
        enc = q8_0_quantize if wtype == "q8_0" else q4_k_quantize
        tensors = {}
        for name, kind, _ in tensor_specs(shape):
            w = weights[name]
            tensors[name] = enc(w) if kind == "linear" else np.asarray(w, np.float32)
        return cls(shape, tensors, keep_f64, wtype=wtype)

    @classmethod
    def from_f32_stream(cls, shape, named_weights) -> "OracleModel":
        """The same model from an iterator of (name, f32 tensor): each linear
        weight is quantised as it arrives and only its Q8_0 blocks are kept
        (lazy storage), so a model far larger than host memory in f32 fits."""
        from quantized_transformer_decode_gb300.inputs import tensor_specs
        kinds = {name: kind for name, kind, _ in tensor_specs(shape)}
        tensors = {}
        for name, w in named_weights:
            tensors[name] = q8_0_quantize(w) if kinds[name] == "linear" else np.asarray(w, np.float32)
            del w
        return cls(shape, tensors, keep_f64=False, lazy=True)

    def new_cache(self, capacity: int, dtype: str = "f32") -> KvCache:
        s = self.shape
        return KvCache(s.n_layers, s.n_kv_heads, s.head_dim, capacity, dtype)

    # -- blocks -------------------------------------------------------------

    def _attention_block(self, li: int, lw: _Layer, x, positions, cache: KvCache):
        s = self.shape
        M = x.shape[0]
        h = rms_norm(x, lw.attn_norm, s.rms_eps)
        q = self._lin(lw.wq, h).reshape(M, s.n_heads, s.head_dim)
        k = self._lin(lw.wk, h).reshape(M, s.n_kv_heads, s.head_dim)
        v = self._lin(lw.wv, h).reshape(M, s.n_kv_heads, s.head_dim)
        q = rope_neox(rms_norm(q, lw.q_norm, s.rms_eps), positions, s.rope_theta)
        k = rope_neox(rms_norm(k, lw.k_norm, s.rms_eps), positions, s.rope_theta)
        cache.append_layer(li, k, v)
        scale = 1.0 / math.sqrt(s.head_dim)
        if cache.dtype == "q8_0" and M == 1:
            # one new row: the integer score path (13.4); a multi-row step
            # (prefill, verify) reads the dequantised rows instead
            o = attention_q8_decode(q, cache, li, cache.len + 1, scale, self.kv_head_for_head)
        else:
            kk, vv = cache.layer_rows(li, cache.len + M)
            o = attention(q, kk, vv, positions, scale, self.kv_head_for_head)
        return add_f32(x, self._lin(lw.wo, o.reshape(M, s.q_width)))

    def _ffn_block(self, lw: _Layer, x):
        s = self.shape
        h2 = rms_norm(x, lw.ffn_norm, s.rms_eps)
        return add_f32(x, self._lin(lw.wd, swiglu(self._lin(lw.wg, h2), self._lin(lw.wu, h2))))

    # -- entry points -------------------------------------------------------

    def forward(self, cache: KvCache, tokens, pos0: int, all_logits: bool = False):
        """Append len(tokens) rows at pos0 and return logits (12.3, 12.4).

        pos0 must equal cache.len (else InvalidSequenceLength) and the rows
        must fit (else KvCacheOverflow). Returns the last row's logits [vocab]
        unless all_logits, then [M, vocab]. The cache length moves once, after
        the layer loop.
        """
        s = self.shape
        tok = np.asarray(tokens, dtype=np.int64).reshape(-1)
        M = tok.size
        if M == 0:
            raise InvalidShape("empty token list")
        if pos0 != cache.len:
            raise InvalidSequenceLength(f"pos0 {pos0} != cache length {cache.len}")
        if cache.len + M > cache.capacity:
            raise KvCacheOverflow(f"len {cache.len} + {M} > capacity {cache.capacity}")
        if tok.min() < 0 or tok.max() >= s.vocab:
            raise InvalidShape("token id out of range")
        positions = np.arange(pos0, pos0 + M)
        x = self.tok_embd.row(tok)
        for li, lw in enumerate(self.layers):
            x = self._attention_block(li, lw, x, positions, cache)
            x = self._ffn_block(lw, x)
        cache.advance(M)
        xf = rms_norm(x, self.output_norm, s.rms_eps)
        if all_logits:
            return self._lin(self.output, xf)
        return self._lin(self.output, xf[-1:])[0]

    def generate_greedy(self, cache: KvCache, prompt, n_steps: int):
        """Prefill the prompt, then n_steps greedy decode steps (12.6).

        Returns (ids, logits): ids[0] is the prefill's argmax and ids[s] the
        argmax of decode step s, which was fed ids[s-1] at position
        len(prompt) + s - 1; logits[s] is the row each id was taken from.
        """
        lg = self.forward(cache, prompt, cache.len)
        ids = [argmax_lowest(lg)]
        logits = [lg]
        for _ in range(n_steps):
            lg = self.forward(cache, [ids[-1]], cache.len)
            ids.append(argmax_lowest(lg))
            logits.append(lg)
        return ids, logits

    def teacher_forced(self, cache: KvCache, prompt, fed_ids: Sequence[int]):
        """Prefill, then decode the given ids one by one; return every logits row."""
        out = [self.forward(cache, prompt, cache.len)]
        for t in fed_ids:
            out.append(self.forward(cache, [int(t)], cache.len))
        return out
