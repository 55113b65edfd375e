"""Cacheless float64 brute-force forward pass, used to pin the oracle.

Written separately from the oracle: it parses the Q8_0 wire bytes itself,
keeps every tensor in f64 (no f32 storage anywhere), holds no KV cache and
recomputes the whole sequence for every query -- the "cacheless entry" that
"A transformer from scratch" (section 12.4, contract 3) names as the oracle for
the cached path. Attention is an explicit loop over query and key positions.
Small configurations only.
"""
from __future__ import annotations

import math
import struct

import numpy as np


def dequant_rows(wire: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Parse [rows][cols/32] Q8_0 blocks (f16 d, 32 x int8) into f64 [rows, cols]."""
    raw = bytes(np.ascontiguousarray(wire, dtype=np.uint8))
    nb = cols // 32
    out = np.empty((rows, cols), dtype=np.float64)
    for r in range(rows):
        for b in range(nb):
            off = (r * nb + b) * 34
            (d,) = struct.unpack_from("<e", raw, off)
            qs = struct.unpack_from("<32b", raw, off + 2)
            out[r, b * 32:(b + 1) * 32] = np.array(qs, dtype=np.float64) * d
    return out


def _norm(v: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    rms = math.sqrt(float(np.dot(v, v)) / v.size + eps)
    return v / rms * w


def _rotate_half(v: np.ndarray, p: int, theta: float) -> np.ndarray:
    d = v.size
    out = v.copy()
    for i in range(d // 2):
        ang = p / theta ** (2.0 * i / d)
        a, b = v[i], v[i + d // 2]
        out[i] = a * math.cos(ang) - b * math.sin(ang)
        out[i + d // 2] = a * math.sin(ang) + b * math.cos(ang)
    return out


class BruteForceModel:
    def __init__(self, shape, tensors: dict):
        s = shape
        self.s = s
        f64 = lambda n: np.asarray(tensors[n], dtype=np.float64)  # noqa: E731
        self.E = dequant_rows(tensors["token_embd"], s.vocab, s.hidden)
        self.out = self.E if s.tied else dequant_rows(tensors["output"], s.vocab, s.hidden)
        self.out_norm = f64("output_norm")
        self.L = []
        for i in range(s.n_layers):
            p = f"blk.{i}."
            self.L.append(dict(
                an=f64(p + "attn_norm"), qn=f64(p + "attn_q_norm"), kn=f64(p + "attn_k_norm"),
                fn=f64(p + "ffn_norm"),
                q=dequant_rows(tensors[p + "attn_q"], s.q_width, s.hidden),
                k=dequant_rows(tensors[p + "attn_k"], s.kv_width, s.hidden),
                v=dequant_rows(tensors[p + "attn_v"], s.kv_width, s.hidden),
                o=dequant_rows(tensors[p + "attn_output"], s.hidden, s.q_width),
                g=dequant_rows(tensors[p + "ffn_gate"], s.intermediate, s.hidden),
                u=dequant_rows(tensors[p + "ffn_up"], s.intermediate, s.hidden),
                d=dequant_rows(tensors[p + "ffn_down"], s.hidden, s.intermediate)))

    def last_logits(self, tokens) -> np.ndarray:
        """Logits of the last position, recomputing every position from scratch."""
        s = self.s
        hd, nh, nkv = s.head_dim, s.n_heads, s.n_kv_heads
        group = nh // nkv
        T = len(tokens)
        xs = [self.E[int(t)].copy() for t in tokens]
        for lw in self.L:
            qs, ks, vs = [], [], []
            for p in range(T):
                h = _norm(xs[p], lw["an"], s.rms_eps)
                q, k, v = lw["q"] @ h, lw["k"] @ h, lw["v"] @ h
                qs.append([_rotate_half(_norm(q[j * hd:(j + 1) * hd], lw["qn"], s.rms_eps), p, s.rope_theta)
                           for j in range(nh)])
                ks.append([_rotate_half(_norm(k[j * hd:(j + 1) * hd], lw["kn"], s.rms_eps), p, s.rope_theta)
                           for j in range(nkv)])
                vs.append([v[j * hd:(j + 1) * hd] for j in range(nkv)])
            for p in range(T):
                o = np.zeros(nh * hd)
                for j in range(nh):
                    g = j // group
                    sc = [float(np.dot(qs[p][j], ks[t][g])) / math.sqrt(hd) for t in range(p + 1)]
                    m = max(sc)
                    e = [math.exp(z - m) for z in sc]
                    tot = sum(e)
                    acc = np.zeros(hd)
                    for t in range(p + 1):
                        acc += (e[t] / tot) * vs[t][g]
                    o[j * hd:(j + 1) * hd] = acc
                xs[p] = xs[p] + lw["o"] @ o
            for p in range(T):
                h2 = _norm(xs[p], lw["fn"], s.rms_eps)
                gt, up = lw["g"] @ h2, lw["u"] @ h2
                act = np.array([z / (1.0 + math.exp(-z)) for z in gt]) * up
                xs[p] = xs[p] + lw["d"] @ act
        return self.out @ _norm(xs[-1], self.out_norm, s.rms_eps)
