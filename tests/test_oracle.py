"""Pins for the CPU oracle: closed forms, invariants, the pages' worked examples,
library routines for special cases and an f64 cacheless brute force.

None of these re-types an oracle formula and compares it with itself; each
check would fail on a plausible slip (a dropped term, a wrong sign, pairing or
index, a transposed operand, the other tie rule).
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

import oracle as orc
from conftest import golden
from quantized_transformer_decode_gb300 import inputs


# ----------------------------------------------------------------- Q8_0 codec

def test_q8_0_wire_layout_and_integer_block():
    # amax 127 gives d = 1.0 exactly (f16 bits 0x3C00, little endian) and the
    # integers encode as themselves: 34 bytes, scale first (section 11.7).
    spec = golden("q8_0_roundtrip.json")
    vals = np.arange(-16, 16, dtype=np.float32)
    vals[0] = -127.0
    b = orc.q8_0_quantize(vals)
    assert b.size == spec["block_bytes"]
    assert b[0] == 0x00 and b[1] == 0x3C
    assert np.array_equal(b[2:].view(np.int8).astype(np.float32), vals)


def test_q8_0_roundtrip_course_bounds():
    spec = golden("q8_0_roundtrip.json")
    for seed in range(20):
        x = inputs.uniform_block_values(seed, 32 * 64)
        d32, q, d16 = orc.q8_0_quantize_parts(x)
        xb = x.reshape(-1, 32).astype(np.float64)
        # course test: within half a step of the f32 scale
        err32 = np.abs(xb - d32[:, None].astype(np.float64) * q)
        assert np.all(err32 <= d32[:, None] / 2 + 1e-6)
        # public seam with the stored f16 scale
        y = orc.q8_0_dequantize(orc.q8_0_quantize(x), x.size).reshape(-1, 32)
        assert np.max(np.abs(y - xb)) <= spec["f16_scale_seam_bound"]
        bound = d32.astype(np.float64) / 2 + 127 * np.abs(d32.astype(np.float64) - d16.astype(np.float64))
        assert np.all(np.abs(y - xb) <= bound[:, None] + 1e-6)


def test_q8_0_zero_block_is_all_zero_bytes():
    b = orc.q8_0_quantize(np.zeros(64, np.float32))
    assert not b.any()


def test_q8_0_ramp_closed_form():
    # v_k = k/31: amax 1, so q_k = round(127 k / 31); 127k/31 is never within
    # 1/62 of a half-integer, far beyond f32 rounding, so exact rationals decide.
    x = (np.arange(32, dtype=np.float32) / np.float32(31)).astype(np.float32)
    _, q, _ = orc.q8_0_quantize_parts(x)
    want = [int(Fraction(127 * k, 31) + Fraction(1, 2)) for k in range(32)]
    assert q[0].tolist() == want
    assert want[-1] == 127 and want[0] == 0


def test_q8_0_single_spike():
    rng = np.random.default_rng(5)
    x = (rng.random(32, dtype=np.float32) * 0.02 - 0.01).astype(np.float32)
    x[7] = -3.0
    _, q, _ = orc.q8_0_quantize_parts(x)
    assert q[0, 7] == -127
    assert np.all(np.delete(q[0], 7) == 0)      # |v| * 127/3 < 0.43


def test_q8_0_exact_ties_round_half_away_from_zero():
    # d = 1 (amax 127), so v * inv_d = v exactly: halves must go away from 0.
    x = np.zeros(32, np.float32)
    x[:8] = [127.0, 2.5, -2.5, 0.5, -0.5, 126.5, 1.5, -1.5]
    _, q, _ = orc.q8_0_quantize_parts(x)
    assert q[0, :8].tolist() == [127, 3, -3, 1, -1, 127, 2, -2]


@pytest.mark.parametrize("amax,bits", [
    (127.0, 0x3C00),                       # d = 1
    (254.0, 0x4000),                       # d = 2
    (127.0 * 2.0 ** -24, 0x0001),          # d = smallest f16 subnormal
    (127.0 * 2.0 ** -25, 0x0000),          # exact tie between 0 and 2^-24 -> even
    (127.0 * 3 * 2.0 ** -25, 0x0002),      # tie between 1 and 2 (x 2^-24) -> even
    (127.0 * 65504.0, 0x7BFF),             # largest finite f16
])
def test_q8_0_f16_scale_is_ieee_round_to_nearest_even(amax, bits):
    x = np.zeros(32, np.float32)
    x[3] = np.float32(amax)
    assert float(np.float32(amax)) == amax
    b = orc.q8_0_quantize(x)
    assert int(b[0]) | (int(b[1]) << 8) == bits


def test_q8_0_tiny_scale_saturates():
    # d subnormal enough that 1/d overflows: nonzero v saturate, zeros stay 0
    x = np.zeros(32, np.float32)
    x[0] = np.float32(1e-38)
    x[1] = np.float32(-5e-39)
    _, q, d16 = orc.q8_0_quantize_parts(x)
    assert q[0, 0] == 127 and q[0, 1] == -127 and np.all(q[0, 2:] == 0)
    assert float(d16[0]) == 0.0


def test_q8_0_errors():
    with pytest.raises(orc.InvalidShape):
        orc.q8_0_quantize(np.zeros(33, np.float32))
    for bad in (np.nan, np.inf, -np.inf):
        x = np.zeros(64, np.float32)
        x[40] = bad
        with pytest.raises(orc.NonFiniteValue):
            orc.q8_0_quantize(x)


def test_q8_0_dequantize_is_scale_times_code():
    x = inputs.uniform_block_values(7, 96)
    b = orc.q8_0_quantize(x).reshape(3, 34)
    y = orc.q8_0_dequantize(b.reshape(-1), 96).reshape(3, 32)
    for i in range(3):
        d = float(np.frombuffer(b[i, :2].tobytes(), "<f2")[0])
        qs = np.frombuffer(b[i, 2:].tobytes(), np.int8)
        assert np.array_equal(y[i], np.array([d * int(c) for c in qs], np.float32))


# ------------------------------------------------------------------- linear

def test_linear_one_hot_selects_a_column_and_brute_force_sum():
    rng = np.random.default_rng(3)
    W = (rng.standard_normal((5, 64)) * 0.02).astype(np.float32)
    lin = orc.QLinear(orc.q8_0_quantize(W), 5, 64, keep_f64=True)
    Wd = orc.matrix_from_blocks(orc.q8_0_quantize(W), 5, 64)
    for j in (0, 31, 32, 63):
        e = np.zeros((1, 64), np.float32)
        e[0, j] = 1.0
        assert np.array_equal(lin(e)[0], Wd[:, j])
    x = rng.standard_normal((2, 64)).astype(np.float32)
    y = lin(x)
    for m in range(2):
        for n in range(5):
            exact = sum(Fraction(float(Wd[n, k])) * Fraction(float(x[m, k])) for k in range(64))
            assert abs(float(y[m, n]) - float(exact)) <= 1e-7 * max(1.0, abs(float(exact)))


def test_linear_f32_storage_matches_f64_storage():
    rng = np.random.default_rng(4)
    W = (rng.standard_normal((9000, 32)) * 0.02).astype(np.float32)
    b = orc.q8_0_quantize(W)
    x = rng.standard_normal((3, 32)).astype(np.float32)
    assert np.array_equal(orc.QLinear(b, 9000, 32, True)(x), orc.QLinear(b, 9000, 32, False)(x))


# ------------------------------------------------------------------ RMSNorm

def test_rms_norm_constant_vector_closed_form():
    rng = np.random.default_rng(1)
    w = (1 + 0.1 * rng.standard_normal(64)).astype(np.float32)
    c = 0.37
    y = orc.rms_norm(np.full(64, c, np.float32), w, 1e-6)
    cc = float(np.float32(c))
    want = cc / math.sqrt(cc * cc + 1e-6) * w.astype(np.float64)
    assert np.allclose(y, want, rtol=1e-7, atol=0)


def test_rms_norm_unit_rms_scale_invariance_and_zero():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, 128)).astype(np.float32) * 3
    y = orc.rms_norm(x, np.ones(128, np.float32), 1e-6).astype(np.float64)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, atol=1e-6)
    y2 = orc.rms_norm(x * 1000, np.ones(128, np.float32), 1e-6)
    assert np.allclose(y, y2, rtol=1e-6, atol=1e-7)
    assert not orc.rms_norm(np.zeros(8, np.float32), np.ones(8, np.float32), 1e-6).any()


def test_rms_norm_per_head_groups_last_axis():
    # per-head Q/K norm (minfer 2.2): each head normalised on its own
    x = np.ones((1, 3, 4), np.float32) * np.array([1.0, 10.0, 100.0], np.float32)[None, :, None]
    y = orc.rms_norm(x, np.ones(4, np.float32), 0.0)
    assert np.allclose(y, 1.0)


# --------------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    x = np.random.default_rng(0).standard_normal((1, 3, 128)).astype(np.float32)
    assert np.array_equal(orc.rope_neox(x, [0], 1e6), x)


def test_rope_pair_zero_turns_one_radian_per_position():
    x = np.zeros((1, 1, 128), np.float32)
    x[0, 0, 0] = 1.0
    y = orc.rope_neox(x, [1], 1e6)[0, 0]
    assert y[0] == np.float32(math.cos(1.0)) and y[64] == np.float32(math.sin(1.0))
    assert np.count_nonzero(y) == 2          # half layout: channel 0 pairs with 64


@pytest.mark.parametrize("i", [1, 5, 63])
def test_rope_pair_frequency(i):
    # theta = 1e6, d = 128: f_i = 1e6^(-2i/128) = 10^(-12 i / 128)
    p = 37
    x = np.zeros((1, 1, 128), np.float32)
    x[0, 0, i + 64] = 1.0
    y = orc.rope_neox(x, [p], 1e6)[0, 0]
    ang = p * 10.0 ** (-12.0 * i / 128.0)
    # (a, b) = (0, 1) -> (-sin, cos)
    assert abs(y[i] + math.sin(ang)) < 1e-7 and abs(y[i + 64] - math.cos(ang)) < 1e-7


def test_rope_preserves_norm():
    x = np.random.default_rng(8).standard_normal((6, 4, 128)).astype(np.float32)
    y = orc.rope_neox(x, np.arange(100, 106), 1e6)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-6)


def test_rope_relative_position_course_numbers():
    g = golden("rope_relative_position.json")
    q = np.array(g["q"], np.float32).reshape(1, 1, 2)
    k = np.array(g["k"], np.float32).reshape(1, 1, 2)

    def score(pq, pk):
        a = orc.rope_neox(q, [pq], 1e6).astype(np.float64)
        b = orc.rope_neox(k, [pk], 1e6).astype(np.float64)
        return float(np.sum(a * b))

    s = [score(*pp) for pp in g["equal_pairs"]]
    assert abs(s[0] - s[1]) <= g["equal_tolerance"] and abs(s[0] - s[2]) <= g["equal_tolerance"]
    assert abs(s[0] - score(*g["different_pair"])) > g["different_min_gap"]


# ---------------------------------------------------------------- attention

def test_gqa_map_pages_example():
    g = golden("gqa_map.json")
    m = orc.kv_head_map(g["n_heads"], g["n_kv_heads"])
    for h, kv in g["head_to_kv"].items():
        assert m[int(h)] == kv
    assert orc.kv_head_map(32, 8)[:8] == [0, 0, 0, 0, 1, 1, 1, 1]


def test_attention_single_position_returns_v():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((1, 4, 16)).astype(np.float32)
    k = rng.standard_normal((1, 2, 16)).astype(np.float32)
    v = rng.standard_normal((1, 2, 16)).astype(np.float32)
    o = orc.attention(q, k, v, [0], 0.25, orc.kv_head_map(4, 2))
    assert np.array_equal(o[0, 0], v[0, 0]) and np.array_equal(o[0, 3], v[0, 1])


def test_attention_zero_query_is_mean_of_visible_values():
    rng = np.random.default_rng(10)
    T = 7
    k = rng.standard_normal((T, 1, 8)).astype(np.float32)
    v = rng.standard_normal((T, 1, 8)).astype(np.float32)
    q = np.zeros((2, 1, 8), np.float32)
    o = orc.attention(q, k, v, [2, 6], 1.0, [0])
    assert np.allclose(o[0, 0], v[:3, 0].astype(np.float64).mean(0), atol=1e-7)
    assert np.allclose(o[1, 0], v[:, 0].astype(np.float64).mean(0), atol=1e-7)


def test_attention_two_keys_sigmoid_with_scale():
    hd = 128
    q = np.zeros((1, 1, hd), np.float32)
    k = np.zeros((2, 1, hd), np.float32)
    v = np.zeros((2, 1, hd), np.float32)
    q[0, 0, 0] = 2.0
    k[0, 0, 0], k[1, 0, 0] = 3.0, -1.0
    v[0, 0, 1], v[1, 0, 2] = 1.0, 1.0
    o = orc.attention(q, k, v, [1], 1.0 / math.sqrt(hd), [0])
    s0, s1 = 6.0 / math.sqrt(hd), -2.0 / math.sqrt(hd)
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    assert abs(o[0, 0, 1] - w0) < 1e-7 and abs(o[0, 0, 2] - (1 - w0)) < 1e-7


def test_attention_is_causal():
    rng = np.random.default_rng(11)
    k = rng.standard_normal((5, 1, 8)).astype(np.float32)
    v = rng.standard_normal((5, 1, 8)).astype(np.float32)
    q = rng.standard_normal((1, 1, 8)).astype(np.float32)
    o1 = orc.attention(q, k, v, [0], 0.3, [0])
    k[1:] *= 50
    v[1:] = 7
    assert np.array_equal(o1, orc.attention(q, k, v, [0], 0.3, [0]))
    assert np.array_equal(o1[0, 0], v[0, 0])


# ----------------------------------------------------------- SwiGLU, argmax

def test_silu_matches_library_logistic():
    z = np.linspace(-40, 40, 1001)
    assert np.allclose(orc.silu(z), z * scipy.special.expit(z), rtol=1e-14, atol=1e-300)
    assert orc.silu(np.array([0.0]))[0] == 0.0
    g = np.array([1.0, -2.0], np.float32)
    u = np.array([3.0, 0.5], np.float32)
    assert np.allclose(orc.swiglu(g, u), g * scipy.special.expit(g.astype(np.float64)) * u, rtol=1e-7)


def test_argmax_pages_example_ties_and_nan():
    g = golden("greedy_argmax.json")
    assert orc.argmax_lowest(np.array(g["logits"], np.float32)) == g["argmax"]
    assert orc.argmax_lowest(np.array([1.0, 3.0, 3.0, 2.0])) == 1
    with pytest.raises(orc.NonFiniteValue):
        orc.argmax_lowest(np.array([0.0, np.nan]))


# ----------------------------------------------------------------- KV cache

def test_kv_cache_contract_pages_example():
    g = golden("kv_cache_contract.json")
    c = orc.KvCache(g["n_layers"], g["kv_heads"], g["head_dim"], g["capacity"])
    k = np.full((g["append_rows"], g["kv_heads"], g["head_dim"]), g["k_fill"], np.float32)
    v = np.full_like(k, g["v_fill"])
    c.append_layer(0, k, v)
    assert c.len == g["len_after_append_before_advance"]
    c.advance(g["append_rows"])
    assert c.len == g["len_after_advance"]
    assert c.layer_rows(0, c.len)[0].size == g["k_slice_elements"]
    c.truncate(g["truncate_to"])
    assert c.len == g["len_after_truncate"]
    c.truncate(5)                      # at or above len: no-op
    assert c.len == 1
    with pytest.raises(orc.KvCacheOverflow):
        c.append_layer(0, np.zeros((8, 2, 4), np.float32), np.zeros((8, 2, 4), np.float32))


# -------------------------------------------------------------- whole model

def test_qwen3_0_6b_projection_widths():
    g = golden("qwen3_widths.json")
    s = inputs.QWEN3_0_6B
    cfg = g["config"]
    assert (s.vocab, s.hidden, s.intermediate, s.n_layers, s.n_heads, s.n_kv_heads, s.head_dim) == (
        cfg["vocab"], cfg["hidden"], cfg["intermediate"], cfg["n_layers"], cfg["n_heads"],
        cfg["n_kv_heads"], cfg["head_dim"])
    small = inputs.Qwen3Shape(vocab=64, hidden=1024, n_layers=1, n_heads=16, n_kv_heads=8,
                              head_dim=128, intermediate=3072)
    m = orc.OracleModel.from_f32(small, inputs.generate_weights(small, 0))
    lw = m.layers[0]
    assert lw.wq.rows == g["q_width"] and lw.wk.rows == g["kv_width"] and lw.wv.rows == g["kv_width"]
    assert (lw.wo.rows, lw.wo.cols) == (1024, g["q_width"])
    for name, ne in g["gguf_ne"].items():
        obj = getattr(lw, {"attn_q": "wq", "attn_k": "wk", "attn_v": "wv", "attn_output": "wo",
                           "ffn_gate": "wg", "ffn_up": "wu", "ffn_down": "wd"}.get(name, "x"), None)
        if obj is not None:                       # GGUF ne order is [in, out]
            assert [obj.cols, obj.rows] == ne
    kv_f16 = s.n_layers * 2 * s.n_kv_heads * s.head_dim * 2
    assert kv_f16 == g["kv_bytes_per_position_f16"]
    c = m.new_cache(4)
    assert m.forward(c, [1, 2], 0).shape == (64,)


def _rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


SMALL_SHAPES = [
    inputs.Qwen3Shape(vocab=96, hidden=64, n_layers=1, n_heads=4, n_kv_heads=1, head_dim=32,
                      intermediate=96, tied=True),
    inputs.Qwen3Shape(vocab=80, hidden=96, n_layers=2, n_heads=2, n_kv_heads=2, head_dim=32,
                      intermediate=64, tied=False, rope_theta=10000.0),
    inputs.Qwen3Shape(vocab=64, hidden=128, n_layers=1, n_heads=6, n_kv_heads=3, head_dim=64,
                      intermediate=160, tied=False, rms_eps=1e-5),
]


@pytest.mark.parametrize("shape", SMALL_SHAPES)
def test_oracle_matches_f64_cacheless_brute_force_small(shape):
    from bruteforce_f64 import BruteForceModel
    w = inputs.generate_weights(shape, 11)
    m = orc.OracleModel.from_f32(shape, w)
    tensors = {n: (orc.q8_0_quantize(a) if k == "linear" else a)
               for n, k, _ in inputs.tensor_specs(shape) for a in [w[n]]}
    bf = BruteForceModel(shape, tensors)
    toks = inputs.prompt_tokens(shape, 11, 9)
    c = m.new_cache(12)
    got = [m.forward(c, toks[:5], 0)]
    for t in toks[5:]:
        got.append(m.forward(c, [t], c.len))
    for j, lg in enumerate(got):
        want = bf.last_logits(toks[:5 + j])
        assert _rel_l2(lg, want) < 2e-6, j
        assert np.max(np.abs(lg - want)) < 1e-5


def test_oracle_matches_f64_cacheless_brute_force_tiny_config():
    from bruteforce_f64 import BruteForceModel
    wl = inputs.WORKLOADS["tiny"]
    s = wl.shape
    w = inputs.generate_weights(s, wl.seed)
    m = orc.OracleModel.from_f32(s, w)
    tensors = {n: (orc.q8_0_quantize(w[n]) if k == "linear" else w[n]) for n, k, _ in inputs.tensor_specs(s)}
    bf = BruteForceModel(s, tensors)
    prompt = inputs.prompt_tokens(s, wl.seed, wl.prompt_len)
    n_steps = 4
    ids, logits = m.generate_greedy(m.new_cache(64), prompt, n_steps)
    seq = list(prompt)
    for j in range(n_steps + 1):
        want = bf.last_logits(seq)
        assert _rel_l2(logits[j], want) < 2e-6
        assert np.max(np.abs(logits[j] - want)) < 1e-5
        assert ids[j] == int(np.argmax(want))
        seq.append(ids[j])


def test_cached_equals_uncached_and_contract_errors():
    s = SMALL_SHAPES[0]
    m = orc.OracleModel.from_f32(s, inputs.generate_weights(s, 3))
    toks = inputs.prompt_tokens(s, 3, 10)
    c1 = m.new_cache(10)
    full = m.forward(c1, toks, 0, all_logits=True)
    c2 = m.new_cache(10)
    rows = [m.forward(c2, toks[:4], 0, all_logits=True)]
    for t in toks[4:]:
        rows.append(m.forward(c2, [t], c2.len, all_logits=True))
    inc = np.concatenate(rows, axis=0)
    assert np.max(np.abs(inc - full)) < 1e-6
    # K cache rows are identical either way (per-token projections and RoPE)
    assert np.max(np.abs(c1.k - c2.k)) < 1e-6
    with pytest.raises(orc.InvalidSequenceLength):
        m.forward(c2, [1], 3)
    with pytest.raises(orc.KvCacheOverflow):
        m.forward(c2, [1], c2.len)
    c2.truncate(6)
    lg = m.forward(c2, toks[6:7], 6)
    assert np.max(np.abs(lg - full[6])) < 1e-6


def test_lazy_block_storage_gives_identical_outputs():
    """The lazy storage mode (Q8_0 blocks kept, rows dequantised per call; for
    models too large to hold dequantised on the host) changes no arithmetic:
    the same greedy ids and bit-identical logits as the eager model."""
    from quantized_transformer_decode_gb300 import inputs
    s = inputs.TINY
    eager = orc.OracleModel.from_f32(s, inputs.generate_weights(s, 0))
    lazy = orc.OracleModel.from_f32_stream(s, ((n, w) for n, _, w in inputs.iter_weights(s, 0)))
    prompt = inputs.prompt_tokens(s, 0, 12)
    ia, la = eager.generate_greedy(eager.new_cache(20), prompt, 3)
    ib, lb = lazy.generate_greedy(lazy.new_cache(20), prompt, 3)
    assert ia == ib
    for x, y in zip(la, lb):
        np.testing.assert_array_equal(np.asarray(x), np.asarray(y))


def test_f16_kv_cache_rounds_to_nearest_even():
    """The f16 cache mode ("A transformer from scratch", 12.4: the course's
    default cache type) stores appended rows as IEEE half, nearest even:
    1 + 2^-11 is a tie between 1 and 1 + 2^-10 and rounds to 1 (even);
    1 + 3 * 2^-12 rounds up to 1 + 2^-10; 70000 overflows to inf; reads
    return the stored halves exactly."""
    c = orc.KvCache(1, 1, 4, 3, dtype="f16")
    k = np.array([[[1 + 2.0 ** -11, 1 + 3 * 2.0 ** -12, 70000.0, -2.0 ** -25]]], np.float32)
    v = np.array([[[0.1, -0.1, 65504.0, 3.0]]], np.float32)
    c.append_layer(0, k, v)
    c.advance(1)
    kk, vv = c.layer_rows(0, 1)
    np.testing.assert_array_equal(kk[0, 0], np.array([1.0, 1 + 2.0 ** -10, np.inf, -0.0], np.float32))
    np.testing.assert_array_equal(vv[0, 0], np.float16(v[0, 0]).astype(np.float32))
    assert kk.dtype == np.float32


def test_f16_kv_single_position_attention_returns_rounded_v():
    """Attention over one cached position returns V (12.3.5); in the f16
    cache mode that is V rounded to half."""
    c = orc.KvCache(1, 1, 8, 2, dtype="f16")
    rng = np.random.default_rng(5)
    k = rng.standard_normal((1, 1, 8)).astype(np.float32)
    v = rng.standard_normal((1, 1, 8)).astype(np.float32)
    c.append_layer(0, k, v)
    kk, vv = c.layer_rows(0, 1)
    q = rng.standard_normal((1, 1, 8)).astype(np.float32)
    o = orc.attention(q, kk, vv, [0], 0.3, [0])
    np.testing.assert_array_equal(o[0, 0], np.float16(v[0, 0]).astype(np.float32))


def test_f16_kv_model_layer0_rows_are_rounded_f32_rows():
    """Layer 0's K/V rows of a prefill depend only on the embedding, so in
    the f16 mode they are exactly the f32 mode's rows rounded to half."""
    from quantized_transformer_decode_gb300 import inputs
    s = inputs.TINY
    om = orc.OracleModel.from_f32(s, inputs.generate_weights(s, 0))
    prompt = inputs.prompt_tokens(s, 0, 10)
    c32, c16 = om.new_cache(12), om.new_cache(12, "f16")
    om.forward(c32, prompt, 0)
    om.forward(c16, prompt, 0)
    k32, v32 = c32.layer_rows(0, 10)
    k16, v16 = c16.layer_rows(0, 10)
    np.testing.assert_array_equal(k16, k32.astype(np.float16).astype(np.float32))
    np.testing.assert_array_equal(v16, v32.astype(np.float16).astype(np.float32))
    g32, _ = om.generate_greedy(om.new_cache(20), prompt, 2)
    g16, _ = om.generate_greedy(om.new_cache(20, "f16"), prompt, 2)
    assert len(g16) == len(g32) == 3


# ---- q8act: dynamic Q8_0 activations ("Model files and quantization", 11.9)

def _qlinear(w32):
    w32 = np.asarray(w32, np.float32)
    return orc.QLinear(orc.q8_0_quantize(w32), w32.shape[0], w32.shape[1], keep_f64=True)


def test_q8act_hand_worked_block():
    """One weight block with d_w = 0.5 (codes 127, -1, 2, 0, ...) against
    activations whose amax is 127, so d_a = 1 and the codes are the values
    rounded half away from zero: 127, 1.5 -> 2, -2.5 -> -3, 0.5 -> 1.
    The integer dot is 127*127 - 1*2 + 2*(-3) + 0*1 = 16121; times
    d_w * d_a = 0.5 gives 8060.5. The f32-activation path would give
    0.5 * (16129 - 1.5 - 5) = 8061.25."""
    w = np.zeros((1, 32), np.float32)
    w[0, :3] = [63.5, -0.5, 1.0]
    x = np.zeros((1, 32), np.float32)
    x[0, :5] = [127.0, 1.5, -2.5, 0.5, -0.49]
    L = _qlinear(w)
    assert float(L.q8act(x)[0, 0]) == 8060.5
    assert float(L(x)[0, 0]) == 8061.25


def test_q8act_equals_f32_path_on_representable_activations():
    """Activations already of the form d * q with amax = 127 d and d a power
    of two quantise to themselves, so the integer path computes the same
    sum as the f32-activation path (up to the f32 rounding of each block's
    (w.d * a.d) * acc product)."""
    rng = np.random.default_rng(5)
    w = rng.standard_normal((24, 96)).astype(np.float32)
    q = rng.integers(-127, 128, size=(3, 96)).astype(np.float32)
    q[:, ::32] = 127.0                                    # every block reaches amax = 127 d
    x = (q * np.float32(2.0 ** -3)).astype(np.float32)
    L = _qlinear(w)
    wq = orc.matrix_from_blocks(L.blocks.reshape(-1), 24, 96).astype(np.float64)
    # each block's product rounds once in f32 (half an ulp of its magnitude),
    # the sum is exact otherwise: bound by 2^-23 * sum |w| |x|
    tol = 2.0 ** -23 * (np.abs(x).astype(np.float64) @ np.abs(wq).T) + 1e-7
    assert np.all(np.abs(L.q8act(x).astype(np.float64) - L(x).astype(np.float64)) <= tol)


def test_q8act_error_within_the_activation_rounding_bound():
    """Per element |x - d16 q| <= d / 2 + 127 |d - d16| <= 0.5625 d (the f16
    scale is within 2^-11 of d), so per output row
    |q8act - f32 path| <= sum over blocks of 0.5625 d_a * sum |w| of the block
    (plus f32 rounding)."""
    rng = np.random.default_rng(6)
    w = rng.standard_normal((16, 128)).astype(np.float32)
    x = (rng.standard_normal((4, 128)) * rng.uniform(0.1, 10.0, size=(4, 1))).astype(np.float32)
    L = _qlinear(w)
    wq = orc.matrix_from_blocks(L.blocks.reshape(-1), 16, 128).astype(np.float64)
    d = np.abs(x).reshape(4, 4, 32).max(axis=2) / 127.0                       # [M, blocks]
    absw = np.abs(wq).reshape(16, 4, 32).sum(axis=2)                           # [rows, blocks]
    bound = 0.5625 * d @ absw.T                                                # [M, rows]
    err = np.abs(L.q8act(x).astype(np.float64) - L(x).astype(np.float64))
    assert np.all(err <= bound + 1e-5 * np.abs(L(x)) + 1e-6)
    assert err.max() > 0          # it is a different path


def test_q8act_power_of_two_scaling_and_zero():
    """Scaling the activations by 4 scales d_a by 4 exactly and leaves the
    codes alone, so the result scales by 4 exactly; a zero row gives zero."""
    rng = np.random.default_rng(7)
    L = _qlinear(rng.standard_normal((8, 64)))
    x = rng.standard_normal((2, 64)).astype(np.float32)
    np.testing.assert_array_equal(L.q8act(4.0 * x), 4.0 * L.q8act(x))
    assert not L.q8act(np.zeros((1, 64), np.float32)).any()


def test_q8act_model_mode_changes_only_the_linears():
    """The model in q8_0 activation mode: its logits stay within the
    activation-rounding noise of the f32 mode (relative L2 a few 1e-3 on the
    tiny model) but are not equal to them; set_activations rejects unknown
    kinds."""
    shape = inputs.TINY
    om = orc.OracleModel.from_f32(shape, inputs.generate_weights(shape, 0))
    prompt = inputs.prompt_tokens(shape, 0, 12)
    a = om.forward(om.new_cache(16), prompt, 0)
    om.set_activations("q8_0")
    b = om.forward(om.new_cache(16), prompt, 0)
    rel = np.linalg.norm(a - b) / np.linalg.norm(a)
    assert 0 < rel < 5e-2
    with pytest.raises(orc.InvalidShape):
        om.set_activations("q4")


# ---- q8_0 KV cache ("The LLM stack", 13.4; "A transformer from scratch", 12.4)

def test_q8_kv_rows_are_the_codec_round_trip_per_position_and_head():
    rng = np.random.default_rng(21)
    c = orc.KvCache(1, 2, 64, 8, "q8_0")
    k = rng.standard_normal((3, 2, 64)).astype(np.float32)
    v = (rng.standard_normal((3, 2, 64)) * 5).astype(np.float32)
    c.append_layer(0, k, v)
    c.advance(3)
    kk, vv = c.layer_rows(0, 3)
    for t in range(3):
        for g in range(2):
            for rows, src in ((kk, k), (vv, v)):
                blocks = orc.q8_0_quantize(src[t, g])
                np.testing.assert_array_equal(rows[t, g], orc.q8_0_dequantize(blocks, 64))
    d16, q = orc.q8_0_unpack(orc.q8_0_quantize(k[1, 0]), 64)
    np.testing.assert_array_equal(c.kq[0, 1, 0], q.reshape(-1))
    np.testing.assert_array_equal(c.kd[0, 1, 0], d16)
    with pytest.raises(orc.InvalidShape):
        orc.KvCache(1, 1, 48, 4, "q8_0")          # head_dim not a multiple of 32


def test_q8_scores_hand_worked_integer_dot():
    """Query [127, 0.5, 0, ...] encodes to codes [127, 1] with d = 1 (half
    away from zero); key [127, 127, 0, ...] to [127, 127] with d = 1. The
    integer score is 127*127 + 1*127 = 16256; the f32 dot would be
    127*127 + 0.5*127 = 16192.5."""
    c = orc.KvCache(1, 1, 32, 2, "q8_0")
    k = np.zeros((1, 1, 32), np.float32)
    k[0, 0, :2] = [127.0, 127.0]
    c.append_layer(0, k, k)
    q = np.zeros((1, 32), np.float32)
    q[0, :2] = [127.0, 0.5]
    s = orc.q8_scores(q, c.kq[0, :1], c.kd[0, :1], [0])
    assert s.shape == (1, 1) and s[0, 0] == 16256.0


def test_q8_decode_attention_one_position_and_two_key_sigmoid():
    """One cached position returns its dequantised V; two keys whose codes
    and scales are exact (d = 1/127 · 127) give the two-key softmax
    sigmoid(scale * (s1 - s2)) on exactly representable V rows."""
    c = orc.KvCache(1, 1, 32, 4, "q8_0")
    rng = np.random.default_rng(3)
    v1 = rng.standard_normal((1, 1, 32)).astype(np.float32)
    k1 = rng.standard_normal((1, 1, 32)).astype(np.float32)
    c.append_layer(0, k1, v1)
    q = rng.standard_normal((1, 1, 32)).astype(np.float32)
    o = orc.attention_q8_decode(q, c, 0, 1, 0.125, [0])
    np.testing.assert_array_equal(o[0, 0], c.v[0, 0, 0])
    # two keys, integer-valued with amax 127 (d = 1): scores are exact integers
    c2 = orc.KvCache(1, 1, 32, 4, "q8_0")
    ka = np.zeros((2, 1, 32), np.float32)
    ka[0, 0, 0], ka[0, 0, 1] = 127.0, 3.0
    ka[1, 0, 0], ka[1, 0, 1] = 127.0, -5.0
    va = np.zeros((2, 1, 32), np.float32)
    va[0, 0, 0], va[1, 0, 0] = 127.0, -127.0
    c2.append_layer(0, ka, va)
    qa = np.zeros((1, 1, 32), np.float32)
    qa[0, 0, 0], qa[0, 0, 1] = 1.0, 127.0                 # codes [1, 127], d = 1
    # s1 = 127 + 381 = 508, s2 = 127 - 635 = -508
    scale = 1.0 / 256.0
    o2 = orc.attention_q8_decode(qa, c2, 0, 2, scale, [0])
    p1 = 1.0 / (1.0 + math.exp(-scale * (508.0 + 508.0)))
    assert abs(float(o2[0, 0, 0]) - (p1 * 127.0 - (1 - p1) * 127.0)) < 1e-4


def test_q8_kv_model_stays_within_its_noise_and_prefill_reads_dequantised_rows():
    """The q8_0 cache changes logits by its quantisation noise only (tiny
    model), and a one-token decode after a prompt differs from the last row
    of the longer prompt (integer scores against dequantised f32 scores)
    while both stay close."""
    shape = inputs.TINY
    om = orc.OracleModel.from_f32(shape, inputs.generate_weights(shape, 0))
    prompt = inputs.prompt_tokens(shape, 0, 12)
    a = om.forward(om.new_cache(16), prompt, 0)
    b = om.forward(om.new_cache(16, "q8_0"), prompt, 0)
    rel = np.linalg.norm(a - b) / np.linalg.norm(a)
    assert 0 < rel < 5e-2
    c = om.new_cache(16, "q8_0")
    om.forward(c, prompt[:-1], 0)
    dec = om.forward(c, prompt[-1:], 11)
    pre = om.forward(om.new_cache(16, "q8_0"), prompt, 0)
    assert not np.array_equal(dec, pre)
    assert np.linalg.norm(dec - pre) / np.linalg.norm(pre) < 5e-2


# ---- Q4_K ("Model files and quantization", 11.8: super-block of 256, f16 d
# and dmin, eight 6-bit sub-scales and sub-mins packed in 12 bytes, 4-bit
# codes; x = d*sc*q - dmin*m)

def _q4k_hand_block():
    """One block built byte by byte: d = 1 (f16 0x3c00), dmin = 0.5 (0x3800),
    sub-scales 1, 2, 3, 4, 5, 6, 7, 63 and sub-mins 0, 1, 2, 3, 4, 5, 6, 63
    packed by hand into the 12 scale bytes (bytes 0-3: scales 0-3, top two
    bits of scales 4-7; bytes 4-7: mins 0-3, top two bits of mins 4-7;
    bytes 8-11: low nibbles of scales 4-7 | low nibbles of mins 4-7 << 4),
    every code equal to its value index mod 16 (byte 32c + l of the codes
    holds value 64c + l in its low nibble and 64c + 32 + l in its high one)."""
    b = np.zeros(144, np.uint8)
    b[0:2] = [0x00, 0x3C]
    b[2:4] = [0x00, 0x38]
    b[4:16] = [1, 2, 3, 196, 0, 1, 2, 195, 69, 86, 103, 255]
    for c in range(4):
        for l in range(32):
            b[16 + 32 * c + l] = (l % 16) * 17
    return b


def test_q4_k_hand_built_block_decodes_to_hand_computed_values():
    x = orc.q4_k_dequantize(_q4k_hand_block(), 256)
    # value index: sub-block j = i // 32, code i % 16; x = sc_j * q - 0.5 * m_j
    assert x[0] == 0.0                        # j 0: 1*0 - 0
    assert x[33] == 1.5                       # j 1: 2*1 - 0.5*1
    assert x[95] == 3 * 15 - 0.5 * 2          # j 2
    assert x[130] == 5 * 2 - 0.5 * 4          # j 4: scale and min from the split bytes
    assert x[191] == 6 * 15 - 0.5 * 5         # j 5
    assert x[255] == 63 * 15 - 0.5 * 63       # j 7: both six-bit fields at their maximum


def test_q4_k_encoder_picks_the_nearest_grid_point():
    """Each value decodes to the point of its sub-block's grid
    d16*sc*q - dmin16*m (q in 0..15) nearest to it (ties either way)."""
    x = inputs.uniform_block_values(31, 256 * 16, -0.3, 0.5)
    b = orc.q4_k_quantize(x)
    y = orc.q4_k_dequantize(b, x.size)
    d16, dm16, sc, m, _ = orc.q4_k_unpack(b, x.size)
    grid = ((d16.astype(np.float32)[:, None] * sc.astype(np.float32))[:, :, None] * np.arange(16, dtype=np.float32)
            - (dm16.astype(np.float32)[:, None] * m.astype(np.float32))[:, :, None]).astype(np.float32)  # [nb, 8, 16]
    xv = x.reshape(-1, 8, 32)
    best = np.min(np.abs(xv[..., None] - grid[:, :, None, :]), axis=-1)
    got = np.abs(xv - y.reshape(-1, 8, 32))
    assert np.all(got <= best + 1e-7)


def test_q4_k_round_trip_bound_and_zero_block():
    """With the encoder's grid the error is at most half a step (d16*sc / 2)
    for values inside [-dmin16*m, 15*d16*sc - dmin16*m] and the zero block is
    all zero bytes."""
    x = (np.random.default_rng(8).standard_normal(256 * 8) * 0.02).astype(np.float32)
    b = orc.q4_k_quantize(x)
    y = orc.q4_k_dequantize(b, x.size)
    d16, dm16, sc, m, _ = orc.q4_k_unpack(b, x.size)
    step = (d16.astype(np.float32)[:, None] * sc.astype(np.float32))            # [nb, 8]
    off = (dm16.astype(np.float32)[:, None] * m.astype(np.float32))
    xv, yv = x.reshape(-1, 8, 32), y.reshape(-1, 8, 32)
    inside = (xv >= -off[..., None]) & (xv <= 15 * step[..., None] - off[..., None])
    err = np.abs(xv - yv)
    assert np.all(err[inside] <= (step[..., None] / 2 + 1e-7).repeat(32, axis=2)[inside])
    assert np.mean(inside) > 0.9
    assert not orc.q4_k_quantize(np.zeros(256, np.float32)).any()
    with pytest.raises(orc.NonFiniteValue):
        orc.q4_k_quantize(np.full(256, np.inf, np.float32))


def test_q4_k_scale_packing_round_trips_every_six_bit_pair():
    sc = np.arange(64 * 8, dtype=np.uint16).reshape(64, 8) % 64
    m = (np.arange(64 * 8, dtype=np.uint16).reshape(64, 8) * 7 + 3) % 64
    s2, m2 = orc.q4k_unpack_scales(orc.q4k_pack_scales(sc, m))
    np.testing.assert_array_equal(s2, sc)
    np.testing.assert_array_equal(m2, m)


def test_q4_k_linear_one_hot_and_model_mode():
    rng = np.random.default_rng(12)
    w = (rng.standard_normal((9, 512)) * 0.05).astype(np.float32)
    L = orc.QLinear(orc.q4_k_quantize(w), 9, 512, keep_f64=True, wtype="q4_k")
    deq = orc.q4_k_dequantize(orc.q4_k_quantize(w), w.size).reshape(9, 512)
    for k in (0, 255, 256, 511):
        x = np.zeros((1, 512), np.float32)
        x[0, k] = 1.0
        np.testing.assert_array_equal(L(x)[0], deq[:, k])
    shape = inputs.TINY
    om = orc.OracleModel.from_f32(shape, inputs.generate_weights(shape, 0), wtype="q4_k")
    lg = om.forward(om.new_cache(8), inputs.prompt_tokens(shape, 0, 4), 0)
    assert lg.shape == (shape.vocab,) and np.all(np.isfinite(lg))
