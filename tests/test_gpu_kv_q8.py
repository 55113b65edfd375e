"""GPU parity of the q8_0 KV cache mode (QW3_FLAG_KV_Q8; "The LLM stack",
13.4) against the oracle run with a q8_0 cache.

Both sides encode each appended (position, kv head) row with the 11.7
encoder from their own f32 (CUDA) or f64-then-f32 (oracle) values, which
differ by the projections' reassociation error, so a code at a rounding
boundary can land one step apart. The checks:

  * the cache: every value within one quantum (the block's scale) of the
    oracle's, beyond the f32 cache's K/V tolerance; nearly all of layer 0
    equal;
  * the integer-score decode step on identical caches: the GPU's rows (codes
    and scales recovered exactly from its dequantised values: the largest
    code of a block is +-127, so d = max|x| / 127 and q = x / d) are copied
    into the oracle's cache for each teacher-forced step; the step's logits
    then meet the f32 bar and the near-tie rule of parity.py;
  * rows that depend on each side's own encoding (the prefill row, the
    free-running ids): held to the distance between the oracle's q8_0-cache
    and f32-cache rows (at least the f32 bar).
"""
import numpy as np
import pytest

from oracle import qw3_oracle as orc
from quantized_transformer_decode_gb300 import inputs
from parity import (MAX_ABS, REL_L2, TIE_MARGIN, assert_argmax, assert_logits_close, build_pair, cuda_ints,
                    row_errors, top2_margin)

pytestmark = pytest.mark.gpu

KV_Q8 = 0x80
MID = inputs.Qwen3Shape(vocab=5003, hidden=1024, n_layers=2, n_heads=16, n_kv_heads=8, head_dim=128,
                        intermediate=3072, tied=True)


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_transformer_decode_gb300 import build
    build.build()
    return t


def _np(t):
    return t.detach().cpu().numpy()


def recover_blocks(x):
    """(codes int8, f16 scales) of dequantised q8_0 rows x [..., d]."""
    xb = np.asarray(x, np.float32).reshape(*x.shape[:-1], -1, 32)
    d = (np.max(np.abs(xb), axis=-1) / np.float32(127.0)).astype(np.float32)
    d16 = d.astype(np.float16)
    assert np.array_equal(d16.astype(np.float32), d), "a block's largest code is not +-127"
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(d[..., None] > 0, xb / d[..., None], 0.0)
    assert np.array_equal(q, np.round(q)) and np.all(np.abs(q) <= 127)
    return q.astype(np.int8).reshape(x.shape), d16


def mode_bounds(om, prompt, steps, cap):
    ids, rows8 = om.generate_greedy(om.new_cache(cap, "q8_0"), prompt, steps)
    rows32 = om.teacher_forced(om.new_cache(cap), prompt, ids[:steps])
    rel, margin = [], []
    for a, b in zip(rows8, rows32):
        ma, rl = row_errors(a, b)
        rel.append(max(REL_L2, rl))
        margin.append(max(TIE_MARGIN, ma))
    return ids, rows8, rel, margin


class GpuRowsCache(orc.KvCache):
    """The oracle's q8_0 cache holding the GPU's cached rows (see the module
    docstring); a row the oracle appends where the GPU has already cached one
    is replaced by the GPU's."""

    def __init__(self, om, capacity):
        s = om.shape
        super().__init__(s.n_layers, s.n_kv_heads, s.head_dim, capacity, "q8_0")
        self.g = None
        self.n_gpu = 0

    def load_gpu(self, gm, n, seq=0):
        g = {}
        for layer in range(self.k.shape[0]):
            k, v = gm.read_kv(layer, seq, 0, n)
            g[layer] = (_np(k), _np(v))
        self.g, self.n_gpu = g, n

    def _put(self, layer, lo, hi):
        k, v = self.g[layer]
        for x, q_arr, d_arr, deq in ((k, self.kq, self.kd, self.k), (v, self.vq, self.vd, self.v)):
            q, d16 = recover_blocks(x[lo:hi])
            q_arr[layer, lo:hi] = q
            d_arr[layer, lo:hi] = d16
            deq[layer, lo:hi] = x[lo:hi]

    def append_layer(self, layer, k_rows, v_rows):
        super().append_layer(layer, k_rows, v_rows)
        hi = min(self.len + k_rows.shape[0], self.n_gpu)
        if hi > self.len:
            self._put(layer, self.len, hi)

    def step_on_gpu_rows(self, om, gm, tok, pos, seq=0):
        self.load_gpu(gm, pos + 1, seq)
        for layer in range(self.k.shape[0]):
            self._put(layer, 0, pos)
        self.len = pos
        return om.forward(self, [tok], pos)


def _greedy_q8(shape, seed, prompt_len, steps, max_prefill=64, max_seq_len=None):
    cap = max_seq_len or prompt_len + steps + 8
    om, gm = build_pair(shape, seed, max_seq_len=cap, max_prefill=max_prefill, flags=KV_Q8)
    prompt = inputs.prompt_tokens(shape, seed, prompt_len)
    try:
        ids, rows, rel, margin = mode_bounds(om, prompt, steps, prompt_len + steps + 1)
        lg, am = gm.prefill(0, cuda_ints(prompt))
        assert_logits_close(_np(lg), rows[0], "prefill last row", max_abs=max(MAX_ABS, margin[0]), rel_l2=rel[0])
        got = int(_np(am)[0])
        assert got == ids[0] or rows[0][ids[0]] - rows[0][got] < margin[0]
        oc = GpuRowsCache(om, prompt_len + steps + 1)
        for s in range(steps):
            lg, am = gm.decode(cuda_ints([ids[s]]), [prompt_len + s])
            want = oc.step_on_gpu_rows(om, gm, ids[s], prompt_len + s)
            assert_logits_close(_np(lg)[0], want, f"decode step {s + 1}")
            assert_argmax(int(_np(am)[0]), orc.argmax_lowest(want), want, f"argmax at step {s + 1}")
        gm.sync()
        gm.reset(0)
        _, am = gm.prefill(0, cuda_ints(prompt), want_logits=False)
        out = gm.generate_greedy(am, steps)
        gm.sync()
        run = [int(_np(am)[0])] + [int(v) for v in _np(out)[:, 0]]
        n = next((i for i, r in enumerate(rows) if top2_margin(r) < margin[i]), len(rows))
        assert run[:n] == ids[:n], f"free-running ids differ before row {n}"
    finally:
        gm.close()


def test_tiny_q8_cache_greedy_and_logits(torch):
    """head_dim 64: two blocks per row, 16 lanes per block."""
    w = inputs.WORKLOADS["tiny"]
    _greedy_q8(w.shape, w.seed, w.prompt_len, w.decode_steps)


@pytest.mark.parametrize("prompt_len,max_prefill", [(40, 64), (300, 512)])
def test_mid_q8_cache_greedy_and_logits(torch, prompt_len, max_prefill):
    """SIMT (40 rows) and tensor-core (300 rows) prefill attention over the
    dequantised rows; decode through the integer score path."""
    _greedy_q8(MID, 3, prompt_len, 6, max_prefill=max_prefill)


def test_q8_cache_long_context_split_over_clusters(torch):
    _greedy_q8(MID, 7, 600, 5, max_prefill=256, max_seq_len=4200)


def test_q8_cache_contents(torch):
    shape = inputs.TINY
    om, gm = build_pair(shape, 0, max_seq_len=64, max_prefill=16, flags=KV_Q8)
    try:
        prompt = inputs.prompt_tokens(shape, 0, 21)
        cache = om.new_cache(64, "q8_0")
        om.forward(cache, prompt, 0)
        om.forward(cache, [17], 21)
        gm.prefill(0, cuda_ints(prompt), want_logits=False)
        gm.decode(cuda_ints([17]), [21], want_logits=False)
        for layer in range(shape.n_layers):
            k, v = gm.read_kv(layer, 0, 0, 22)
            for got, want, scales, name in ((_np(k), cache.k[layer, :22], cache.kd[layer, :22], "K"),
                                            (_np(v), cache.v[layer, :22], cache.vd[layer, :22], "V")):
                recover_blocks(got)                       # every GPU row is a valid q8_0 row
                quantum = np.repeat(scales.astype(np.float32), 32, axis=-1)
                excess = np.abs(got - want) - quantum
                assert excess.max() <= 1e-4, f"{name} layer {layer}: {excess.max():.3e} past one quantum"
                if layer == 0:
                    assert np.mean(got == want) > 0.98, f"{name} layer 0: {np.mean(got == want):.4f} equal"
    finally:
        gm.close()


@pytest.mark.parametrize("B", [2, 8])
def test_q8_cache_batched_decode(torch, B):
    shape = inputs.TINY
    om, gm = build_pair(shape, 0, max_seqs=B, max_seq_len=96, max_prefill=32, flags=KV_Q8)
    lens = [5 + 11 * b for b in range(B)]
    seqs = list(range(B))[::-1]
    try:
        toks = []
        for b in range(B):
            pre = inputs.batch_prefix_tokens(shape, 0, b, lens[b])
            _, am = gm.prefill(seqs[b], cuda_ints(pre), want_logits=False)
            toks.append(int(_np(am)[0]))
        caches = [GpuRowsCache(om, 96) for _ in range(B)]
        pos = list(lens)
        for step in range(3):
            lg, am = gm.decode(cuda_ints(toks), pos, seqs=seqs)
            lg, am = _np(lg), _np(am)
            want = [caches[b].step_on_gpu_rows(om, gm, toks[b], pos[b], seqs[b]) for b in range(B)]
            for b in range(B):
                assert_logits_close(lg[b], want[b], f"B={B} seq {b} step {step}")
                assert_argmax(int(am[b]), orc.argmax_lowest(want[b]), want[b], f"B={B} seq {b} step {step}")
                toks[b] = int(am[b])
                pos[b] += 1
    finally:
        gm.close()


def test_q8_cache_rejects_two_cache_types(torch):
    from quantized_transformer_decode_gb300.qw3 import Qw3Error, Qw3Model
    shape = inputs.TINY
    with pytest.raises(Qw3Error):
        Qw3Model.from_f32(shape, inputs.iter_weights(shape, 0), max_seq_len=16, max_prefill=16, flags=KV_Q8 | 0x20)
