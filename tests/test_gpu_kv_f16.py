"""GPU parity of the f16 KV cache mode (QW3_FLAG_KV_F16) against the oracle
run with a half cache ("A transformer from scratch", 12.4: half is the
course's default cache type).

Both sides round each appended key and value to IEEE half, nearest even, from
their own f32 (CUDA) or f64 (oracle) value. The two pre-rounding values differ
by the projections' reassociation error, so an element at a rounding boundary
can land one half ulp apart. The checks, in that light:

  * the cache: every element within one half ulp of the oracle's, nearly all
    equal;
  * decode arithmetic on identical caches: the GPU's cache, the step's own
    new row included, is copied into the oracle's for each teacher-forced
    step, and the step's logits then meet the f32 mode's bar (max-abs 2e-3,
    rel-L2 1e-4) and the near-tie rule of parity.py;
  * rows that depend on each side's own rounding (the prefill row, the
    free-running ids): a flip moves a cached element by one ulp, at most
    2^-10 of its magnitude, on the few elements that flip, while the half
    cache itself moves every element by up to half an ulp. So the GPU's row
    is held to the distance between the oracle's own f16-cache and f32-cache
    rows (at least the f32 bar): rel-L2 <= max(1e-4, rel(o16, o32)), and a
    near tie of this mode is a row whose top-2 margin is below
    max(1e-4, max-abs(o16 - o32)).
"""
import numpy as np
import pytest

from oracle import qw3_oracle as orc
from quantized_transformer_decode_gb300 import inputs
from parity import (MAX_ABS, REL_L2, TIE_MARGIN, assert_argmax, assert_logits_close, build_pair, cuda_ints,
                    row_errors, top2_margin)

pytestmark = pytest.mark.gpu

KV_F16 = 0x20
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


def mode_bounds(om, prompt, steps, cap):
    """Oracle ids and rows with a half cache, and per row the f16 mode's
    rel-L2 bound and near-tie margin (the distance to the f32-cache row)."""
    ids, rows16 = om.generate_greedy(om.new_cache(cap, "f16"), prompt, steps)
    rows32 = om.teacher_forced(om.new_cache(cap), prompt, ids[:steps])
    rel, margin = [], []
    for a, b in zip(rows16, rows32):
        ma, rl = row_errors(a, b)
        rel.append(max(REL_L2, rl))
        margin.append(max(TIE_MARGIN, ma))
    return ids, rows16, rel, margin


class GpuRowsCache(orc.KvCache):
    """The oracle's half cache holding the GPU's cached rows: rows [0, n) of
    a sequence are copied in (the GPU's values are halves: the copy is
    exact), and a row the oracle appends at a position the GPU has already
    cached is replaced by the GPU's, so that the oracle's forward scores
    exactly the cache the GPU scored."""

    def __init__(self, om, capacity):
        s = om.shape
        super().__init__(s.n_layers, s.n_kv_heads, s.head_dim, capacity, "f16")
        self.gk = np.zeros_like(self.k)
        self.gv = np.zeros_like(self.v)
        self.n_gpu = 0

    def load_gpu(self, gm, n, seq=0):
        for layer in range(self.k.shape[0]):
            k, v = gm.read_kv(layer, seq, 0, n)
            self.gk[layer, :n] = _np(k).astype(np.float16)
            self.gv[layer, :n] = _np(v).astype(np.float16)
        self.n_gpu = n

    def append_layer(self, layer, k_rows, v_rows):
        super().append_layer(layer, k_rows, v_rows)
        hi = min(self.len + k_rows.shape[0], self.n_gpu)
        if hi > self.len:
            self.k[layer, self.len:hi] = self.gk[layer, self.len:hi]
            self.v[layer, self.len:hi] = self.gv[layer, self.len:hi]

    def step_on_gpu_rows(self, om, gm, tok, pos, seq=0):
        """The oracle's logits for `tok` at `pos` over the GPU's rows
        [0, pos + 1) (call after the GPU's decode of that step)."""
        self.load_gpu(gm, pos + 1, seq)
        self.k[:, :pos] = self.gk[:, :pos]
        self.v[:, :pos] = self.gv[:, :pos]
        self.len = pos
        return om.forward(self, [tok], pos)


def _greedy_f16(shape, seed, prompt_len, steps, max_prefill=64, max_seq_len=None):
    cap = max_seq_len or prompt_len + steps + 8
    om, gm = build_pair(shape, seed, max_seq_len=cap, max_prefill=max_prefill, flags=KV_F16)
    prompt = inputs.prompt_tokens(shape, seed, prompt_len)
    try:
        ids, rows, rel, margin = mode_bounds(om, prompt, steps, prompt_len + steps + 1)
        lg, am = gm.prefill(0, cuda_ints(prompt))
        assert_logits_close(_np(lg), rows[0], "prefill last row", max_abs=MAX_ABS, rel_l2=rel[0])
        got = int(_np(am)[0])
        assert got == ids[0] or rows[0][ids[0]] - rows[0][got] < margin[0]
        # teacher-forced decode on the GPU's own cache
        oc = GpuRowsCache(om, prompt_len + steps + 1)
        for s in range(steps):
            lg, am = gm.decode(cuda_ints([ids[s]]), [prompt_len + s])
            want = oc.step_on_gpu_rows(om, gm, ids[s], prompt_len + s)
            assert_logits_close(_np(lg)[0], want, f"decode step {s + 1}")
            assert_argmax(int(_np(am)[0]), orc.argmax_lowest(want), want, f"argmax at step {s + 1}")
        gm.sync()
        # free-running: ids bit-exact up to this mode's first near tie
        gm.reset(0)
        _, am = gm.prefill(0, cuda_ints(prompt), want_logits=False)
        out = gm.generate_greedy(am, steps)
        gm.sync()
        run = [int(_np(am)[0])] + [int(v) for v in _np(out)[:, 0]]
        n = next((i for i, r in enumerate(rows) if top2_margin(r) < margin[i]), len(rows))
        assert run[:n] == ids[:n], f"free-running ids differ before row {n}"
    finally:
        gm.close()


def test_tiny_f16_cache_greedy_and_logits(torch):
    w = inputs.WORKLOADS["tiny"]
    _greedy_f16(w.shape, w.seed, w.prompt_len, w.decode_steps)


@pytest.mark.parametrize("prompt_len,max_prefill", [(40, 64), (300, 512)])
def test_mid_f16_cache_greedy_and_logits(torch, prompt_len, max_prefill):
    """300 prompt rows in one chunk take the tensor-core prefill attention
    (which packs the half cache into fp16 hi/lo pairs of power-of-two-scaled
    values); 40 the SIMT
    one. Decode at batch 1 runs the per-kernel chain in this mode."""
    _greedy_f16(MID, 3, prompt_len, 6, max_prefill=max_prefill)


def test_f16_cache_long_context_split_over_clusters(torch):
    """A capacity past the long-context threshold makes decode attention split
    each kv head over several clusters (half tiles of 64 positions)."""
    _greedy_f16(MID, 7, 600, 5, max_prefill=256, max_seq_len=4200)


def test_f16_cache_contents_within_one_half_ulp(torch):
    """Every cached value is a half; it differs from the oracle's by at most
    one half ulp beyond the f32 cache's own tolerance on K and V (max-abs
    1e-4: the pre-rounding values differ by the projections' reassociation
    error, and by more in layer 1, whose input went through layer 0's
    differently rounded cache). Layer 0's inputs are the embedding rows
    themselves, so nearly all of its values agree exactly."""
    shape = inputs.TINY
    om, gm = build_pair(shape, 0, max_seq_len=64, max_prefill=16, flags=KV_F16)
    try:
        prompt = inputs.prompt_tokens(shape, 0, 21)
        cache = om.new_cache(64, "f16")
        om.forward(cache, prompt, 0)
        om.forward(cache, [17], 21)
        gm.prefill(0, cuda_ints(prompt), want_logits=False)
        gm.decode(cuda_ints([17]), [21], want_logits=False)
        for layer in range(shape.n_layers):
            k, v = gm.read_kv(layer, 0, 0, 22)
            for got, want, name in ((_np(k), cache.k[layer, :22], "K"), (_np(v), cache.v[layer, :22], "V")):
                want = np.asarray(want, dtype=np.float32)
                assert np.array_equal(got, got.astype(np.float16).astype(np.float32)), name
                ulp = np.spacing(np.abs(want).astype(np.float16)).astype(np.float32)
                excess = np.abs(got - want) - ulp
                assert excess.max() <= 1e-4, f"{name} layer {layer}: {excess.max():.3e} past one half ulp"
                rel = row_errors(got, want)[1]
                assert rel <= 5e-4, f"{name} layer {layer}: rel-L2 {rel:.3e}"
                if layer == 0:
                    assert np.mean(got == want) > 0.98, f"{name} layer 0: {np.mean(got == want):.4f} equal"
    finally:
        gm.close()


@pytest.mark.parametrize("B", [2, 8])
def test_f16_cache_batched_decode(torch, B):
    """B sequences of different lengths per decode call (B = 2: GEMV path,
    B = 8: tiled GEMM path), each step checked against the oracle run on
    that sequence's GPU cache."""
    shape = inputs.TINY
    om, gm = build_pair(shape, 0, max_seqs=B, max_seq_len=96, max_prefill=32, flags=KV_F16)
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


def test_f16_cache_halves_the_cache_allocation(torch):
    """The mode's point: the cache takes half the device bytes."""
    shape = inputs.TINY
    free0 = torch.cuda.mem_get_info()[0]
    _, g32 = build_pair(shape, 0, max_seq_len=32768, max_prefill=16)
    free32 = torch.cuda.mem_get_info()[0]
    g32.close()
    _, g16 = build_pair(shape, 0, max_seq_len=32768, max_prefill=16, flags=KV_F16)
    free16 = torch.cuda.mem_get_info()[0]
    g16.close()
    cache32 = shape.n_layers * 2 * shape.n_kv_heads * 32768 * shape.head_dim * 4
    used32, used16 = free0 - free32, free0 - free16
    assert used32 - used16 > 0.4 * cache32
