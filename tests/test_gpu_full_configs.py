"""GPU parity at the full sizes of the prefill, batched-decode and 8B
workloads, through the C ABI, in the launch configuration the benchmark uses.

Where the oracle cannot finish the full workload (it is a plain f64 numpy
statement of the model), the check uses outputs it can compute one by one
(sampled sequences of the batch, layer-0 K/V rows, which depend on their own
token only), outputs it wrote once into tests/golden/ by a script that runs
only the oracle (the batch-64 and 8B greedy runs), and properties that hold at
any size (a decode step after a prefill equals the last row of the prefill
that includes its token).
"""
import os

import numpy as np
import pytest

from oracle import qw3_oracle as orc
from quantized_transformer_decode_gb300 import inputs
from parity import TIE_MARGIN, assert_argmax, assert_ids_prefix, assert_logits_close, cuda_ints

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


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


def test_prefill_4096_last_row(torch):
    """0.6B shape, one 4096-token prompt (tensor-core GEMMs): last-row logits
    and argmax against the oracle, and sampled KV rows of two layers."""
    from quantized_transformer_decode_gb300.qw3 import Qw3Model
    w = inputs.WORKLOADS["qwen3-0.6b-prefill4096"]
    S = w.prompt_len
    om = orc.OracleModel.from_f32(w.shape, inputs.generate_weights(w.shape, w.seed))
    cache = om.new_cache(S)
    prompt = inputs.prompt_tokens(w.shape, w.seed, S)
    want = om.forward(cache, prompt, 0)
    with Qw3Model.from_f32(w.shape, inputs.iter_weights(w.shape, w.seed), max_seq_len=S + 1, max_prefill=S) as gm:
        lg, am = gm.prefill(0, cuda_ints(prompt))
        gm.sync()
        assert_logits_close(_np(lg), want, "prefill 4096 last row")
        assert int(_np(am)[0]) == orc.argmax_lowest(want)
        pos = np.array([0, 1, 777, 2048, S - 1])
        for layer in (0, w.shape.n_layers - 1):
            k, v = gm.read_kv(layer, 0, 0, S)
            k, v = _np(k), _np(v)
            assert_logits_close(k[pos], cache.k[layer, pos], f"K layer {layer}")
            assert_logits_close(v[pos], cache.v[layer, pos], f"V layer {layer}")


def test_batch64_greedy_against_stored_oracle(torch):
    """0.6B shape, 64 sequences with their own 2048-token prefixes, decoded
    together at B = 64 (tensor-core GEMMs at 64 rows, batched attention) for
    64 greedy steps through qw3_generate_greedy, the call the benchmark
    times. The oracle's outputs for 8 of the sequences were written by
    tests/golden/make_qwen3_0_6b_batch64_golden.py: their ids (prefill
    argmax, then 64 steps) must match bit for bit up to the first near tie
    of the oracle's rows (parity.py); then, teacher-forced with the oracle's
    ids, the stored logits rows (sequence 0 after 64 steps, sequence 63
    after 1) must meet the bar."""
    from quantized_transformer_decode_gb300.qw3 import Qw3Model
    import torch as t
    g = np.load(os.path.join(GOLDEN, "qwen3_0_6b_batch64_greedy.npz"))
    seqs, ids, margins = [int(v) for v in g["seqs"]], g["ids"], g["margins"]
    w = inputs.WORKLOADS["qwen3-0.6b-batch64"]
    B, P, N = w.batch, w.prompt_len, int(g["n_steps"])
    assert int(g["prompt_len"]) == P and int(g["seed"]) == w.seed
    with Qw3Model.from_f32(w.shape, inputs.iter_weights(w.shape, w.seed), max_seqs=B, max_seq_len=P + N + 1,
                           max_prefill=P) as gm:
        firsts = []
        for b in range(B):
            _, am = gm.prefill(b, cuda_ints(inputs.batch_prefix_tokens(w.shape, w.seed, b, P)), want_logits=False)
            firsts.append(am)
        toks = t.cat(firsts)
        out = _np(gm.generate_greedy(toks, N))          # [N][B]
        first = _np(toks)
        for i, b in enumerate(seqs):
            run = [int(first[b])] + [int(v) for v in out[:, b]]
            n = next((k for k in range(N + 1) if margins[i][k] < TIE_MARGIN), N + 1)
            assert run[:n] == [int(v) for v in ids[i][:n]], f"sequence {b}: ids differ before row {n}"
        # teacher-forced: rewind every sequence to its prefix and feed the
        # oracle's ids to the sampled ones
        for b in range(B):
            gm.truncate(b, P)
        stored = {(int(si), int(step)): k for k, (si, step) in enumerate(g["rows"])}
        last = max(step for _, step in stored)
        cur = [int(first[b]) for b in range(B)]
        for i, b in enumerate(seqs):
            cur[b] = int(ids[i][0])
        for s in range(last):
            lg, am = gm.decode(cuda_ints(cur), [P + s] * B)
            lgn, amn = _np(lg), _np(am)
            for (si, step), k in stored.items():
                if step == s + 1:
                    assert_logits_close(lgn[seqs[si]], g["logits"][k], f"sequence {seqs[si]} step {step}")
            cur = [int(v) for v in amn]
            for i, b in enumerate(seqs):
                if s + 1 <= N:
                    cur[b] = int(ids[i][s + 1])
        gm.sync()


QWEN3_8B_2L = inputs.QWEN3_8B.with_layers(2)


def test_8b_geometry_two_layers(torch):
    """Every kernel at the 8B widths (hidden 4096, 32/8 heads, intermediate
    12288, untied lm_head) against the oracle on a 2-layer model: prefill
    (tensor cores), teacher-forced decode, greedy ids."""
    from quantized_transformer_decode_gb300.qw3 import Qw3Model
    shape, seed, P, steps = QWEN3_8B_2L, 2, 96, 6
    om = orc.OracleModel.from_f32(shape, inputs.generate_weights(shape, seed))
    prompt = inputs.prompt_tokens(shape, seed, P)
    ids, logits = om.generate_greedy(om.new_cache(P + steps + 1), prompt, steps)
    with Qw3Model.from_f32(shape, inputs.iter_weights(shape, seed), max_seq_len=P + steps + 1, max_prefill=64) as gm:
        lg, am = gm.prefill(0, cuda_ints(prompt))
        assert_logits_close(_np(lg), logits[0], "8B-geometry prefill")
        assert_argmax(int(_np(am)[0]), ids[0], logits[0], "8B-geometry prefill")
        for s in range(steps):
            lg, am = gm.decode(cuda_ints([ids[s]]), [P + s])
            assert_logits_close(_np(lg)[0], logits[s + 1], f"8B-geometry step {s + 1}")
            assert_argmax(int(_np(am)[0]), ids[s + 1], logits[s + 1], f"8B-geometry step {s + 1}")
        gm.reset(0)
        _, am = gm.prefill(0, cuda_ints(prompt), want_logits=False)
        out = gm.generate_greedy(am, steps)
        gm.sync()
        assert_ids_prefix([int(_np(am)[0])] + [int(v) for v in _np(out)[:, 0]], ids, logits)


@pytest.fixture(scope="module")
def model_8b(torch):
    """The Qwen3-8B-shape model at full size (36 layers, 8.7 GB of Q8_0
    weights), room for two sequences of the 8192-token prompt plus 64 steps."""
    from quantized_transformer_decode_gb300.qw3 import Qw3Model
    w = inputs.WORKLOADS["qwen3-8b"]
    gm = Qw3Model.from_f32(w.shape, inputs.iter_weights(w.shape, w.seed), max_seqs=2,
                           max_seq_len=w.prompt_len + 66, max_prefill=4096)
    yield gm
    gm.close()


def test_8b_greedy_against_stored_oracle(model_8b):
    """Qwen3-8B shape, the 8192-token prompt, then 64 greedy steps at batch 1
    through qw3_generate_greedy. tests/golden/make_qwen3_8b_golden.py wrote
    the oracle's ids (prefill argmax, then each step's) with each row's top-2
    margin, and its logits rows at steps 0, 1, 32 and 64. The ids must match
    bit for bit up to the oracle's first near tie (parity.py); then, fed the
    oracle's ids (teacher-forced), the stored rows must meet the bar."""
    g = np.load(os.path.join(GOLDEN, "qwen3_8b_greedy.npz"))
    w = inputs.WORKLOADS["qwen3-8b"]
    s, P, N = w.shape, w.prompt_len, int(g["n_steps"])
    assert int(g["prompt_len"]) == P and int(g["seed"]) == w.seed
    ids = [int(v) for v in g["ids"]]
    margins = g["margins"] if "margins" in g.files else np.full(N + 1, np.inf)     # absent: all strict
    stored = {int(k): g["logits"][i] for i, k in enumerate(g["steps"])}
    gm = model_8b
    gm.reset(0)
    gm.reset(1)
    prompt = inputs.prompt_tokens(s, w.seed, P)
    lg, am = gm.prefill(0, cuda_ints(prompt), want_logits=True)
    assert_logits_close(_np(lg), stored[0], "8B prefill last row")
    out = _np(gm.generate_greedy(am, N, seqs=[0]))
    run = [int(_np(am)[0])] + [int(v) for v in out[:, 0]]
    n = next((k for k in range(N + 1) if margins[k] < TIE_MARGIN), N + 1)
    assert run[:n] == ids[:n], f"8B greedy ids differ before row {n}"
    gm.truncate(0, P)
    for k in range(N):
        want = stored.get(k + 1)
        lg, am = gm.decode(cuda_ints([ids[k]]), [P + k], seqs=[0], want_logits=want is not None)
        if want is not None:
            assert_logits_close(_np(lg)[0], want, f"8B step {k + 1}")
            assert_argmax(int(_np(am)[0]), ids[k + 1], want, f"8B step {k + 1}")
    gm.sync()


def test_8b_full_size_properties(model_8b):
    """Qwen3-8B shape at full size (36 layers, 8.7 GB of Q8_0 weights, an
    8192-token prompt): layer-0 K/V rows at sampled positions against the
    oracle's layer 0 for those tokens, and the cached == uncached property
    (course 12.4): decoding token t after the 8192-token prefill gives the
    logits of the last row of an 8193-token prefill."""
    w = inputs.WORKLOADS["qwen3-8b"]
    s, P = w.shape, w.prompt_len
    prompt = inputs.prompt_tokens(s, w.seed, P + 1)
    gm = model_8b
    gm.reset(0)
    gm.reset(1)
    _, am = gm.prefill(0, cuda_ints(prompt[:P]), want_logits=False)
    lg_dec, am_dec = gm.decode(cuda_ints(prompt[P:P + 1]), [P], seqs=[0])
    lg_full, am_full = gm.prefill(1, cuda_ints(prompt))
    gm.sync()
    assert_logits_close(_np(lg_dec)[0], _np(lg_full), "decode after prefill vs longer prefill")
    assert int(_np(am_dec)[0]) == int(_np(am_full)[0])
    k, v = gm.read_kv(0, 0, 0, P)
    k, v = _np(k), _np(v)
    # the oracle's layer 0 for single tokens at their own positions
    w0 = {}
    for name, kind, arr in inputs.iter_weights(s, w.seed):
        if name in ("token_embd", "blk.0.attn_norm", "blk.0.attn_k", "blk.0.attn_v", "blk.0.attn_k_norm"):
            w0[name] = orc.q8_0_quantize(arr) if kind == "linear" else np.asarray(arr, np.float32)
        if name.startswith("blk.1."):
            break
    emb = orc.QLinear(w0["token_embd"], s.vocab, s.hidden, keep_f64=False)
    wk = orc.QLinear(w0["blk.0.attn_k"], s.kv_width, s.hidden, keep_f64=True)
    wv = orc.QLinear(w0["blk.0.attn_v"], s.kv_width, s.hidden, keep_f64=True)
    for p in (0, 1, 4095, P - 1):
        x = emb.row(np.array([prompt[p]]))
        h = orc.rms_norm(x, w0["blk.0.attn_norm"], s.rms_eps)
        kk = orc.rms_norm(wk(h).reshape(1, s.n_kv_heads, s.head_dim), w0["blk.0.attn_k_norm"], s.rms_eps)
        kk = orc.rope_neox(kk, [p], s.rope_theta)
        vv = wv(h).reshape(1, s.n_kv_heads, s.head_dim)
        assert_logits_close(k[p], kk[0], f"8B layer-0 K at {p}")
        assert_logits_close(v[p], vv[0], f"8B layer-0 V at {p}")
