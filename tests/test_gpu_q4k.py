"""GPU parity of Q4_K weights ("Model files and quantization", 11.8) against
the oracle: the encoder bit for bit, the decoder exactly, the raw-row GEMV
within its f32 accumulation bound, and whole models built with
QW3_FLAG_WEIGHTS_Q4_K (both sides encode the same seeded f32 weights with
their own encoders, whose bytes are checked equal) at the logits bar and the
near-tie rule of parity.py.
"""
import numpy as np
import pytest

from oracle import qw3_oracle as orc
from quantized_transformer_decode_gb300 import inputs
from parity import assert_argmax, assert_ids_prefix, assert_logits_close, cuda_ints

pytestmark = pytest.mark.gpu

Q4K = 0x100
MID = inputs.Qwen3Shape(vocab=5003, hidden=1024, n_layers=2, n_heads=16, n_kv_heads=8, head_dim=128,
                        intermediate=3072, tied=True)
MID_UNTIED = inputs.Qwen3Shape(vocab=3001, hidden=512, n_layers=2, n_heads=8, n_kv_heads=2, head_dim=128,
                               intermediate=1536, tied=False)


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


def special_blocks():
    rng = np.random.default_rng(5)
    blocks = [
        np.zeros(256, np.float32),                                   # all zero
        np.full(256, 0.37, np.float32),                              # constant positive
        np.full(256, -1.25, np.float32),                             # constant negative
        np.abs(rng.standard_normal(256)).astype(np.float32),         # all positive: min 0 offset
        -np.abs(rng.standard_normal(256)).astype(np.float32),        # all negative
        (rng.standard_normal(256) * 1e-6).astype(np.float32),        # scales near the f16 subnormals
        (rng.standard_normal(256) * 300.0).astype(np.float32),       # wide range
        np.where(np.arange(256) % 32 == 0, 5.0, 0.0).astype(np.float32),   # one spike per sub-block
    ]
    ramp = np.linspace(-3, 7, 256, dtype=np.float32)
    blocks.append(ramp)
    return np.concatenate(blocks)


@pytest.mark.parametrize("case", ["weights", "uniform", "special"])
def test_q4k_quantize_bit_exact(torch, case):
    from quantized_transformer_decode_gb300 import qw3
    x = {"weights": (np.random.default_rng(1).standard_normal(256 * 4000) * 0.02).astype(np.float32),
         "uniform": inputs.uniform_block_values(2, 256 * 3000, -0.7, 1.9),
         "special": special_blocks()}[case]
    want = orc.q4_k_quantize(x)
    got = _np(qw3.q4_k_quantize(torch.from_numpy(x).cuda()))
    assert np.array_equal(got, want), f"{int(np.sum(got != want))} bytes differ"


def test_q4k_quantize_nonfinite_block_zeroed_with_status(torch):
    from quantized_transformer_decode_gb300 import qw3
    x = np.ones(256 * 3, np.float32)
    x[256 + 7] = np.nan
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _np(qw3.q4_k_quantize(torch.from_numpy(x).cuda(), st))
    assert not got[144:288].any()
    assert np.array_equal(got[:144], orc.q4_k_quantize(np.ones(256, np.float32)))
    assert int(st.item()) == 5


def test_q4k_dequantize_exact(torch):
    from quantized_transformer_decode_gb300 import qw3
    x = np.concatenate([special_blocks(), inputs.uniform_block_values(3, 256 * 500)])
    blocks = orc.q4_k_quantize(x)
    y = _np(qw3.q4_k_dequantize(torch.from_numpy(blocks).cuda(), x.size))
    np.testing.assert_array_equal(y, orc.q4_k_dequantize(blocks, x.size))


@pytest.mark.parametrize("rows,cols,B", [(8, 256, 1), (1000, 1024, 1), (4096, 1024, 3), (1024, 3072, 8),
                                         (77, 12288, 4), (333, 2048, 2)])
def test_q4k_gemv(torch, rows, cols, B):
    from quantized_transformer_decode_gb300 import qw3
    rng = np.random.default_rng([rows, cols, B, 4])
    blocks = orc.q4_k_quantize(rng.standard_normal((rows, cols), dtype=np.float32) * np.float32(0.02))
    d16, dm16, sc, m, q = orc.q4_k_unpack(blocks, rows * cols)
    w = orc.q4_k_dequantize(blocks, rows * cols).reshape(rows, cols).astype(np.float64)
    x = rng.standard_normal((B, cols)).astype(np.float32)
    want = x.astype(np.float64) @ w.T
    y = _np(qw3.q4_k_gemv(torch.from_numpy(blocks).cuda(), rows, cols, torch.from_numpy(x).cuda()))
    # the kernel sums d1 * sum(q x) - m1 * sum(x) per sub-block in f32: bound
    # by K * 2^-23 times the sum of |d1 q x| + |m1 x|
    d1 = (d16.astype(np.float64)[:, None] * sc).repeat(32, axis=1).reshape(rows, cols)
    m1 = (dm16.astype(np.float64)[:, None] * m).repeat(32, axis=1).reshape(rows, cols)
    mag = np.abs(x.astype(np.float64)) @ (np.abs(d1 * q.reshape(rows, cols)) + np.abs(m1)).T
    bound = mag * cols * 2.0 ** -23 + 1e-30
    err = np.abs(y - want)
    assert np.all(err <= bound), float(np.max(err / bound))


def _pair(torch, shape, seed, **kw):
    from quantized_transformer_decode_gb300.qw3 import Qw3Model
    om = orc.OracleModel.from_f32(shape, inputs.generate_weights(shape, seed), wtype="q4_k")
    gm = Qw3Model.from_f32(shape, inputs.iter_weights(shape, seed), flags=Q4K, **kw)
    return om, gm


@pytest.mark.parametrize("case", ["tiny", "mid", "mid_tc_prefill", "untied"])
def test_q4k_model_greedy_and_logits(torch, case):
    shape, seed, P, steps, max_prefill = {
        "tiny": (inputs.TINY, 0, 32, 12, 64), "mid": (MID, 3, 40, 6, 64),
        "mid_tc_prefill": (MID, 4, 300, 4, 512), "untied": (MID_UNTIED, 5, 20, 5, 16)}[case]
    om, gm = _pair(torch, shape, seed, max_seq_len=P + steps + 8, max_prefill=max_prefill)
    try:
        prompt = inputs.prompt_tokens(shape, seed, P)
        ids, rows = om.generate_greedy(om.new_cache(P + steps + 1), prompt, steps)
        lg, am = gm.prefill(0, cuda_ints(prompt))
        assert_logits_close(_np(lg), rows[0], "prefill last row")
        assert_argmax(int(_np(am)[0]), ids[0], rows[0], "prefill argmax")
        for s in range(steps):
            lg, am = gm.decode(cuda_ints([ids[s]]), [P + s])
            assert_logits_close(_np(lg)[0], rows[s + 1], f"decode step {s + 1}")
            assert_argmax(int(_np(am)[0]), ids[s + 1], rows[s + 1], f"step {s + 1}")
        gm.reset(0)
        _, am = gm.prefill(0, cuda_ints(prompt), want_logits=False)
        out = gm.generate_greedy(am, steps)
        gm.sync()
        assert_ids_prefix([int(_np(am)[0])] + [int(v) for v in _np(out)[:, 0]], ids, rows)
    finally:
        gm.close()


@pytest.mark.parametrize("B", [2, 8, 16])
def test_q4k_batched_decode(torch, B):
    """B = 2, 8: the Q4_K GEMV chain with B rows; B = 16: the tensor-core
    GEMMs on tiles packed from the Q4_K rows."""
    shape = inputs.TINY
    om, gm = _pair(torch, shape, 0, max_seqs=B, max_seq_len=96, max_prefill=32)
    lens = [5 + 3 * b for b in range(B)]
    seqs = list(range(B))[::-1]
    try:
        caches = []
        for b in range(B):
            pre = inputs.batch_prefix_tokens(shape, 0, b, lens[b])
            c = om.new_cache(96)
            lg = om.forward(c, pre, 0)
            caches.append((c, orc.argmax_lowest(lg)))
            gm.prefill(seqs[b], cuda_ints(pre), want_logits=False)
        toks = [t for _, t in caches]
        pos = list(lens)
        for step in range(3):
            lg, am = gm.decode(cuda_ints(toks), pos, seqs=seqs)
            lg, am = _np(lg), _np(am)
            for b in range(B):
                o = om.forward(caches[b][0], [toks[b]], pos[b])
                assert_logits_close(lg[b], o, f"B={B} seq {b} step {step}")
                assert_argmax(int(am[b]), orc.argmax_lowest(o), o, f"B={B} seq {b} step {step}")
                toks[b] = int(am[b])
                pos[b] += 1
    finally:
        gm.close()


def test_q4k_all_logits_and_flag_checks(torch):
    from quantized_transformer_decode_gb300.qw3 import Qw3Error, Qw3Model
    shape = inputs.TINY
    om, gm = _pair(torch, shape, 6, max_seq_len=64, max_prefill=16)
    try:
        prompt = inputs.prompt_tokens(shape, 6, 21)
        want = om.forward(om.new_cache(64), prompt, 0, all_logits=True)
        lg, am = gm.forward_all_logits(0, cuda_ints(prompt))
        for i in range(want.shape[0]):
            assert_logits_close(_np(lg)[i], want[i], f"row {i}")
    finally:
        gm.close()
    with pytest.raises(Qw3Error):        # Q8_0 activations need Q8_0 weights
        Qw3Model.from_f32(shape, inputs.iter_weights(shape, 0), max_seq_len=16, max_prefill=16, flags=Q4K | 0x40)
    bad = inputs.Qwen3Shape(vocab=512, hidden=384, n_layers=1, n_heads=4, n_kv_heads=2, head_dim=64,
                            intermediate=768, tied=True)
    with pytest.raises(Qw3Error):        # hidden not a multiple of 256
        Qw3Model.from_f32(bad, inputs.iter_weights(bad, 0), max_seq_len=16, max_prefill=16, flags=Q4K)
