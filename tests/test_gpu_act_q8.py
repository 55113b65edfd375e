"""GPU parity of the q8_0 activation mode ("Model files and quantization",
11.9: activations re-quantized to Q8_0 per 32-block on the fly, i32 block
dots times d_w * d_a) against the oracle's QLinear.q8act / set_activations.

Kernel level (qw3_q8_0_gemv_q8act), both sides see the same f32 x, so the
activation codes are the same integers and the results differ only by f32
rounding: each block's (d_w * d_a) * acc product rounds once, and the f32
additions of a row add at most cols/32 roundings of the running sum.

Model level (QW3_FLAG_ACT_Q8), the CUDA path's f32 activations differ from
the oracle's by reassociation error before they are quantized, so a value at
a code boundary lands one code apart; that moves the next layer's inputs by
a fraction of a quantum, which flips many of its codes, and so on: the two
q8_0-activation runs drift apart to the scale of the quantization noise
itself (the pages report the same of their own CPU q8_0 path against their
f32 GPU path: greedy tokens agree, logits differ visibly). So each row is
checked against the mode's own effect, the distance between the oracle's
q8_0-activation and f32-activation rows: the CUDA row is no farther from the
oracle's q8_0 row than that, its own distance to the CUDA f32-activation
row is of the same size (the quantization did happen, at the right
strength), and greedy ids agree wherever the oracle's top-2 margin exceeds
that distance. The exact arithmetic (same input, same codes) is checked at
the kernel level above.
"""
import numpy as np
import pytest

from oracle import qw3_oracle as orc
from quantized_transformer_decode_gb300 import inputs
from parity import MAX_ABS, REL_L2, TIE_MARGIN, assert_logits_close, build_pair, cuda_ints, row_errors

pytestmark = pytest.mark.gpu

ACT_Q8 = 0x40
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


def _q8act_bound(L, x):
    """f32 rounding bound of the integer path: 2^-23 per block product plus
    (cols/32) * 2^-24 of the running sum, both against sum |w| |x|."""
    wq = orc.matrix_from_blocks(L.blocks.reshape(-1), L.rows, L.cols).astype(np.float64)
    mag = np.abs(x.astype(np.float64)) @ np.abs(wq).T * 1.01 + 1e-30
    return mag * (2.0 ** -23 + (L.cols / 32) * 2.0 ** -24)


@pytest.mark.parametrize("rows,cols,B", [(8, 256, 1), (1000, 1024, 1), (4096, 1024, 3), (1024, 3072, 8),
                                         (6144, 1024, 2), (77, 12288, 1)])
def test_q8act_gemv_matches_oracle_on_the_same_input(torch, rows, cols, B):
    from quantized_transformer_decode_gb300 import qw3
    rng = np.random.default_rng([rows, cols, B, 8])
    wf = rng.standard_normal((rows, cols), dtype=np.float32) * np.float32(0.02)
    blocks = orc.q8_0_quantize(wf)
    L = orc.QLinear(blocks, rows, cols, keep_f64=False)
    x = (rng.standard_normal((B, cols)) * rng.uniform(0.01, 30.0, size=(B, 1))).astype(np.float32)
    want = L.q8act(x)
    y = _np(qw3.q8_0_gemv_q8act(torch.from_numpy(blocks).cuda(), rows, cols, torch.from_numpy(x).cuda()))
    err = np.abs(y.astype(np.float64) - want.astype(np.float64))
    bound = _q8act_bound(L, x)
    assert np.all(err <= bound), float(np.max(err / bound))
    # it is the integer path: much closer to the oracle's q8act than to the
    # f32-activation product
    assert np.max(np.abs(y - L(x))) > 10 * np.max(err)


def test_q8act_gemv_ties_round_half_away(torch):
    """Activation values at exact half-codes (d_a = 1): a round-half-even
    encoder would give different codes for 0.5, 2.5, -2.5 and a different
    result; the one-hot weight rows read single codes back."""
    from quantized_transformer_decode_gb300 import qw3
    cols = 256
    x = np.zeros((1, cols), np.float32)
    x[0, :6] = [127.0, 0.5, 1.5, 2.5, -2.5, -0.5]
    w = np.zeros((6, cols), np.float32)
    for r in range(6):
        w[r, 0] = 127.0
        w[r, r] += 0.0 if r == 0 else 1.0        # row r reads code r (times d_w = 1) plus 127 * 127
    blocks = orc.q8_0_quantize(w)
    L = orc.QLinear(blocks, 6, cols, keep_f64=False)
    want = L.q8act(x)[0]
    assert list(want - 127.0 * 127.0)[1:] == [1.0, 2.0, 3.0, -3.0, -1.0]
    y = _np(qw3.q8_0_gemv_q8act(torch.from_numpy(blocks).cuda(), 6, cols, torch.from_numpy(x).cuda()))[0]
    np.testing.assert_array_equal(y, want)


def test_q8act_gemv_nonfinite_and_zero(torch):
    from quantized_transformer_decode_gb300 import qw3
    rng = np.random.default_rng(3)
    rows, cols = 16, 512
    blocks = orc.q8_0_quantize(rng.standard_normal((rows, cols), dtype=np.float32))
    Wd = torch.from_numpy(blocks).cuda()
    x = np.zeros((2, cols), np.float32)
    x[1, 40] = np.nan
    y = _np(qw3.q8_0_gemv_q8act(Wd, rows, cols, torch.from_numpy(x).cuda()))
    assert not y[0].any()
    assert np.all(np.isnan(y[1]))


def test_q8act_gemv_argument_checks(torch):
    from quantized_transformer_decode_gb300 import qw3
    W = torch.zeros(34 * 8, dtype=torch.uint8, device="cuda")
    x = torch.zeros(64, dtype=torch.float32, device="cuda")
    y = torch.zeros(8, dtype=torch.float32, device="cuda")
    with pytest.raises(qw3.Qw3Error):
        qw3.qw3_q8_0_gemv_q8act(W.data_ptr(), 1, 32, x.data_ptr(), 1, y.data_ptr())      # cols % 256
    with pytest.raises(qw3.Qw3Error):
        qw3.qw3_q8_0_gemv_q8act(W.data_ptr(), 1, 256, x.data_ptr() + 4, 1, y.data_ptr())  # x alignment


def _mode_rows(om, prompt, steps, cap):
    """Oracle ids and rows in the q8_0 activation mode, and per row the
    distance to the f32-activation rows fed the same tokens."""
    om.set_activations("q8_0")
    ids, rows8 = om.generate_greedy(om.new_cache(cap), prompt, steps)
    om.set_activations("f32")
    rows32 = om.teacher_forced(om.new_cache(cap), prompt, ids[:steps])
    om.set_activations("q8_0")
    dist = [row_errors(a, b) for a, b in zip(rows8, rows32)]
    return ids, rows8, dist


def _assert_row(g8, g32, want, dist, what):
    ma, rel = dist
    r8 = row_errors(g8, want)
    assert r8[1] <= max(REL_L2, rel) and r8[0] <= max(MAX_ABS, ma), \
        f"{what}: {r8} from the oracle's q8_0 row, mode distance {dist}"
    rq = row_errors(g8, g32)[1]
    assert 0.5 * rel <= rq <= 2.0 * rel, f"{what}: q8_0 vs f32 on the GPU {rq:.3e}, oracle {rel:.3e}"


@pytest.mark.parametrize("case", ["tiny", "mid", "mid_batched"])
def test_act_q8_model_against_oracle_mode(torch, case):
    from quantized_transformer_decode_gb300.qw3 import Qw3Model
    shape, seed, P, steps, B = {"tiny": (inputs.TINY, 0, 32, 8, 1), "mid": (MID, 3, 40, 6, 1),
                                "mid_batched": (MID, 3, 40, 4, 8)}[case]
    cap = P + steps + 8
    om, gm = build_pair(shape, seed, max_seqs=B, max_seq_len=cap, max_prefill=64, flags=ACT_Q8)
    g32 = Qw3Model.from_f32(shape, inputs.iter_weights(shape, seed), max_seqs=B, max_seq_len=cap, max_prefill=64)
    try:
        prompt = inputs.prompt_tokens(shape, seed, P)
        ids, rows, dist = _mode_rows(om, prompt, steps, P + steps + 1)
        for b in range(B):
            lg, am = gm.prefill(b, cuda_ints(prompt))
            lf, _ = g32.prefill(b, cuda_ints(prompt))
            _assert_row(_np(lg), _np(lf), rows[0], dist[0], f"prefill row, seq {b}")
        for s in range(steps):
            lg, am = gm.decode(cuda_ints([ids[s]] * B), [P + s] * B)
            lf, _ = g32.decode(cuda_ints([ids[s]] * B), [P + s] * B)
            lg, lf = _np(lg), _np(lf)
            for b in range(B):
                _assert_row(lg[b], lf[b], rows[s + 1], dist[s + 1], f"step {s + 1}, seq {b}")
                got, want = int(_np(am)[b]), ids[s + 1]
                margin = max(TIE_MARGIN, dist[s + 1][0])
                assert got == want or rows[s + 1][want] - rows[s + 1][got] < margin
    finally:
        gm.close()
        g32.close()
