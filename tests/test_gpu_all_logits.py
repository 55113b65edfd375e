"""GPU parity of the all-logits forward (qw3_forward_all_logits: "A
transformer from scratch", 12.3.7 and 12.5, the multi-row step a speculative
verify runs) against the oracle's forward with all_logits=True: every
appended row's logits at the stated bar (max-abs 2e-3, rel-L2 1e-4) and each
row's argmax under the near-tie rule of parity.py.
"""
import numpy as np
import pytest

from oracle import qw3_oracle as orc
from quantized_transformer_decode_gb300 import inputs
from parity import assert_argmax, assert_logits_close, build_pair, cuda_ints

pytestmark = pytest.mark.gpu

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


def _check_rows(lg, am, want, what):
    assert lg.shape == want.shape
    for i in range(want.shape[0]):
        assert_logits_close(lg[i], want[i], f"{what} row {i}")
        assert_argmax(int(am[i]), orc.argmax_lowest(want[i]), want[i], f"{what} row {i}")


@pytest.mark.parametrize("case", ["tiny", "mid_chunks", "mid_tc"])
def test_all_logits_after_a_prompt(torch, case):
    """A verify block of `n` rows after a prompt: the SIMT GEMM path (tiny),
    several max_prefill chunks (each chunk's rows land at their offset), and
    one chunk wide enough for the tensor-core GEMM and prefill attention."""
    shape, seed, P, n, max_prefill = {
        "tiny": (inputs.TINY, 0, 32, 5, 64),
        "mid_chunks": (MID, 4, 40, 70, 32),
        "mid_tc": (MID, 5, 24, 260, 512),
    }[case]
    om, gm = build_pair(shape, seed, max_seq_len=P + n + 8, max_prefill=max_prefill)
    try:
        prompt = inputs.prompt_tokens(shape, seed, P)
        block = inputs.prompt_tokens(shape, seed + 100, n)
        cache = om.new_cache(P + n)
        om.forward(cache, prompt, 0)
        want = om.forward(cache, block, P, all_logits=True)
        gm.prefill(0, cuda_ints(prompt), want_logits=False)
        lg, am = gm.forward_all_logits(0, cuda_ints(block))
        _check_rows(_np(lg), _np(am), want, case)
        assert gm.seq_len(0) == P + n
    finally:
        gm.close()


def test_all_logits_from_position_zero_equals_prefill_rows(torch):
    """On an empty sequence the all-logits forward is a prefill that keeps
    every row: its last row is qw3_prefill's row."""
    shape = inputs.TINY
    om, gm = build_pair(shape, 1, max_seqs=2, max_seq_len=64, max_prefill=16)
    try:
        prompt = inputs.prompt_tokens(shape, 1, 37)
        want = om.forward(om.new_cache(64), prompt, 0, all_logits=True)
        lg, am = gm.forward_all_logits(0, cuda_ints(prompt))
        _check_rows(_np(lg), _np(am), want, "from zero")
        last, am1 = gm.prefill(1, cuda_ints(prompt))
        assert_logits_close(_np(last), _np(lg)[-1], "prefill vs all-logits last row")
    finally:
        gm.close()


def test_verify_accept_prefix_then_decode(torch):
    """The speculative-verify pattern: score a draft block, keep the accepted
    prefix (truncate), continue with decode; the decode rows equal the
    oracle's on the truncated cache."""
    shape = inputs.TINY
    om, gm = build_pair(shape, 2, max_seq_len=96, max_prefill=64)
    try:
        prompt = inputs.prompt_tokens(shape, 2, 20)
        draft = inputs.prompt_tokens(shape, 77, 6)
        gm.prefill(0, cuda_ints(prompt), want_logits=False)
        lg, am = gm.forward_all_logits(0, cuda_ints(draft))
        keep = 3                                   # accept draft[:3]
        gm.truncate(0, 20 + keep)
        nxt = int(_np(am)[keep - 1])
        lg2, am2 = gm.decode(cuda_ints([nxt]), [20 + keep])
        cache = om.new_cache(96)
        om.forward(cache, prompt, 0)
        om.forward(cache, draft[:keep], 20)
        want = om.forward(cache, [nxt], 20 + keep)
        assert_logits_close(_np(lg2)[0], want, "decode after a truncated verify block")
        assert_argmax(int(_np(am2)[0]), orc.argmax_lowest(want), want)
    finally:
        gm.close()


def test_single_row_equals_decode(torch):
    """n = 1: the all-logits forward (GEMM path) and a decode step (GEMV
    path) give the same row within the bar."""
    shape = inputs.TINY
    om, gm = build_pair(shape, 3, max_seqs=2, max_seq_len=64, max_prefill=16)
    try:
        prompt = inputs.prompt_tokens(shape, 3, 12)
        for sq in (0, 1):
            gm.prefill(sq, cuda_ints(prompt), want_logits=False)
        a, _ = gm.forward_all_logits(0, cuda_ints([9]))
        b, _ = gm.decode(cuda_ints([9]), [12], seqs=[1])
        assert_logits_close(_np(a)[0], _np(b)[0], "all-logits n=1 vs decode")
    finally:
        gm.close()


def test_all_logits_errors_leave_state_unchanged(torch):
    from quantized_transformer_decode_gb300.qw3 import Qw3Error, qw3_forward_all_logits
    shape = inputs.TINY
    _, gm = build_pair(shape, 0, max_seq_len=16, max_prefill=8)
    try:
        toks = cuda_ints(list(range(10)))
        lg = torch.empty((10, shape.vocab), dtype=torch.float32, device="cuda")
        gm.prefill(0, cuda_ints([1, 2, 3, 4, 5, 6, 7]), want_logits=False)
        with pytest.raises(Qw3Error):
            qw3_forward_all_logits(gm.h, 0, toks.data_ptr(), 10, lg.data_ptr(), 0)   # 7 + 10 > 16
        with pytest.raises(Qw3Error):
            qw3_forward_all_logits(gm.h, 0, toks.data_ptr(), 2, 0, 0)               # no logits buffer
        assert gm.seq_len(0) == 7
    finally:
        gm.close()
