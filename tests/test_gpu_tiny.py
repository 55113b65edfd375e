"""GPU parity of the whole model on small configurations, through the C ABI.

The tiny Qwen3-shaped decoder (2 layers, hidden 256, 4/2 heads, head_dim
64, seed 0, prompt 32, 16 greedy steps) and a mid-sized one with the 0.6B
layer geometry (hidden 1024, 16/8 heads, head_dim 128, intermediate 3072)
but 2 layers and a ragged vocabulary, so that every kernel instantiation of
the decode and prefill paths runs against the oracle in seconds.
"""
import numpy as np
import pytest

from oracle import qw3_oracle as orc
from quantized_transformer_decode_gb300 import inputs
from parity import assert_argmax, assert_ids_prefix, assert_logits_close, build_pair, cuda_ints

pytestmark = pytest.mark.gpu

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


def run_greedy_case(torch, shape, seed, prompt_len, steps, flags=0, max_prefill=64, max_seq_len=None):
    """Prefill + free-running greedy (ids bit-exact) + teacher-forced logits."""
    om, gm = build_pair(shape, seed, max_seq_len=max_seq_len or prompt_len + steps + 8, max_prefill=max_prefill,
                        flags=flags)
    prompt = inputs.prompt_tokens(shape, seed, prompt_len)
    try:
        ids, ologits = om.generate_greedy(om.new_cache(prompt_len + steps + 1), prompt, steps)
        # teacher-forced: feed the oracle's ids, compare every row
        lg, am = gm.prefill(0, cuda_ints(prompt))
        assert_logits_close(_np(lg), ologits[0], "prefill last row")
        assert_argmax(int(_np(am)[0]), ids[0], ologits[0], "prefill argmax")
        for s in range(steps):
            lg, am = gm.decode(cuda_ints([ids[s]]), [prompt_len + s])
            assert_logits_close(_np(lg)[0], ologits[s + 1], f"decode step {s + 1}")
            assert_argmax(int(_np(am)[0]), ids[s + 1], ologits[s + 1], f"argmax at step {s + 1}")
        gm.sync()
        # free-running on a fresh sequence state: ids bit-exact
        gm.reset(0)
        _, am = gm.prefill(0, cuda_ints(prompt), want_logits=False)
        out = gm.generate_greedy(am, steps)
        gm.sync()
        got = [int(_np(am)[0])] + [int(v) for v in _np(out)[:, 0]]
        assert_ids_prefix(got, ids, ologits)
        assert gm.seq_len(0) == prompt_len + steps
        return om, gm, ids
    except Exception:
        gm.close()
        raise


def test_tiny_greedy_and_logits(torch):
    w = inputs.WORKLOADS["tiny"]
    _, gm, _ = run_greedy_case(torch, w.shape, w.seed, w.prompt_len, w.decode_steps)
    gm.close()


@pytest.mark.parametrize("flags", [0, 0x20, 0x80])
def test_tiny_tensor_core_prefill_head_dim_64(torch, flags):
    """head_dim 64 through the tensor-core prefill: a 300-token prompt in
    one chunk takes the tcgen05 GEMMs and the tcgen05 causal attention (one
    64-deep step per S product, 64-column O accumulators), with the f32,
    f16 and q8_0 caches; then decode against the oracle (the f16 and q8_0
    caches through the checks of their own test modules)."""
    if flags:
        from test_gpu_kv_f16 import _greedy_f16
        from test_gpu_kv_q8 import _greedy_q8
        (_greedy_f16 if flags == 0x20 else _greedy_q8)(inputs.TINY, 3, 300, 4, max_prefill=512)
        return
    _, gm, _ = run_greedy_case(torch, inputs.TINY, 3, 300, 4, max_prefill=512)
    gm.close()


PER_KERNEL = 0x8      # batch-1 decode through the per-kernel chain
TEST_NO_WAIT = 0x10   # waits on other CTAs give up at their first miss


@pytest.mark.parametrize("flags", [0x1, 0x2, 0x3])
def test_tiny_per_kernel_launch_modes(torch, flags):
    """The per-kernel decode path with direct launches, with and without
    programmatic dependent launch, against the oracle."""
    w = inputs.WORKLOADS["tiny"]
    _, gm, _ = run_greedy_case(torch, w.shape, w.seed, w.prompt_len, 6, flags=flags | PER_KERNEL)
    assert gm.decode_plan(1)[0] is False
    gm.close()


@pytest.mark.parametrize("prompt_len", [70, 600])
def test_long_capacity_split_over_clusters(torch, prompt_len):
    """A model built for 4096+ positions decodes batch 1 with each kv head's
    context split over several clusters whose partials merge in global
    memory; against the oracle at short and medium contexts (many splits
    hold no position at 70). Teacher-forced logits on every step; ids
    under the near-tie rule (at 600 tokens step 6 has two logits 1.7e-5
    apart: either is the greedy token at f32 precision)."""
    shape, seed, steps = MID, 7, 8
    om, gm = build_pair(shape, seed, max_seq_len=4200, max_prefill=256, flags=PER_KERNEL)
    try:
        prompt = inputs.prompt_tokens(shape, seed, prompt_len)
        ids, ologits = om.generate_greedy(om.new_cache(prompt_len + steps + 1), prompt, steps)
        lg, am = gm.prefill(0, cuda_ints(prompt))
        assert_logits_close(_np(lg), ologits[0], "prefill last row")
        assert_argmax(int(_np(am)[0]), ids[0], ologits[0], "prefill argmax")
        for s in range(steps):
            lg, am = gm.decode(cuda_ints([ids[s]]), [prompt_len + s])
            assert_logits_close(_np(lg)[0], ologits[s + 1], f"decode step {s + 1}")
            assert_argmax(int(_np(am)[0]), ids[s + 1], ologits[s + 1], f"argmax at step {s + 1}")
        gm.reset(0)
        _, am = gm.prefill(0, cuda_ints(prompt), want_logits=False)
        out = gm.generate_greedy(am, steps)
        gm.sync()
        assert_ids_prefix([int(_np(am)[0])] + [int(v) for v in _np(out)[:, 0]], ids, ologits)
    finally:
        gm.close()


def test_decode_plans(torch):
    w = inputs.WORKLOADS["tiny"]
    _, gm = build_pair(w.shape, w.seed, max_seq_len=64, max_prefill=32)
    assert gm.decode_plan(1) == (True, 1)
    assert gm.decode_plan(1)[0] is True
    gm.close()
    _, gm = build_pair(w.shape, w.seed, max_seq_len=64, max_prefill=32, flags=PER_KERNEL)
    assert gm.decode_plan(1) == (False, 2 + 5 * w.shape.n_layers)
    gm.close()


@pytest.mark.parametrize("case", ["tiny", "mid", "mid_long", "untied"])
def test_per_kernel_chain_greedy_and_logits(torch, case):
    """The per-kernel batch-1 chain (one launch per projection and
    attention) against the oracle (ids bit-exact, teacher-forced logits);
    the default batch-1 path, the persistent step kernel, runs the same
    cases in the tests above and below."""
    if case == "tiny":
        w = inputs.WORKLOADS["tiny"]
        _, gm, _ = run_greedy_case(torch, w.shape, w.seed, w.prompt_len, w.decode_steps, flags=PER_KERNEL)
    elif case == "mid":
        _, gm, _ = run_greedy_case(torch, MID, 4, prompt_len=70, steps=12, max_prefill=32, flags=PER_KERNEL)
    elif case == "mid_long":
        _, gm, _ = run_greedy_case(torch, MID, 6, prompt_len=460, steps=5, max_prefill=256, flags=PER_KERNEL)
    else:
        _, gm, _ = run_greedy_case(torch, MID_UNTIED, 5, prompt_len=40, steps=6, flags=PER_KERNEL)
    assert gm.decode_plan(1)[0] is False
    gm.close()


def test_step_kernel_long_context(torch):
    """The step kernel with more cached positions per attention unit than
    one ring slot of K/V rows holds, against the oracle."""
    _, gm, _ = run_greedy_case(torch, MID, 6, prompt_len=460, steps=5, max_prefill=256)
    assert gm.decode_plan(1)[0] is True
    gm.close()


def test_paths_agree_bitwise_on_ids(torch):
    """Persistent step kernel and per-kernel path: same greedy ids, logits close."""
    shape = MID
    prompt = inputs.prompt_tokens(shape, 4, 40)
    outs = []
    for flags in (0, PER_KERNEL):
        _, gm = build_pair(shape, 4, max_seq_len=64, max_prefill=64, flags=flags)
        _, am = gm.prefill(0, cuda_ints(prompt), want_logits=False)
        lg, am2 = gm.decode(am, [40])
        out = gm.generate_greedy(am2, 8)
        gm.sync()
        outs.append((_np(lg)[0], [int(v) for v in _np(out)[:, 0]]))
        gm.close()
    assert outs[0][1] == outs[1][1]
    assert_logits_close(outs[0][0], outs[1][0], "persistent vs per-kernel", max_abs=1e-4, rel_l2=1e-5)


def test_mid_greedy_and_logits(torch):
    _, gm, _ = run_greedy_case(torch, MID, 4, prompt_len=70, steps=12, max_prefill=32)
    gm.close()


def test_untied_lm_head(torch):
    _, gm, _ = run_greedy_case(torch, MID_UNTIED, 5, prompt_len=40, steps=6)
    gm.close()


def test_kv_cache_contents(torch):
    """K after Q/K-norm and RoPE, V as projected, at the right positions."""
    shape = inputs.TINY
    om, gm = build_pair(shape, 0, max_seq_len=64, max_prefill=16)
    prompt = inputs.prompt_tokens(shape, 0, 21)
    cache = om.new_cache(64)
    om.forward(cache, prompt, 0)
    nxt = 17
    om.forward(cache, [nxt], 21)
    gm.prefill(0, cuda_ints(prompt), want_logits=False)
    gm.decode(cuda_ints([nxt]), [21], want_logits=False)
    for layer in range(shape.n_layers):
        k, v = gm.read_kv(layer, 0, 0, 22)
        assert_logits_close(_np(k), cache.k[layer, :22], f"K layer {layer}", max_abs=1e-4, rel_l2=1e-5)
        assert_logits_close(_np(v), cache.v[layer, :22], f"V layer {layer}", max_abs=1e-4, rel_l2=1e-5)
    gm.close()


@pytest.mark.parametrize("B", [2, 3, 4, 8])
def test_batched_decode_matches_per_sequence_oracle(torch, B):
    """B sequences of different lengths in one decode call (B <= 4: GEMV path,
    B = 8: the tiled GEMM path), against the oracle run per sequence."""
    shape = inputs.TINY
    om, gm = build_pair(shape, 0, max_seqs=B, max_seq_len=96, max_prefill=32)
    lens = [5 + 11 * b for b in range(B)]
    seqs = list(range(B))[::-1]            # slot order differs from batch order
    caches = []
    try:
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
        gm.sync()
        for b in range(B):
            assert gm.seq_len(seqs[b]) == lens[b] + 3
    finally:
        gm.close()


def test_batched_generate_greedy(torch):
    shape = inputs.TINY
    B, steps = 3, 8
    om, gm = build_pair(shape, 0, max_seqs=B, max_seq_len=64, max_prefill=32)
    try:
        firsts, want, rows = [], [], []
        for b in range(B):
            pre = inputs.batch_prefix_tokens(shape, 0, b, 9 + b)
            ids, lg = om.generate_greedy(om.new_cache(64), pre, steps)
            want.append(ids)
            rows.append(lg)
            _, am = gm.prefill(b, cuda_ints(pre), want_logits=False)
            firsts.append(int(_np(am)[0]))
        out = _np(gm.generate_greedy(cuda_ints(firsts), steps))
        gm.sync()
        for b in range(B):
            assert_ids_prefix([firsts[b]] + [int(v) for v in out[:, b]], want[b], rows[b], f"sequence {b}")
    finally:
        gm.close()


def test_chunked_prefill_equals_single_pass(torch):
    """A prompt longer than max_prefill runs in chunks; the result is the
    oracle's single forward over the whole prompt."""
    shape = inputs.TINY
    om, gm = build_pair(shape, 0, max_seq_len=128, max_prefill=16)
    prompt = inputs.prompt_tokens(shape, 0, 53)
    lg, am = gm.prefill(0, cuda_ints(prompt))
    o = om.forward(om.new_cache(128), prompt, 0)
    assert_logits_close(_np(lg), o, "chunked prefill")
    assert_argmax(int(_np(am)[0]), orc.argmax_lowest(o), o, "chunked prefill")
    gm.close()


def test_prefill_in_two_calls(torch):
    shape = inputs.TINY
    om, gm = build_pair(shape, 0, max_seq_len=128, max_prefill=64)
    prompt = inputs.prompt_tokens(shape, 0, 40)
    gm.prefill(0, cuda_ints(prompt[:23]), want_logits=False)
    lg, _ = gm.prefill(0, cuda_ints(prompt[23:]))
    c = om.new_cache(128)
    om.forward(c, prompt[:23], 0)
    o = om.forward(c, prompt[23:], 23)
    assert_logits_close(_np(lg), o, "second prefill call")
    gm.close()


def test_contract_errors_leave_state_unchanged(torch):
    """Course 12.4: pos must equal the length; rows must fit. An error leaves
    every sequence length as it was."""
    from quantized_transformer_decode_gb300.qw3 import Qw3Error
    shape = inputs.TINY
    _, gm = build_pair(shape, 0, max_seqs=2, max_seq_len=40, max_prefill=16)
    prompt = inputs.prompt_tokens(shape, 0, 36)
    gm.prefill(0, cuda_ints(prompt), want_logits=False)
    with pytest.raises(Qw3Error) as e:
        gm.decode(cuda_ints([1]), [35])
    assert e.value.status == 3
    with pytest.raises(Qw3Error) as e:
        gm.prefill(0, cuda_ints(prompt[:5]))
    assert e.value.status == 4
    with pytest.raises(Qw3Error) as e:
        gm.generate_greedy(cuda_ints([1]), 5)
    assert e.value.status == 4
    with pytest.raises(Qw3Error) as e:
        gm.decode(cuda_ints([1, 2]), [36, 36], seqs=[0, 0])
    assert e.value.status == 1
    with pytest.raises(Qw3Error) as e:
        gm.decode(cuda_ints([1]), [0], seqs=[2])
    assert e.value.status == 1
    assert gm.seq_len(0) == 36 and gm.seq_len(1) == 0
    gm.generate_greedy(cuda_ints([1]), 4)
    gm.sync()
    assert gm.seq_len(0) == 40
    gm.close()


def test_truncate_then_redecode_is_reproducible(torch):
    shape = inputs.TINY
    _, gm = build_pair(shape, 0, max_seq_len=64, max_prefill=32)
    prompt = inputs.prompt_tokens(shape, 0, 20)
    gm.prefill(0, cuda_ints(prompt), want_logits=False)
    a, _ = gm.decode(cuda_ints([7]), [20])
    b, _ = gm.decode(cuda_ints([9]), [21])
    gm.truncate(0, 20)
    assert gm.seq_len(0) == 20
    a2, _ = gm.decode(cuda_ints([7]), [20])
    b2, _ = gm.decode(cuda_ints([9]), [21])
    np.testing.assert_array_equal(_np(a), _np(a2))
    np.testing.assert_array_equal(_np(b), _np(b2))
    gm.truncate(0, 99)
    assert gm.seq_len(0) == 22
    gm.close()


def test_trace_records_every_kernel(torch):
    shape = inputs.TINY
    _, gm = build_pair(shape, 0, max_seq_len=64, max_prefill=32, flags=0x4 | PER_KERNEL)
    assert gm.decode_plan(1)[0] is False
    gm.prefill(0, cuda_ints(inputs.prompt_tokens(shape, 0, 8)), want_logits=False)
    gm.decode(cuda_ints([3]), [8])
    tr = gm.read_trace()
    n_kernels = 2 + 5 * shape.n_layers
    assert tr.shape[0] >= 2 * n_kernels
    entry = tr[0:2 * n_kernels:2, 0].astype(np.int64)
    exits = tr[0:2 * n_kernels:2, 4].astype(np.int64)
    assert np.all(entry > 0) and np.all(exits >= entry)
    gm.close()


def test_step_kernel_trace(torch):
    """Step-kernel trace of the latest step: for the first CTA, per phase
    (cycle counter) inputs staged <= outputs published, phases in order."""
    shape = inputs.TINY
    _, gm = build_pair(shape, 0, max_seq_len=64, max_prefill=32, flags=0x4)
    assert gm.decode_plan(1)[0] is True
    _, am = gm.prefill(0, cuda_ints(inputs.prompt_tokens(shape, 0, 8)), want_logits=False)
    gm.generate_greedy(am, 3)
    tr = gm.read_trace(100000).astype(np.int64).reshape(-1)
    nph = 6 * shape.n_layers + 2
    first = tr[: nph * 4].reshape(nph, 4)
    assert first[0, 0] > 0 and first[0, 3] >= first[0, 0]
    for ph in range(1, nph):
        if ph % 6 in (1, 4, 5, 0) or ph == nph - 1:   # projection phases and the lm_head
            assert first[ph, 0] > 0 and first[ph, 3] >= first[ph, 0], ph
    outs = [first[ph, 3] for ph in range(1, nph) if first[ph, 3] > 0]
    assert np.all(np.diff(outs) >= 0)
    gm.close()


def test_step_kernel_wait_timeout_reported(torch):
    """With QW3_FLAG_TEST_NO_WAIT every wait on another CTA's data gives up at
    its first miss: the step runs to its end, qw3_sync reports
    QW3_ERR_TIMEOUT once, and the model stays usable (a fresh prefill and a
    batch-2 decode, which do not use the step kernel, match the oracle)."""
    from quantized_transformer_decode_gb300.qw3 import Qw3Error, QW3_ERR_TIMEOUT
    shape = inputs.TINY
    om, gm = build_pair(shape, 0, max_seqs=2, max_seq_len=64, max_prefill=32, flags=TEST_NO_WAIT)
    try:
        assert gm.decode_plan(1)[0] is True
        prompt = inputs.prompt_tokens(shape, 0, 20)
        _, am = gm.prefill(0, cuda_ints(prompt), want_logits=False)
        gm.generate_greedy(am, 4)
        with pytest.raises(Qw3Error) as e:
            gm.sync()
        assert e.value.status == QW3_ERR_TIMEOUT
        gm.sync()   # the status was cleared
        gm.reset(0)
        for b in range(2):
            gm.prefill(b, cuda_ints(prompt), want_logits=False)
        lg, _ = gm.decode(cuda_ints([5, 5]), [20, 20])
        gm.sync()
        cache = om.new_cache(32)
        om.forward(cache, prompt, 0)
        want = om.forward(cache, [5], 20)
        assert_logits_close(_np(lg)[0], want, "batch-2 decode after a timed-out step")
        assert_logits_close(_np(lg)[1], want, "batch-2 decode after a timed-out step")
    finally:
        gm.close()


@pytest.mark.parametrize("n", [1, 2, 7, 15])
def test_create_failure_cleans_up(torch, n, monkeypatch):
    """A failed device allocation during qw3_create returns QW3_ERR_OOM and
    frees what was allocated (QW3_FAULT_ALLOC_AT makes the n-th one fail);
    the next create succeeds."""
    from quantized_transformer_decode_gb300.qw3 import Qw3Error, QW3_ERR_OOM
    shape = inputs.TINY
    monkeypatch.setenv("QW3_FAULT_ALLOC_AT", str(n))
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        with pytest.raises(Qw3Error) as e:
            build_pair(shape, 0, max_seq_len=64, max_prefill=32)
        assert e.value.status == QW3_ERR_OOM
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    assert torch.cuda.mem_get_info()[0] >= free0 - (64 << 20)
    monkeypatch.delenv("QW3_FAULT_ALLOC_AT")
    _, gm = build_pair(shape, 0, max_seq_len=64, max_prefill=32)
    gm.close()
