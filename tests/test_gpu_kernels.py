"""GPU parity of the standalone entry points: Q8_0 encoder and decoder
(bit-exact against the oracle) and the raw-block GEMV (against an f64 dot of
the oracle's dequantised matrix), called through the C ABI."""
import numpy as np
import pytest

from oracle import qw3_oracle as orc
from quantized_transformer_decode_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_transformer_decode_gb300 import build
    build.build()
    return t


def _quantize(torch, x):
    from quantized_transformer_decode_gb300 import qw3
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    xb = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    blocks = qw3.q8_0_quantize(xb, status)
    torch.cuda.synchronize()
    return blocks.cpu().numpy(), int(status.item())


def special_blocks():
    """Blocks the pages' encoder definition fixes by hand (course 11.7)."""
    rows = []
    rows.append(np.zeros(32, np.float32))                                   # d == 0
    rows.append(np.float32(127.0) * np.linspace(-1, 1, 32, dtype=np.float32))
    tie = np.zeros(32, np.float32)                                          # amax 127 -> d = 1, inv_d = 1
    tie[0] = 127.0
    tie[1:8] = [0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5]                     # exact halves
    rows.append(tie)
    spike = np.zeros(32, np.float32)
    spike[17] = -3.0                                                        # single spike -> -127 only there
    rows.append(spike)
    rows.append(np.full(32, 1e-30, np.float32))                             # subnormal f16 scale -> 0
    rows.append(np.full(32, 6e-6, np.float32) * np.arange(32, dtype=np.float32))  # subnormal-f16 d
    big = np.zeros(32, np.float32)
    big[3] = np.float32(127.0 * 65504.0)                                    # d = 65504, largest f16
    rows.append(big)
    huge = np.zeros(32, np.float32)
    huge[5] = np.float32(1e30)                                              # d overflows f16 -> inf
    rows.append(huge)
    tiny = np.zeros(32, np.float32)
    tiny[0] = np.float32(1.27e-37)                                          # d ~ 1e-39: 1/d overflows f32
    tiny[1] = -np.float32(1.27e-37)
    tiny[2] = np.float32(5e-38)
    rows.append(tiny)
    return np.concatenate(rows)


def test_quantize_bit_exact_uniform(torch):
    x = inputs.uniform_block_values(7, 32 * 40000 + 32 * 3)
    got, st = _quantize(torch, x)
    assert st == 0
    np.testing.assert_array_equal(got, orc.q8_0_quantize(x))


def test_quantize_bit_exact_special_blocks(torch):
    x = special_blocks()
    got, st = _quantize(torch, x)
    assert st == 0
    with np.errstate(all="ignore"):
        want = orc.q8_0_quantize(x)
    np.testing.assert_array_equal(got.reshape(-1, 34), want.reshape(-1, 34))


def test_quantize_weight_distribution_bit_exact(torch):
    shape = inputs.TINY
    for name, kind, arr in inputs.iter_weights(shape, 0):
        if kind == "linear":
            got, st = _quantize(torch, arr.reshape(-1))
            assert st == 0
            np.testing.assert_array_equal(got, orc.q8_0_quantize(arr), err_msg=name)


def test_quantize_nonfinite_block_zeroed_with_status(torch):
    x = inputs.uniform_block_values(3, 32 * 4)
    x[40] = np.nan
    x[100] = np.inf
    got, st = _quantize(torch, x)
    assert st == 5
    g = got.reshape(4, 34)
    assert not g[1].any() and not g[3].any()
    ok = np.concatenate([x[0:32], x[64:96]])
    np.testing.assert_array_equal(np.concatenate([g[0], g[2]]), orc.q8_0_quantize(ok))


def test_quantize_empty_is_noop(torch):
    from quantized_transformer_decode_gb300 import qw3
    qw3.qw3_q8_0_quantize(0, 0, 0)


def test_dequantize_exact(torch):
    from quantized_transformer_decode_gb300 import qw3
    x = np.concatenate([inputs.uniform_block_values(11, 32 * 5000), special_blocks()[:32 * 7]])
    blocks = orc.q8_0_quantize(x)
    b = torch.from_numpy(blocks).cuda()
    y = qw3.q8_0_dequantize(b, x.size).cpu().numpy()
    np.testing.assert_array_equal(y, orc.q8_0_dequantize(blocks, x.size))


def _gemv_bound(w, x):
    """f32-accumulation error bound: K * 2^-23 relative to sum |w_k x_k|."""
    K = w.shape[1]
    return (np.abs(x.astype(np.float64)) @ np.abs(w.astype(np.float64)).T) * (K * 2.0 ** -23) + 1e-30


@pytest.mark.parametrize("rows,cols,B", [(1, 32, 1), (7, 256, 1), (129, 1024, 2), (1000, 3072, 3),
                                         (333, 4128, 4), (64, 2048, 8), (4096, 1024, 5)])
def test_raw_gemv(torch, rows, cols, B):
    from quantized_transformer_decode_gb300 import qw3
    rng = np.random.default_rng([rows, cols, B])
    wf = (rng.standard_normal((rows, cols), dtype=np.float32) * np.float32(0.02))
    blocks = orc.q8_0_quantize(wf)
    w = orc.matrix_from_blocks(blocks, rows, cols)
    x = rng.standard_normal((B, cols), dtype=np.float32)
    want = x.astype(np.float64) @ w.astype(np.float64).T
    y = qw3.q8_0_gemv(torch.from_numpy(blocks).cuda(), rows, cols, torch.from_numpy(x).cuda()).cpu().numpy()
    err = np.abs(y - want)
    assert np.all(err <= _gemv_bound(w, x)), float(np.max(err / _gemv_bound(w, x)))


def test_raw_gemv_one_hot_returns_a_column(torch):
    """A one-hot x returns column k of d*q exactly (single product, no sum)."""
    from quantized_transformer_decode_gb300 import qw3
    rows, cols = 77, 512
    rng = np.random.default_rng(5)
    blocks = orc.q8_0_quantize(rng.standard_normal((rows, cols), dtype=np.float32))
    w = orc.matrix_from_blocks(blocks, rows, cols)
    for k in (0, 31, 32, 511):
        x = np.zeros((1, cols), np.float32)
        x[0, k] = 1.0
        y = qw3.q8_0_gemv(torch.from_numpy(blocks).cuda(), rows, cols, torch.from_numpy(x).cuda()).cpu().numpy()
        np.testing.assert_array_equal(y[0], w[:, k])


def test_raw_gemv_unaligned_input_takes_the_general_path(torch):
    """x 4 bytes off a 16-byte boundary: the 2-byte-load path, same result
    bound as the 128-bit streaming path."""
    from quantized_transformer_decode_gb300 import qw3
    rows, cols = 129, 1024
    rng = np.random.default_rng(17)
    blocks = orc.q8_0_quantize(rng.standard_normal((rows, cols), dtype=np.float32) * np.float32(0.02))
    w = orc.matrix_from_blocks(blocks, rows, cols)
    x = rng.standard_normal((1, cols), dtype=np.float32)
    xd = torch.zeros(cols + 1, dtype=torch.float32, device="cuda")
    xd[1:] = torch.from_numpy(x[0]).cuda()
    y = torch.empty((1, rows), dtype=torch.float32, device="cuda")
    Wd = torch.from_numpy(blocks).cuda()
    qw3.qw3_q8_0_gemv(Wd.data_ptr(), rows, cols, xd.data_ptr() + 4, 1, y.data_ptr())
    want = x.astype(np.float64) @ w.astype(np.float64).T
    err = np.abs(_np_cpu(y) - want)
    assert np.all(err <= _gemv_bound(w, x))


def _np_cpu(t):
    import torch as _t
    _t.cuda.synchronize()
    return t.cpu().numpy()
