"""qw3_q8_0_gemv_splitk_noalloc (static scratch, no allocation) against
qw3_q8_0_gemv on the same buffers, two calls in a row, through the C ABI.

This file is collected last so that it also runs after every other test in
the same process (and it passes alone in a fresh one)."""
import numpy as np
import pytest

from oracle import qw3_oracle as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_transformer_decode_gb300 import build
    build.build()
    return t


def _bound(w, x):
    """f32 accumulation in two different orders: 2 K 2^-23 sum |w_k x_k|."""
    K = w.shape[1]
    return (np.abs(x.astype(np.float64)) @ np.abs(w.astype(np.float64)).T) * (2 * K * 2.0 ** -23) + 1e-30


@pytest.mark.parametrize("rows,cols,B", [(8, 16384, 1), (77, 4128, 3), (1024, 3072, 1), (5, 65536, 8),
                                         (4096, 1024, 2), (1, 32, 1)])
def test_two_calls_match_the_allocating_entry(torch, rows, cols, B):
    from quantized_transformer_decode_gb300 import qw3
    rng = np.random.default_rng([rows, cols, B, 9])
    blocks = orc.q8_0_quantize(rng.standard_normal((rows, cols), dtype=np.float32) * np.float32(0.02))
    w = orc.matrix_from_blocks(blocks, rows, cols)
    x = rng.standard_normal((B, cols), dtype=np.float32)
    Wd = torch.from_numpy(blocks).cuda()
    xd = torch.from_numpy(x).cuda()
    ref = torch.empty((B, rows), dtype=torch.float32, device="cuda")
    y1 = torch.full((B, rows), np.nan, dtype=torch.float32, device="cuda")
    y2 = torch.full((B, rows), np.nan, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    qw3.qw3_q8_0_gemv(Wd.data_ptr(), rows, cols, xd.data_ptr(), B, ref.data_ptr(), s)
    qw3.qw3_q8_0_gemv_splitk_noalloc(Wd.data_ptr(), rows, cols, xd.data_ptr(), B, y1.data_ptr(), s)
    qw3.qw3_q8_0_gemv_splitk_noalloc(Wd.data_ptr(), rows, cols, xd.data_ptr(), B, y2.data_ptr(), s)
    torch.cuda.synchronize()
    r, a, b = ref.cpu().numpy(), y1.cpu().numpy(), y2.cpu().numpy()
    bound = _bound(w, x)
    assert np.all(np.abs(a - r) <= bound), float(np.max(np.abs(a - r) / bound))
    assert np.all(np.abs(b - r) <= bound), float(np.max(np.abs(b - r) / bound))
    np.testing.assert_array_equal(a, b)   # fixed reduction order: the second call repeats the first


def test_sizes_beyond_the_scratch_are_rejected(torch):
    from quantized_transformer_decode_gb300 import qw3
    buf = torch.zeros(64, dtype=torch.float32, device="cuda")
    p = buf.data_ptr()
    with pytest.raises(qw3.Qw3Error) as e:
        qw3.qw3_q8_0_gemv_splitk_noalloc(p, 524289, 32, p, 1, p)
    assert e.value.status == qw3.QW3_ERR_SHAPE and "524288" in str(e.value)
    with pytest.raises(qw3.Qw3Error) as e:
        qw3.qw3_q8_0_gemv_splitk_noalloc(p, 262144, 32, p, 8, p)
    assert e.value.status == qw3.QW3_ERR_SHAPE
    with pytest.raises(qw3.Qw3Error) as e:
        qw3.qw3_q8_0_gemv_splitk_noalloc(p, 8, 48, p, 1, p)
    assert e.value.status == qw3.QW3_ERR_SHAPE
