"""GPU parity of the tensor-core GEMM (qw3_q8_0_gemm: raw Q8_0 weights, f32
activations; the product prefill and large batches run) against the oracle's
dequantised weights in an f64 matmul ("Model files and quantization", 11.6).

The bar is f32 accumulation: elementwise within 2^-17 of sum |w x| (the
operand split keeps 22 bits, and each tensor-core accumulation chain is a
few K steps long before it is added into an f32 master with round to
nearest), and no systematic shrinkage: on all-positive data, where the
tensor core's truncating accumulation would pull every result toward zero
by ~1.6e-8 per MMA along K (1e-4 at K = 12288), the mean relative error must
stay within 5e-6.
"""
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


def _case(rows, cols, M, seed, positive=False):
    rng = np.random.default_rng([rows, cols, M, seed])
    w = rng.standard_normal((rows, cols)).astype(np.float32) * np.float32(0.02)
    x = rng.standard_normal((M, cols)).astype(np.float32)
    if positive:
        w, x = np.abs(w), np.abs(x)
    blocks = orc.q8_0_quantize(w.reshape(-1))
    wd = orc.q8_0_dequantize(blocks, rows * cols).reshape(rows, cols).astype(np.float64)
    return blocks, x, x.astype(np.float64) @ wd.T, np.abs(x.astype(np.float64)) @ np.abs(wd).T


def _gemm(torch, blocks, rows, cols, x):
    from quantized_transformer_decode_gb300 import qw3
    return qw3.q8_0_gemm(torch.from_numpy(blocks).cuda(), rows, cols, torch.from_numpy(x).cuda()).cpu().numpy()


# (rows, cols, M): ragged row and column tiles; one K step; 16 K steps over
# m-tile pairs (4096 x 1280 fills the GPU with two m-tiles per CTA; 6144 x
# 896 has 7 row tiles, so the last CTA row holds one); the longest
# contraction of the 8B geometry
@pytest.mark.parametrize("rows,cols,M", [(1000, 1024, 300), (128, 64, 1), (257, 3072, 33), (4096, 1024, 1280),
                                         (6144, 1024, 896), (1024, 12288, 256), (77, 4096, 130)])
def test_gemm_elementwise(torch, rows, cols, M):
    blocks, x, want, mag = _case(rows, cols, M, 0)
    y = _gemm(torch, blocks, rows, cols, x)
    err = np.abs(y - want)
    bound = mag * 2.0 ** -17 + 1e-30
    assert np.all(err <= bound), f"worst error {float(np.max(err / bound)):.2f} x the bound"
    rel = np.linalg.norm(y - want) / np.linalg.norm(want)
    assert rel <= 5e-6, f"rel-L2 {rel:.3e}"


@pytest.mark.parametrize("cols", [4096, 12288])
def test_gemm_no_systematic_shrinkage(torch, cols):
    rows, M = 1024, 256
    blocks, x, want, _ = _case(rows, cols, M, 1, positive=True)
    y = _gemm(torch, blocks, rows, cols, x)
    bias = float(np.mean((y - want) / want))
    assert abs(bias) <= 5e-6, f"mean relative error {bias:.3e}"


def test_gemm_argument_checks(torch):
    from quantized_transformer_decode_gb300 import qw3
    from quantized_transformer_decode_gb300.qw3 import Qw3Error
    assert qw3.qw3_q8_0_gemm_workspace_bytes(128, 96, 4) == -1          # cols % 64
    assert qw3.qw3_q8_0_gemm_workspace_bytes(128, 64, 4) > 0
    blocks, x, _, _ = _case(128, 64, 4, 2)
    W = torch.from_numpy(blocks).cuda()
    xg = torch.from_numpy(x).cuda()
    y = torch.zeros((4, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(Qw3Error):                                         # workspace too small
        qw3.qw3_q8_0_gemm(W.data_ptr(), 128, 64, xg.data_ptr(), 4, y.data_ptr(), ws.data_ptr(), 16)
    with pytest.raises(Qw3Error):                                         # cols not a multiple of 64
        qw3.qw3_q8_0_gemm(W.data_ptr(), 128, 96, xg.data_ptr(), 4, y.data_ptr(), ws.data_ptr(), 16)
    qw3.qw3_q8_0_gemm(W.data_ptr(), 128, 64, xg.data_ptr(), 0, y.data_ptr(), ws.data_ptr(), 16)   # M == 0: no-op
    torch.cuda.synchronize()
    assert not y.any()
