"""The C-ABI library builds, loads and exports every entry point of
include/qw3.h, and its host-side argument checks answer before any device
work. No compute call runs here (no GPU needed)."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
HEADER = ROOT / "include" / "qw3.h"


@pytest.fixture(scope="module")
def L():
    from quantized_transformer_decode_gb300 import build, qw3
    build.build()
    return qw3.lib()


def header_functions():
    text = HEADER.read_text()
    return re.findall(r"QW3_API\s+[\w\s\*]*?\b(qw3_\w+)\s*\(", text)


def test_header_lists_the_binding_exports():
    from quantized_transformer_decode_gb300 import qw3
    assert header_functions() == list(qw3.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in header_functions():
        assert hasattr(L, name), name


def test_dynamic_symbol_table_is_exactly_the_api(L):
    import subprocess
    from quantized_transformer_decode_gb300 import qw3
    out = subprocess.run(["nm", "-D", "--defined-only", str(qw3.LIB_PATH)], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("nm not available")
    exported = sorted(ln.split()[-1] for ln in out.stdout.splitlines() if " T " in ln)
    assert exported == sorted(header_functions())


def test_status_strings(L):
    from quantized_transformer_decode_gb300 import qw3
    assert qw3.qw3_status_string(0) == "ok"
    assert "overflow" in qw3.qw3_status_string(qw3.QW3_ERR_KV_OVERFLOW)
    assert qw3.qw3_status_string(99) == "unknown status"


def test_struct_layouts_match_the_header(L):
    from quantized_transformer_decode_gb300 import qw3
    assert ctypes.sizeof(qw3.Qw3Config) == 14 * 4
    assert ctypes.sizeof(qw3.Qw3LayerWeights) == 11 * ctypes.sizeof(ctypes.c_void_p)
    assert qw3.Qw3Weights.on_device.offset == 4 * ctypes.sizeof(ctypes.c_void_p)


def _cfg(**kw):
    from quantized_transformer_decode_gb300 import qw3
    base = dict(vocab=4096, hidden=256, n_layers=2, n_heads=4, n_kv_heads=2, head_dim=64, intermediate=768,
                rms_eps=1e-6, rope_theta=1e6, tied_lm_head=1, max_seqs=1, max_seq_len=64, max_prefill=32,
                flags=0)
    base.update(kw)
    return qw3.Qw3Config(**base)


def _weights(n_layers=2):
    from quantized_transformer_decode_gb300 import qw3
    layers = (qw3.Qw3LayerWeights * n_layers)()
    for i in range(n_layers):
        for f, _ in qw3.Qw3LayerWeights._fields_:
            setattr(layers[i], f, 16)   # non-null; never dereferenced: validation fails first
    return qw3.Qw3Weights(token_embd=16, output=None, output_norm=16, layers=layers, on_device=1), layers


@pytest.mark.parametrize("kw,status", [
    (dict(hidden=250), 2),                    # H % 32
    (dict(intermediate=770), 2),              # I % 32
    (dict(n_heads=5), 2),                     # nh % nkv
    (dict(head_dim=96), 2),                   # head_dim not 64/128
    (dict(n_heads=32, n_kv_heads=2), 2),      # group 16 unsupported
    (dict(n_heads=130, n_kv_heads=65), 2),    # more than 64 kv heads
    (dict(max_seq_len=0), 2),
    (dict(rope_theta=0.0), 2),
    (dict(vocab=0), 2),
])
def test_create_rejects_bad_configs_before_device_work(L, kw, status):
    from quantized_transformer_decode_gb300 import qw3
    w, _keep = _weights()
    h = ctypes.c_void_p()
    rc = L.qw3_create(ctypes.byref(_cfg(**kw)), ctypes.byref(w), None, ctypes.byref(h))
    assert rc == status
    assert h.value is None
    assert qw3.qw3_last_error(0)


def test_create_rejects_null_pointers(L):
    w, _keep = _weights()
    h = ctypes.c_void_p()
    assert L.qw3_create(None, ctypes.byref(w), None, ctypes.byref(h)) == 1
    assert L.qw3_create(ctypes.byref(_cfg()), ctypes.byref(w), None, None) == 1
    untied = _cfg(tied_lm_head=0)
    assert L.qw3_create(ctypes.byref(untied), ctypes.byref(w), None, ctypes.byref(h)) == 1


def test_codec_entries_check_sizes_first(L):
    assert L.qw3_q8_0_quantize(16, 33, 16, None, None) == 2         # n % 32
    assert L.qw3_q8_0_quantize(18, 32, 16, None, None) == 1         # x misaligned
    assert L.qw3_q8_0_quantize(16, 32, 17, None, None) == 1         # blocks misaligned
    assert L.qw3_q8_0_quantize(None, 32, 16, None, None) == 1
    assert L.qw3_q8_0_quantize(None, 0, None, None, None) == 0      # empty is a no-op
    assert L.qw3_q8_0_dequantize(16, 31, 16, None) == 2
    assert L.qw3_q8_0_dequantize(16, -32, 16, None) == 1
    assert L.qw3_q8_0_gemv(16, 8, 48, 16, 1, 16, None) == 2         # cols % 32
    assert L.qw3_q8_0_gemv(16, 8, 64, 16, 9, 16, None) == 1         # B > 8
    assert L.qw3_q8_0_gemv(16, 0, 64, 16, 1, 16, None) == 0         # no rows: nothing to do


def test_gemm_entry_checks_arguments_before_device_work(L):
    """qw3_q8_0_gemm: sizes, alignment and the workspace are checked on the
    host, so every case here returns before a CUDA call (pointers are never
    dereferenced)."""
    ws = L.qw3_q8_0_gemm_workspace_bytes
    assert ws(128, 96, 4) == -1                                      # cols % 64
    assert ws(-1, 64, 4) == -1 and ws(128, 64, -1) == -1
    # pieces of 8704 bytes per (128-row tile, 64 columns) + 8 bytes of row
    # factors per padded row, then the packed activations: 4 bytes per value
    # of the padded rows + their inverse factors
    assert ws(128, 64, 4) == 8704 + 128 * 8 + 128 * 64 * 4 + 128 * 4
    assert ws(300, 1024, 130) == 3 * 16 * 8704 + 384 * 8 + 256 * 1024 * 4 + 256 * 4
    g = L.qw3_q8_0_gemm
    assert g(16, 8, 96, 16, 4, 16, 16, 1 << 20, None) == 2          # cols % 64
    assert g(None, 8, 64, 16, 4, 16, 16, 1 << 20, None) == 1        # null W
    assert g(17, 8, 64, 16, 4, 16, 16, 1 << 20, None) == 1          # W misaligned
    assert g(16, 8, 64, 24, 4, 16, 16, 1 << 20, None) == 1          # x not 16-byte aligned
    assert g(16, 8, 64, 16, 4, 16, 24, 1 << 20, None) == 1          # workspace misaligned
    assert g(16, 8, 64, 16, 4, 16, 16, 100, None) == 1              # workspace too small
    assert g(16, 8, 64, 16, 4, 16, None, 0, None) == 1              # no workspace
    assert g(16, 0, 64, 16, 4, 16, None, 0, None) == 0              # no rows: nothing to do
    assert g(16, 8, 64, 16, 0, 16, None, 0, None) == 0              # no activation rows


def test_model_calls_reject_null_model(L):
    n = ctypes.c_int32()
    assert L.qw3_seq_len(None, 0, ctypes.byref(n)) == 1
    assert L.qw3_reset(None, 0) == 1
    assert L.qw3_decode(None, 1, None, 16, None, None, None) == 1
    assert L.qw3_prefill(None, 0, 16, 1, None, None) == 1
    assert L.qw3_forward_all_logits(None, 0, 16, 1, 16, None) == 1
    assert L.qw3_destroy(None) == 0
    assert L.qw3_stream(None) is None


def test_missing_library_fails_loudly(tmp_path):
    """No fallback: with the shared library absent the binding raises instead
    of computing anything on the CPU."""
    import os
    import subprocess
    import sys
    code = ("import quantized_transformer_decode_gb300.qw3 as q\n"
            "try:\n    q.lib()\nexcept RuntimeError as e:\n    print('raised', e)\n")
    env = dict(os.environ, QW3_LIB=str(tmp_path / "absent" / "libqw3.so"))
    p = subprocess.run([sys.executable, "-c", code], cwd=str(ROOT), env=env, capture_output=True, text=True,
                       timeout=120)
    assert p.returncode == 0 and p.stdout.startswith("raised") and "not built" in p.stdout
