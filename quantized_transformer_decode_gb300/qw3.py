"""Python binding of libqw3, the C ABI declared in include/qw3.h.

Argument marshalling only: every step of the forward pass runs in the CUDA
library. The module-level functions carry the C names and take raw pointers
(ints) like the C entry points; `Qw3Model` wraps them for torch tensors.
Importing this module does not need a GPU; loading the library does need
libqw3.so, and a missing library is an error, never a fallback.
"""
from __future__ import annotations

import ctypes
import os
from pathlib import Path
from typing import Iterable, Optional, Sequence

import numpy as np

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libqw3.so"

QW3_OK = 0
QW3_ERR_INVALID_ARG = 1
QW3_ERR_SHAPE = 2
QW3_ERR_SEQ_POS = 3
QW3_ERR_KV_OVERFLOW = 4
QW3_ERR_NONFINITE = 5
QW3_ERR_OOM = 6
QW3_ERR_CUDA = 7
QW3_ERR_TIMEOUT = 8

QW3_FLAG_NO_GRAPH = 0x1
QW3_FLAG_NO_PDL = 0x2
QW3_FLAG_TRACE = 0x4
QW3_FLAG_PER_KERNEL = 0x8
QW3_FLAG_TEST_NO_WAIT = 0x10
QW3_FLAG_KV_F16 = 0x20
QW3_FLAG_ACT_Q8 = 0x40
QW3_FLAG_KV_Q8 = 0x80
QW3_FLAG_WEIGHTS_Q4_K = 0x100

# Every entry point of include/qw3.h, in declaration order.
EXPORTS = (
    "qw3_create", "qw3_destroy", "qw3_prefill", "qw3_forward_all_logits", "qw3_decode", "qw3_generate_greedy",
    "qw3_reset", "qw3_truncate", "qw3_seq_len", "qw3_debug_read_kv", "qw3_debug_read_trace",
    "qw3_decode_plan", "qw3_sync", "qw3_stream", "qw3_status_string", "qw3_last_error",
    "qw3_q8_0_quantize", "qw3_q8_0_dequantize", "qw3_q8_0_gemv", "qw3_q8_0_gemv_q8act",
    "qw3_q4_k_quantize", "qw3_q4_k_dequantize", "qw3_q4_k_gemv", "qw3_q8_0_gemv_splitk_noalloc",
    "qw3_q8_0_gemm_workspace_bytes", "qw3_q8_0_gemm",
)


class Qw3Config(ctypes.Structure):
    _fields_ = [
        ("vocab", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_layers", ctypes.c_int32),
        ("n_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("intermediate", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
        ("tied_lm_head", ctypes.c_int32), ("max_seqs", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
        ("max_prefill", ctypes.c_int32), ("flags", ctypes.c_int32),
    ]


class Qw3LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "attn_q", "attn_k", "attn_v", "attn_output", "ffn_gate", "ffn_up", "ffn_down",
        "attn_norm", "attn_q_norm", "attn_k_norm", "ffn_norm")]


class Qw3Weights(ctypes.Structure):
    _fields_ = [
        ("token_embd", ctypes.c_void_p), ("output", ctypes.c_void_p), ("output_norm", ctypes.c_void_p),
        ("layers", ctypes.POINTER(Qw3LayerWeights)), ("on_device", ctypes.c_int32),
    ]


class Qw3Error(RuntimeError):
    """A libqw3 call returned a non-zero status."""

    def __init__(self, status: int, message: str):
        super().__init__(f"[{status}] {message}")
        self.status = status


_lib = None

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64


def lib() -> ctypes.CDLL:
    """Load libqw3.so (built by quantized_transformer_decode_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    path = Path(os.environ.get("QW3_LIB", LIB_PATH))
    if not path.exists():
        raise RuntimeError(f"{path} is not built: run `python -m quantized_transformer_decode_gb300.build`")
    L = ctypes.CDLL(str(path))
    sig = {
        "qw3_create": (ctypes.c_int, [ctypes.POINTER(Qw3Config), ctypes.POINTER(Qw3Weights), _P, ctypes.POINTER(_P)]),
        "qw3_destroy": (ctypes.c_int, [_P]),
        "qw3_prefill": (ctypes.c_int, [_P, _I32, _P, _I32, _P, _P]),
        "qw3_forward_all_logits": (ctypes.c_int, [_P, _I32, _P, _I32, _P, _P]),
        "qw3_decode": (ctypes.c_int, [_P, _I32, _P, _P, _P, _P, _P]),
        "qw3_generate_greedy": (ctypes.c_int, [_P, _I32, _P, _I32, _P, _P]),
        "qw3_reset": (ctypes.c_int, [_P, _I32]),
        "qw3_truncate": (ctypes.c_int, [_P, _I32, _I32]),
        "qw3_seq_len": (ctypes.c_int, [_P, _I32, ctypes.POINTER(_I32)]),
        "qw3_debug_read_kv": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _P, _P]),
        "qw3_debug_read_trace": (ctypes.c_int, [_P, _P, _I32, ctypes.POINTER(_I32)]),
        "qw3_decode_plan": (ctypes.c_int, [_P, _I32, ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
        "qw3_sync": (ctypes.c_int, [_P]),
        "qw3_stream": (_P, [_P]),
        "qw3_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "qw3_last_error": (ctypes.c_char_p, [_P]),
        "qw3_q8_0_quantize": (ctypes.c_int, [_P, _I64, _P, _P, _P]),
        "qw3_q8_0_dequantize": (ctypes.c_int, [_P, _I64, _P, _P]),
        "qw3_q8_0_gemv": (ctypes.c_int, [_P, _I32, _I32, _P, _I32, _P, _P]),
        "qw3_q8_0_gemv_q8act": (ctypes.c_int, [_P, _I32, _I32, _P, _I32, _P, _P]),
        "qw3_q4_k_quantize": (ctypes.c_int, [_P, _I64, _P, _P, _P]),
        "qw3_q4_k_dequantize": (ctypes.c_int, [_P, _I64, _P, _P]),
        "qw3_q4_k_gemv": (ctypes.c_int, [_P, _I32, _I32, _P, _I32, _P, _P]),
        "qw3_q8_0_gemv_splitk_noalloc": (ctypes.c_int, [_P, _I32, _I32, _P, _I32, _P, _P]),
        "qw3_q8_0_gemm_workspace_bytes": (_I64, [_I32, _I32, _I32]),
        "qw3_q8_0_gemm": (ctypes.c_int, [_P, _I32, _I32, _P, _I32, _P, _P, _I64, _P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _check(rc: int, handle=None) -> None:
    if rc != QW3_OK:
        L = lib()
        msg = (L.qw3_last_error(handle) or b"").decode(errors="replace")
        raise Qw3Error(rc, msg or L.qw3_status_string(rc).decode())


def _i32_array(vals: Optional[Sequence[int]]):
    if vals is None:
        return None
    arr = (ctypes.c_int32 * len(vals))(*[int(v) for v in vals])
    return arr


# ---------------------------------------------------------------- C names

def qw3_create(cfg: Qw3Config, weights: Qw3Weights, stream: int = 0) -> int:
    h = _P()
    rc = lib().qw3_create(ctypes.byref(cfg), ctypes.byref(weights), stream or None, ctypes.byref(h))
    _check(rc)
    return h.value


def qw3_destroy(h: int) -> None:
    _check(lib().qw3_destroy(h), h)


def qw3_prefill(h: int, seq: int, tokens_ptr: int, n: int, last_logits_ptr: int = 0, argmax_ptr: int = 0) -> None:
    _check(lib().qw3_prefill(h, seq, tokens_ptr, n, last_logits_ptr or None, argmax_ptr or None), h)


def qw3_forward_all_logits(h: int, seq: int, tokens_ptr: int, n: int, logits_ptr: int, argmax_ptr: int = 0) -> None:
    _check(lib().qw3_forward_all_logits(h, seq, tokens_ptr, n, logits_ptr or None, argmax_ptr or None), h)


def qw3_decode(h: int, B: int, seqs: Optional[Sequence[int]], tokens_ptr: int, pos: Sequence[int],
               logits_ptr: int = 0, argmax_ptr: int = 0) -> None:
    _check(lib().qw3_decode(h, B, _i32_array(seqs), tokens_ptr, _i32_array(pos), logits_ptr or None,
                            argmax_ptr or None), h)


def qw3_generate_greedy(h: int, B: int, seqs: Optional[Sequence[int]], n_steps: int, first_ptr: int,
                        out_ptr: int) -> None:
    _check(lib().qw3_generate_greedy(h, B, _i32_array(seqs), n_steps, first_ptr, out_ptr or None), h)


def qw3_reset(h: int, seq: int) -> None:
    _check(lib().qw3_reset(h, seq), h)


def qw3_truncate(h: int, seq: int, keep_len: int) -> None:
    _check(lib().qw3_truncate(h, seq, keep_len), h)


def qw3_seq_len(h: int, seq: int) -> int:
    n = _I32()
    _check(lib().qw3_seq_len(h, seq, ctypes.byref(n)), h)
    return n.value


def qw3_debug_read_kv(h: int, layer: int, seq: int, pos0: int, n: int, k_ptr: int, v_ptr: int) -> None:
    _check(lib().qw3_debug_read_kv(h, layer, seq, pos0, n, k_ptr, v_ptr), h)


def qw3_debug_read_trace(h: int, max_records: int) -> np.ndarray:
    out = np.zeros((max_records, 8), dtype=np.uint64)
    n = _I32()
    _check(lib().qw3_debug_read_trace(h, out.ctypes.data, max_records, ctypes.byref(n)), h)
    return out[:n.value]


def qw3_decode_plan(h: int, B: int) -> tuple[bool, int]:
    """(uses the persistent step kernel, kernel launches per step)."""
    pers, lps = _I32(), _I32()
    _check(lib().qw3_decode_plan(h, B, ctypes.byref(pers), ctypes.byref(lps)), h)
    return bool(pers.value), lps.value


def qw3_sync(h: int) -> None:
    _check(lib().qw3_sync(h), h)


def qw3_stream(h: int) -> int:
    return lib().qw3_stream(h) or 0


def qw3_status_string(status: int) -> str:
    return lib().qw3_status_string(status).decode()


def qw3_last_error(h: int = 0) -> str:
    return (lib().qw3_last_error(h or None) or b"").decode(errors="replace")


def qw3_q8_0_quantize(x_ptr: int, n: int, blocks_ptr: int, status_ptr: int = 0, stream: int = 0) -> None:
    _check(lib().qw3_q8_0_quantize(x_ptr, n, blocks_ptr, status_ptr or None, stream or None))


def qw3_q8_0_dequantize(blocks_ptr: int, n: int, y_ptr: int, stream: int = 0) -> None:
    _check(lib().qw3_q8_0_dequantize(blocks_ptr, n, y_ptr, stream or None))


def qw3_q8_0_gemv(W_ptr: int, rows: int, cols: int, x_ptr: int, B: int, y_ptr: int, stream: int = 0) -> None:
    _check(lib().qw3_q8_0_gemv(W_ptr, rows, cols, x_ptr, B, y_ptr, stream or None))


def qw3_q8_0_gemv_q8act(W_ptr: int, rows: int, cols: int, x_ptr: int, B: int, y_ptr: int, stream: int = 0) -> None:
    _check(lib().qw3_q8_0_gemv_q8act(W_ptr, rows, cols, x_ptr, B, y_ptr, stream or None))


def qw3_q4_k_quantize(x_ptr: int, n: int, blocks_ptr: int, status_ptr: int = 0, stream: int = 0) -> None:
    _check(lib().qw3_q4_k_quantize(x_ptr, n, blocks_ptr, status_ptr or None, stream or None))


def qw3_q4_k_dequantize(blocks_ptr: int, n: int, y_ptr: int, stream: int = 0) -> None:
    _check(lib().qw3_q4_k_dequantize(blocks_ptr, n, y_ptr, stream or None))


def qw3_q4_k_gemv(W_ptr: int, rows: int, cols: int, x_ptr: int, B: int, y_ptr: int, stream: int = 0) -> None:
    _check(lib().qw3_q4_k_gemv(W_ptr, rows, cols, x_ptr, B, y_ptr, stream or None))


def qw3_q8_0_gemv_splitk_noalloc(W_ptr: int, rows: int, cols: int, x_ptr: int, B: int, y_ptr: int,
                                 stream: int = 0) -> None:
    _check(lib().qw3_q8_0_gemv_splitk_noalloc(W_ptr, rows, cols, x_ptr, B, y_ptr, stream or None))


def qw3_q8_0_gemm_workspace_bytes(rows: int, cols: int, M: int) -> int:
    return int(lib().qw3_q8_0_gemm_workspace_bytes(rows, cols, M))


def qw3_q8_0_gemm(W_ptr: int, rows: int, cols: int, x_ptr: int, M: int, y_ptr: int, ws_ptr: int, ws_bytes: int,
                  stream: int = 0) -> None:
    _check(lib().qw3_q8_0_gemm(W_ptr, rows, cols, x_ptr, M, y_ptr, ws_ptr or None, ws_bytes, stream or None))


# ---------------------------------------------------------- torch wrapper

def _torch():
    import torch
    return torch


def _stream_ptr() -> int:
    torch = _torch()
    return torch.cuda.current_stream().cuda_stream


def q8_0_quantize(x, status=None):
    """Encode a CUDA f32 tensor (numel % 32 == 0) to Q8_0 bytes on the
    current torch stream. Returns a uint8 tensor of numel/32*34 bytes."""
    torch = _torch()
    x = x.contiguous()
    out = torch.empty(x.numel() // 32 * 34, dtype=torch.uint8, device=x.device)
    qw3_q8_0_quantize(x.data_ptr(), x.numel(), out.data_ptr(), status.data_ptr() if status is not None else 0,
                      _stream_ptr())
    return out


def q8_0_dequantize(blocks, n: int):
    torch = _torch()
    y = torch.empty(n, dtype=torch.float32, device=blocks.device)
    qw3_q8_0_dequantize(blocks.data_ptr(), n, y.data_ptr(), _stream_ptr())
    return y


def q8_0_gemv(W, rows: int, cols: int, x):
    torch = _torch()
    x = x.contiguous()
    B = x.shape[0] if x.dim() == 2 else 1
    y = torch.empty((B, rows), dtype=torch.float32, device=x.device)
    qw3_q8_0_gemv(W.data_ptr(), rows, cols, x.data_ptr(), B, y.data_ptr(), _stream_ptr())
    return y


def q8_0_gemm(W, rows: int, cols: int, x):
    """y = x . W^T for raw Q8_0 W [rows][cols] and CUDA f32 x [M][cols] on the
    tensor cores (qw3_q8_0_gemm), the workspace allocated here."""
    torch = _torch()
    x = x.contiguous()
    M = x.shape[0]
    y = torch.empty((M, rows), dtype=torch.float32, device=x.device)
    nbytes = qw3_q8_0_gemm_workspace_bytes(rows, cols, M)
    if nbytes < 0:
        raise Qw3Error(QW3_ERR_SHAPE, "cols must be a multiple of 64")
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=x.device)
    qw3_q8_0_gemm(W.data_ptr(), rows, cols, x.data_ptr(), M, y.data_ptr(), ws.data_ptr(), nbytes, _stream_ptr())
    return y


def q8_0_gemv_q8act(W, rows: int, cols: int, x):
    """y = W . Q8_0(x) row by row (qw3_q8_0_gemv_q8act)."""
    torch = _torch()
    x = x.contiguous()
    B = x.shape[0] if x.dim() == 2 else 1
    y = torch.empty((B, rows), dtype=torch.float32, device=x.device)
    qw3_q8_0_gemv_q8act(W.data_ptr(), rows, cols, x.data_ptr(), B, y.data_ptr(), _stream_ptr())
    return y


def q4_k_quantize(x, status=None):
    """f32 CUDA tensor (numel % 256 == 0) -> uint8 Q4_K wire bytes."""
    torch = _torch()
    x = x.contiguous()
    out = torch.empty(x.numel() // 256 * 144, dtype=torch.uint8, device=x.device)
    qw3_q4_k_quantize(x.data_ptr(), x.numel(), out.data_ptr(), status.data_ptr() if status is not None else 0,
                      _stream_ptr())
    return out


def q4_k_dequantize(blocks, n: int):
    torch = _torch()
    y = torch.empty(n, dtype=torch.float32, device=blocks.device)
    qw3_q4_k_dequantize(blocks.data_ptr(), n, y.data_ptr(), _stream_ptr())
    return y


def q4_k_gemv(W, rows: int, cols: int, x):
    torch = _torch()
    x = x.contiguous()
    B = x.shape[0] if x.dim() == 2 else 1
    y = torch.empty((B, rows), dtype=torch.float32, device=x.device)
    qw3_q4_k_gemv(W.data_ptr(), rows, cols, x.data_ptr(), B, y.data_ptr(), _stream_ptr())
    return y


class _Ordered:
    """Orders the model's stream after torch's current stream on entry and
    torch's current stream after the model's stream on exit, so tensors that
    torch wrote are ready and temporaries freed by torch are not reused while
    the library still reads them."""

    def __init__(self, model: "Qw3Model"):
        self.m = model

    def __enter__(self):
        torch = _torch()
        self.cur = torch.cuda.current_stream()
        self.m.stream.wait_stream(self.cur)
        return self

    def __exit__(self, *exc):
        self.cur.wait_stream(self.m.stream)
        return False


class Qw3Model:
    """A libqw3 model on its own torch-owned CUDA stream.

    Build it from f32 weights (quantised on the device by the library's Q8_0
    encoder) or from Q8_0 bytes in GGUF layout.
    """

    def __init__(self, shape, tensors_dev: dict, *, max_seqs: int = 1, max_seq_len: int = 1024,
                 max_prefill: int = 512, flags: int = 0):
        torch = _torch()
        self.shape = shape
        self.stream = torch.cuda.Stream()
        self.max_seqs, self.max_seq_len, self.max_prefill = max_seqs, max_seq_len, max_prefill
        cfg = Qw3Config(vocab=shape.vocab, hidden=shape.hidden, n_layers=shape.n_layers, n_heads=shape.n_heads,
                        n_kv_heads=shape.n_kv_heads, head_dim=shape.head_dim, intermediate=shape.intermediate,
                        rms_eps=shape.rms_eps, rope_theta=shape.rope_theta, tied_lm_head=1 if shape.tied else 0,
                        max_seqs=max_seqs, max_seq_len=max_seq_len, max_prefill=max_prefill, flags=flags)
        layers = (Qw3LayerWeights * shape.n_layers)()
        names = ("attn_q", "attn_k", "attn_v", "attn_output", "ffn_gate", "ffn_up", "ffn_down",
                 "attn_norm", "attn_q_norm", "attn_k_norm", "ffn_norm")
        for i in range(shape.n_layers):
            for nm in names:
                setattr(layers[i], nm, tensors_dev[f"blk.{i}.{nm}"].data_ptr())
        w = Qw3Weights(token_embd=tensors_dev["token_embd"].data_ptr(),
                       output=tensors_dev["output"].data_ptr() if not shape.tied else None,
                       output_norm=tensors_dev["output_norm"].data_ptr(), layers=layers, on_device=1)
        # the weights were written on torch's current stream
        self.stream.wait_stream(torch.cuda.current_stream())
        self.h = qw3_create(cfg, w, self.stream.cuda_stream)
        self.flags = flags

    @classmethod
    def from_f32(cls, shape, weights: Iterable, device: str = "cuda", **kw) -> "Qw3Model":
        """weights: iterable of (name, kind, f32 numpy array) in any order;
        linear tensors are quantised on the device with qw3_q8_0_quantize, or
        qw3_q4_k_quantize when flags hold QW3_FLAG_WEIGHTS_Q4_K."""
        torch = _torch()
        tensors = {}
        status = torch.zeros(1, dtype=torch.int32, device=device)
        enc = q4_k_quantize if kw.get("flags", 0) & QW3_FLAG_WEIGHTS_Q4_K else q8_0_quantize
        for name, kind, arr in weights:
            t = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).to(device)
            tensors[name] = enc(t.reshape(-1), status) if kind == "linear" else t
            del t
        if int(status.item()) != 0:
            raise Qw3Error(int(status.item()), "non-finite weight values")
        m = cls(shape, tensors, **kw)
        del tensors
        return m

    @classmethod
    def from_q8_0(cls, shape, tensors_host: dict, device: str = "cuda", **kw) -> "Qw3Model":
        """tensors_host: GGUF name -> Q8_0 wire bytes (linear) or f32 (norm)."""
        torch = _torch()
        dev = {k: torch.from_numpy(np.ascontiguousarray(v)).to(device) for k, v in tensors_host.items()}
        return cls(shape, dev, **kw)

    # -- calls ---------------------------------------------------------------

    def prefill(self, seq: int, tokens, want_logits: bool = True):
        """Append tokens (CUDA int32 tensor) to sequence seq; return
        (last-row logits or None, argmax int32 tensor [1])."""
        torch = _torch()
        tokens = tokens.to(torch.int32).contiguous()
        logits = torch.empty(self.shape.vocab, dtype=torch.float32, device=tokens.device) if want_logits else None
        am = torch.empty(1, dtype=torch.int32, device=tokens.device)
        with _Ordered(self):
            qw3_prefill(self.h, seq, tokens.data_ptr(), tokens.numel(),
                        logits.data_ptr() if logits is not None else 0, am.data_ptr())
        return logits, am

    def forward_all_logits(self, seq: int, tokens):
        """Append tokens (CUDA int32 tensor [n]) to sequence seq; return
        (logits [n, vocab], argmax int32 [n]) of every appended row."""
        torch = _torch()
        tokens = tokens.to(torch.int32).contiguous()
        n = tokens.numel()
        logits = torch.empty((n, self.shape.vocab), dtype=torch.float32, device=tokens.device)
        am = torch.empty(n, dtype=torch.int32, device=tokens.device)
        with _Ordered(self):
            qw3_forward_all_logits(self.h, seq, tokens.data_ptr(), n, logits.data_ptr(), am.data_ptr())
        return logits, am

    def decode(self, tokens, pos: Sequence[int], seqs: Optional[Sequence[int]] = None, want_logits: bool = True):
        """One decode step for B = len(pos) sequences; tokens CUDA int32 [B]."""
        torch = _torch()
        B = len(pos)
        tokens = tokens.to(torch.int32).contiguous()
        logits = torch.empty((B, self.shape.vocab), dtype=torch.float32,
                             device=tokens.device) if want_logits else None
        am = torch.empty(B, dtype=torch.int32, device=tokens.device)
        with _Ordered(self):
            qw3_decode(self.h, B, seqs, tokens.data_ptr(), pos, logits.data_ptr() if logits is not None else 0,
                       am.data_ptr())
        return logits, am

    def generate_greedy(self, first_tokens, n_steps: int, seqs: Optional[Sequence[int]] = None, out=None):
        torch = _torch()
        first_tokens = first_tokens.to(torch.int32).contiguous()
        B = first_tokens.numel()
        if out is None:
            out = torch.empty((n_steps, B), dtype=torch.int32, device=first_tokens.device)
        with _Ordered(self):
            qw3_generate_greedy(self.h, B, seqs, n_steps, first_tokens.data_ptr(), out.data_ptr())
        return out

    def reset(self, seq: int) -> None:
        qw3_reset(self.h, seq)

    def truncate(self, seq: int, keep_len: int) -> None:
        qw3_truncate(self.h, seq, keep_len)

    def seq_len(self, seq: int) -> int:
        return qw3_seq_len(self.h, seq)

    def read_kv(self, layer: int, seq: int, pos0: int, n: int):
        torch = _torch()
        s = self.shape
        k = torch.empty((n, s.n_kv_heads, s.head_dim), dtype=torch.float32, device="cuda")
        v = torch.empty_like(k)
        with _Ordered(self):
            qw3_debug_read_kv(self.h, layer, seq, pos0, n, k.data_ptr(), v.data_ptr())
        return k, v

    def read_trace(self, max_records: int = 4096) -> np.ndarray:
        return qw3_debug_read_trace(self.h, max_records)

    def decode_plan(self, B: int = 1) -> tuple[bool, int]:
        return qw3_decode_plan(self.h, B)

    def sync(self) -> None:
        qw3_sync(self.h)

    def close(self) -> None:
        if getattr(self, "h", None):
            qw3_destroy(self.h)
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
        return False

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
