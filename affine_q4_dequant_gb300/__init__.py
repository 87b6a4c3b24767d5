"""affine_q4_dequant_gb300 -- Python binding of libq4a.so, the GB300 (sm_103a)
row-batched affine-4-bit dequantising GEMV.

This module only marshals arguments: it hands device pointers, sizes and the
current CUDA stream to the C ABI declared in include/q4a.h. Every step of the
computation runs in the library's CUDA kernels. There is no CPU fallback: if
the library is missing or fails to load, importing this module raises.

PyTorch supplies device memory and streams. Storage conventions:
  codes     torch.uint8  [rows][in_dim]     one 4-bit code per byte
  w         torch.uint8  [rows][in_dim/2]   packed rows (see pack())
  s, b      torch.bfloat16 (or int16/uint16 bit views) [rows][in_dim/64]
  x         torch.float16 (or int16/uint16 bit views) [nb][in_dim]
  y         torch.float32 [nb][out_dim]
"""

from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import _build

__all__ = [
    "Q4AError", "lib_path", "pack", "xsum", "gemv", "gemv_silu", "gemv_experts", "gemv_rmsnorm",
    "gemv_rmsnorm_grouped", "gemv_gate_up_silu", "gemv_rmsnorm_gate_up_silu", "lowbit_pack",
    "gemv_lowbit", "quantize", "gemv_f32x", "silu_mul_xsum", "moe_combine", "check_device_error",
    "STATUS", "MAX_SEGMENTS",
]

MAX_SEGMENTS = 512
STATUS = {0: "OK", 1: "ERR_NULL", 2: "ERR_SHAPE", 3: "ERR_ALIGN", 4: "ERR_UNSUPPORTED",
          5: "ERR_CUDA", 6: "ERR_TIMEOUT"}


class Q4AError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str):
        self.status = status
        self.status_name = STATUS.get(status, str(status))
        super().__init__(f"{fn}: {self.status_name} ({detail})")


def lib_path() -> str:
    return _build.LIB


def _load() -> ctypes.CDLL:
    if not os.path.exists(_build.LIB):
        raise ImportError(
            f"libq4a.so not found at {_build.LIB}; build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(_build.LIB)
    P, I64, I32, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    sigs = {
        "q4a_status_string": (ctypes.c_char_p, [I32]),
        "q4a_last_cuda_error": (I32, []),
        "q4a_pack": (I32, [P, P, I64, I64, P]),
        "q4a_xsum": (I32, [P, P, I32, I64, P]),
        "q4a_gemv": (I32, [P, P, P, P, P, I32, I64, I64, P]),
        "q4a_gemv_silu": (I32, [P, P, P, P, P, F, I32, I64, I64, P]),
        "q4a_lowbit_pack": (I32, [P, P, P, I64, I64, P]),
        "q4a_quantize": (I32, [P, P, P, P, I64, I64, P]),
        "q4a_gemv_f32x": (I32, [P, P, P, P, P, I32, I64, I64, P]),
        "q4a_gemv_gate_up_silu": (I32, [P, P, P, P, P, I32, I64, I64, P]),
        "q4a_gemv_rmsnorm_gate_up_silu": (I32, [P, P, P, P, P, P, F, F, I32, I64, I64, P]),
        "q4a_gemv_lowbit": (I32, [P, I32, P, P, P, P, P, I32, I64, I64, P]),
        "q4a_gemv_experts": (I32, [P, P, P, P, P, P, P, P, I32, I32, I64, I64, I64, P]),
        "q4a_gemv_rmsnorm": (I32, [P, P, P, P, P, P, F, F, I32, I64, I64, P]),
        "q4a_gemv_rmsnorm_grouped": (I32, [P, P, P, P, P, P, F, F, I32, I32, I64, I64, P]),
        "q4a_silu_mul_xsum": (I32, [P, P, P, I64, I64, P]),
        "q4a_moe_combine": (I32, [P, P, P, P, I32, I32, I64, I64, P, P, P, P]),
        "q4a_check_device_error": (I32, [P]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def _check(fn: str, status: int) -> None:
    if status != 0:
        detail = _lib.q4a_status_string(status).decode()
        if status == 5:
            detail += f"; cudaError {_lib.q4a_last_cuda_error()}"
        raise Q4AError(fn, status, detail)


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream=None) -> int:
    """The cudaStream_t to launch on: the given torch stream, else the current stream of the
    current device (a plain integer handle; the call happens per launch, so it stays cheap)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _dev(t: torch.Tensor, name: str, dtypes) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


_U8 = (torch.uint8,)
_F16 = (torch.float16, torch.int16, torch.uint16)
_BF16 = (torch.bfloat16, torch.int16, torch.uint16)
_F32 = (torch.float32,)
_I32 = (torch.int32,)


def pack(codes: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    rows, in_dim = codes.shape
    if out is None:
        out = torch.empty((rows, in_dim // 2), dtype=torch.uint8, device=codes.device)
    _check("q4a_pack", _lib.q4a_pack(_dev(out, "out", _U8), _dev(codes, "codes", _U8), rows, in_dim,
                                     _stream(stream)))
    return out


def gemv_gate_up_silu(w, s, b, x, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """h = fp16(silu(W_gate x) * (W_up x)); w holds the gate rows, then the up rows."""
    nb, in_dim = x.shape
    inter = w.shape[0] // 2
    if out is None:
        out = torch.empty((nb, inter), dtype=torch.float16, device=x.device)
    _check("q4a_gemv_gate_up_silu", _lib.q4a_gemv_gate_up_silu(
        _dev(out, "h", _F16), _dev(w, "w", _U8), _dev(s, "s", _BF16), _dev(b, "b", _BF16),
        _dev(x, "x", _F16), nb, inter, in_dim, _stream(stream)))
    return out


def gemv_rmsnorm_gate_up_silu(w, s, b, x_raw, norm_w, eps: float = 1e-6, shift: float = 0.0,
                              out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """gemv_gate_up_silu on RMS-normalised fp32 activations (one normalisation group)."""
    nb, in_dim = x_raw.shape
    inter = w.shape[0] // 2
    if out is None:
        out = torch.empty((nb, inter), dtype=torch.float16, device=x_raw.device)
    _check("q4a_gemv_rmsnorm_gate_up_silu", _lib.q4a_gemv_rmsnorm_gate_up_silu(
        _dev(out, "h", _F16), _dev(w, "w", _U8), _dev(s, "s", _BF16), _dev(b, "b", _BF16),
        _dev(x_raw, "x_raw", _F32), _dev(norm_w, "norm_w", _BF16), float(eps), float(shift), nb, inter,
        in_dim, _stream(stream)))
    return out


def quantize(w: torch.Tensor, stream=None):
    """4-bit min/max quantisation of fp32 weights [rows][in]: (packed codes, s bf16, b bf16)."""
    rows, in_dim = w.shape
    packed = torch.empty((rows, in_dim // 2), dtype=torch.uint8, device=w.device)
    s = torch.empty((rows, in_dim // 64), dtype=torch.bfloat16, device=w.device)
    b = torch.empty((rows, in_dim // 64), dtype=torch.bfloat16, device=w.device)
    _check("q4a_quantize", _lib.q4a_quantize(_dev(packed, "w_packed", _U8), _dev(s, "s", _BF16),
                                             _dev(b, "b", _BF16), _dev(w, "w", _F32), rows, in_dim,
                                             _stream(stream)))
    return packed, s, b


def gemv_f32x(w, s, b, x, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = W x from fp32 activations (narrow projections of prefill)."""
    nb, in_dim = x.shape
    out_dim = w.shape[0]
    if out is None:
        out = torch.empty((nb, out_dim), dtype=torch.float32, device=x.device)
    _check("q4a_gemv_f32x", _lib.q4a_gemv_f32x(
        _dev(out, "y", _F32), _dev(w, "w", _U8), _dev(s, "s", _BF16), _dev(b, "b", _BF16),
        _dev(x, "x", _F32), nb, out_dim, in_dim, _stream(stream)))
    return out


def lowbit_pack(w_packed: torch.Tensor, with_lowest: bool = True, stream=None):
    """Derived low-bit codes of a packed 4-bit matrix: (w_up [rows][in/4], w_lo [rows][in/8]
    or None). w_up alone is the 2-bit matrix; w_up with w_lo the 3-bit one."""
    rows, half = w_packed.shape
    in_dim = 2 * half
    w_up = torch.empty((rows, in_dim // 4), dtype=torch.uint8, device=w_packed.device)
    w_lo = torch.empty((rows, in_dim // 8), dtype=torch.uint8, device=w_packed.device) if with_lowest else None
    _check("q4a_lowbit_pack", _lib.q4a_lowbit_pack(
        _dev(w_up, "w_up", _U8), ctypes.c_void_p(0) if w_lo is None else _dev(w_lo, "w_lo", _U8),
        _dev(w_packed, "w_packed", _U8), rows, in_dim, _stream(stream)))
    return w_up, w_lo


def gemv_lowbit(bits: int, w_up, w_lo, s, b, x, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = W.x with W from derived 2-bit (bits=2, w_lo unused) or 3-bit codes."""
    out_dim = w_up.shape[0]
    nb, in_dim = x.shape
    if out is None:
        out = torch.empty((nb, out_dim), dtype=torch.float32, device=x.device)
    lo = ctypes.c_void_p(0) if (w_lo is None or bits == 2) else _dev(w_lo, "w_lo", _U8)
    _check("q4a_gemv_lowbit", _lib.q4a_gemv_lowbit(
        _dev(out, "y", _F32), int(bits), _dev(w_up, "w_up", _U8), lo, _dev(s, "s", _BF16),
        _dev(b, "b", _BF16), _dev(x, "x", _F16), nb, out_dim, in_dim, _stream(stream)))
    return out


def xsum(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    nb, in_dim = x.shape
    if out is None:
        out = torch.empty((nb, in_dim // 64), dtype=torch.float32, device=x.device)
    _check("q4a_xsum", _lib.q4a_xsum(_dev(out, "out", _F32), _dev(x, "x", _F16), nb, in_dim,
                                     _stream(stream)))
    return out


def gemv(w, s, b, x, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    out_dim = w.shape[0]
    nb, in_dim = x.shape
    if out is None:
        out = torch.empty((nb, out_dim), dtype=torch.float32, device=x.device)
    _check("q4a_gemv", _lib.q4a_gemv(_dev(out, "y", _F32), _dev(w, "w", _U8), _dev(s, "s", _BF16),
                                     _dev(b, "b", _BF16), _dev(x, "x", _F16), nb, out_dim, in_dim,
                                     _stream(stream)))
    return out


def gemv_rmsnorm(w, s, b, x_raw, norm_w, eps: float = 1e-6, shift: float = 0.0,
                 out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    out_dim = w.shape[0]
    nb, in_dim = x_raw.shape
    if out is None:
        out = torch.empty((nb, out_dim), dtype=torch.float32, device=x_raw.device)
    _check("q4a_gemv_rmsnorm", _lib.q4a_gemv_rmsnorm(
        _dev(out, "y", _F32), _dev(w, "w", _U8), _dev(s, "s", _BF16), _dev(b, "b", _BF16),
        _dev(x_raw, "x_raw", _F32), _dev(norm_w, "norm_w", _BF16), float(eps), float(shift), nb,
        out_dim, in_dim, _stream(stream)))
    return out


def gemv_silu(w: torch.Tensor, s: torch.Tensor, b: torch.Tensor, x: torch.Tensor, div: float,
              out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = silu((W.x) / div) elementwise; otherwise as gemv()."""
    nb, in_dim = x.shape
    out_dim = w.shape[0]
    if out is None:
        out = torch.empty((nb, out_dim), dtype=torch.float32, device=x.device)
    _check("q4a_gemv_silu", _lib.q4a_gemv_silu(
        _dev(out, "y", _F32), _dev(w, "w", _U8), _dev(s, "s", _BF16), _dev(b, "b", _BF16),
        _dev(x, "x", _F16), float(div), nb, out_dim, in_dim, _stream(stream)))
    return out


def gemv_experts(w_bank, s_bank, b_bank, x, x_rows, expert_ids, token_offsets, n_experts: int,
                 out_dim: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """expert_ids / token_offsets are HOST int32 arrays (numpy or lists); x_rows is a
    CUDA int32 tensor or None."""
    expert_ids = np.ascontiguousarray(expert_ids, dtype=np.int32)
    token_offsets = np.ascontiguousarray(token_offsets, dtype=np.int32)
    n_rows = int(token_offsets[-1])
    in_dim = x.shape[1]
    if out is None:
        out = torch.empty((n_rows, out_dim), dtype=torch.float32, device=x.device)
    xr = ctypes.c_void_p(0) if x_rows is None else _dev(x_rows, "x_rows", _I32)
    _check("q4a_gemv_experts", _lib.q4a_gemv_experts(
        _dev(out, "y", _F32), _dev(w_bank, "w_bank", _U8), _dev(s_bank, "s_bank", _BF16),
        _dev(b_bank, "b_bank", _BF16), _dev(x, "x", _F16), xr,
        ctypes.c_void_p(expert_ids.ctypes.data), ctypes.c_void_p(token_offsets.ctypes.data),
        int(expert_ids.shape[0]), int(n_experts), n_rows, int(out_dim), int(in_dim),
        _stream(stream)))
    return out


def gemv_rmsnorm_grouped(w, s, b, x_raw, norm_w, norm_groups: int, eps: float = 1e-6, shift: float = 0.0,
                         out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """gemv_rmsnorm with norm_groups equal segments per row, each normalised on its own."""
    nb, in_dim = x_raw.shape
    out_dim = w.shape[0]
    if out is None:
        out = torch.empty((nb, out_dim), dtype=torch.float32, device=x_raw.device)
    _check("q4a_gemv_rmsnorm_grouped", _lib.q4a_gemv_rmsnorm_grouped(
        _dev(out, "y", _F32), _dev(w, "w", _U8), _dev(s, "s", _BF16), _dev(b, "b", _BF16),
        _dev(x_raw, "x_raw", _F32), _dev(norm_w, "norm_w", _BF16), float(eps), float(shift),
        int(norm_groups), nb, out_dim, in_dim, _stream(stream)))
    return out


def silu_mul_xsum(gate_up: torch.Tensor, h: torch.Tensor | None = None,
                  hsum: torch.Tensor | None = None, stream=None, want_hsum: bool = True):
    rows, two_inter = gate_up.shape
    inter = two_inter // 2
    if h is None:
        h = torch.empty((rows, inter), dtype=torch.float16, device=gate_up.device)
    if hsum is None and want_hsum:
        hsum = torch.empty((rows, inter // 64), dtype=torch.float32, device=gate_up.device)
    hp = ctypes.c_void_p(0) if hsum is None else _dev(hsum, "hsum", _F32)
    _check("q4a_silu_mul_xsum", _lib.q4a_silu_mul_xsum(
        _dev(h, "h", _F16), hp, _dev(gate_up, "gate_up", _F32), rows, inter, _stream(stream)))
    return h, hsum


def moe_combine(y: torch.Tensor, slot: torch.Tensor, w: torch.Tensor, y_shared: torch.Tensor | None = None,
                gate: torch.Tensor | None = None, x: torch.Tensor | None = None,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[t] = sum_k w[t][k] * y[slot[t][k]] (+ sigmoid(gate . x[t]) * y_shared[t]).
    y fp32 [n_slots][hidden]; slot int32 [n_tok][k]; w fp32 [n_tok][k]; y_shared fp32
    [n_tok][hidden] or None; gate bf16 [hidden]; x fp32 [n_tok][hidden]."""
    n_slots, hidden = y.shape
    n_tok, top_k = slot.shape
    if out is None:
        out = torch.empty((n_tok, hidden), dtype=torch.float32, device=y.device)
    null = ctypes.c_void_p(0)
    _check("q4a_moe_combine", _lib.q4a_moe_combine(
        _dev(out, "out", _F32), _dev(y, "y", _F32), _dev(slot, "slot", _I32), _dev(w, "w", _F32),
        int(n_tok), int(top_k), int(n_slots), int(hidden),
        null if y_shared is None else _dev(y_shared, "y_shared", _F32),
        null if y_shared is None else _dev(gate, "gate", _BF16),
        null if y_shared is None else _dev(x, "x", _F32), _stream(stream)))
    return out


def check_device_error(stream=None) -> None:
    _check("q4a_check_device_error", _lib.q4a_check_device_error(_stream(stream)))
