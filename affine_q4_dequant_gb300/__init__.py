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
    "Q4AError", "lib_path", "pack", "xsum", "gemv", "gemv_silu", "gemv_experts", "gemv_experts_lowbit",
    "gemv_experts_gate_up_silu",
    "gemv_rmsnorm",
    "gemv_rmsnorm_grouped", "gemv_inject_rmsnorm_grouped", "gemv_gate_up_silu", "gemv_rmsnorm_gate_up_silu", "decode_mlp", "lowbit_pack",
    "gemv_lowbit", "quantize", "gemv_f32x", "silu_mul_xsum", "moe_combine", "check_device_error", "debug_withhold_stage",
    "gemv_kernel_choice",
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
        "q4a_decode_mlp": (I32, [P, P, P, P, P, P, P, F, F, P, P, P, I32, I64, I64, P]),
        "q4a_gemv_lowbit": (I32, [P, I32, P, P, P, P, P, I32, I64, I64, P]),
        "q4a_gemv_experts": (I32, [P, P, P, P, P, P, P, P, I32, I32, I64, I64, I64, P]),
        "q4a_gemv_experts_gate_up_silu": (I32, [P, P, P, P, P, P, P, P, I32, I32, I64, I64, I64, P]),
        "q4a_gemv_experts_lowbit": (I32, [P, I32, P, P, P, P, P, I32, P, P, P, I32, I32, I64, I64, I64, P]),
        "q4a_gemv_rmsnorm": (I32, [P, P, P, P, P, P, F, F, I32, I64, I64, P]),
        "q4a_gemv_rmsnorm_grouped": (I32, [P, P, P, P, P, P, F, F, I32, I32, I64, I64, P]),
        "q4a_gemv_inject_rmsnorm_grouped": (I32, [P, P, P, P, P, P, P, P, P, F, F, I32, I32, I64, I64, P]),
        "q4a_silu_mul_xsum": (I32, [P, P, P, I64, I64, P]),
        "q4a_moe_combine": (I32, [P, P, P, P, I32, I32, I64, I64, P, P, P, P]),
        "q4a_check_device_error": (I32, [P]),
        "q4a_debug_withhold_stage": (I32, [I32]),
        "q4a_gemv_kernel_choice": (I32, [P, P, I32, I64, I64]),
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


_U8 = (torch.uint8,)
_F16 = (torch.float16, torch.int16, torch.uint16)
_BF16 = (torch.bfloat16, torch.int16, torch.uint16)
_F32 = (torch.float32,)
_I32 = (torch.int32,)
_ANY = None   # any dtype (prefetch hints)
_NULL = ctypes.c_void_p(0)


def _ptrs(*specs):
    """Device pointers for specs (tensor, name, dtypes, shape); a spec may be None (a NULL
    pointer). Every shape is checked first, then dtypes, CUDA residency, contiguity and the
    device: a mis-shaped buffer would be read or written past its end by the kernels, so it is
    refused here, before anything launches. (Plain comparisons and C-level tensor queries: this
    runs on every call.)"""
    for sp in specs:
        if sp is None:
            continue
        t, name, _, shape = sp
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a CUDA tensor")
        if shape is not None and t.shape != shape:
            raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(int(v) for v in shape)}")
    dev = None
    out = []
    for sp in specs:
        if sp is None:
            out.append(_NULL)
            continue
        t, name, dtypes, _ = sp
        if dtypes is not None and t.dtype not in dtypes:
            raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
        d = t.get_device()
        if d < 0:
            raise TypeError(f"{name} must be a CUDA tensor")
        if dev is None:
            dev = torch.cuda.current_device()
        if d != dev:
            raise ValueError(f"{name} is on {t.device}, but the current device is cuda:{dev}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        out.append(t.data_ptr())
    return out

def _dims(t: torch.Tensor, name: str, ndim: int = 2):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.dim() != ndim:
        raise ValueError(f"{name}: {t.dim()} dimensions, expected {ndim}")
    return tuple(int(v) for v in t.shape)


def _mat(w, s, b, out_dim: int, in_dim: int, wname="w", sname="s", bname="b", code_cols=None):
    """Specs of a packed matrix: codes [out_dim][code_cols] (in_dim/2 by default), scales and
    biases [out_dim][in_dim/64]."""
    if in_dim % 64 != 0:
        raise ValueError(f"in_dim {in_dim} is not a multiple of 64")
    code_cols = in_dim // 2 if code_cols is None else code_cols
    return [(w, wname, _U8, (out_dim, code_cols)), (s, sname, _BF16, (out_dim, in_dim // 64)),
            (b, bname, _BF16, (out_dim, in_dim // 64))]


def _empty(shape, dtype, like):
    return torch.empty(shape, dtype=dtype, device=like.device)


def pack(codes: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    rows, in_dim = _dims(codes, "codes")
    out = _empty((rows, in_dim // 2), torch.uint8, codes) if out is None else out
    po, pc = _ptrs((out, "out", _U8, (rows, in_dim // 2)), (codes, "codes", _U8, None))
    _check("q4a_pack", _lib.q4a_pack(po, pc, rows, in_dim, _stream(stream)))
    return out


def xsum(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    nb, in_dim = _dims(x, "x")
    out = _empty((nb, in_dim // 64), torch.float32, x) if out is None else out
    po, px = _ptrs((out, "out", _F32, (nb, in_dim // 64)), (x, "x", _F16, None))
    _check("q4a_xsum", _lib.q4a_xsum(po, px, nb, in_dim, _stream(stream)))
    return out


def gemv(w, s, b, x, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = W x (fp32 [nb][out_dim]) from fp16 activations x [nb][in_dim]."""
    out_dim = _dims(w, "w")[0]
    nb, in_dim = _dims(x, "x")
    out = _empty((nb, out_dim), torch.float32, x) if out is None else out
    py, pw, ps, pb, px = _ptrs((out, "y", _F32, (nb, out_dim)), *_mat(w, s, b, out_dim, in_dim), (x, "x", _F16, None))
    _check("q4a_gemv", _lib.q4a_gemv(py, pw, ps, pb, px, nb, out_dim, in_dim, _stream(stream)))
    return out


def gemv_silu(w: torch.Tensor, s: torch.Tensor, b: torch.Tensor, x: torch.Tensor, div: float,
              out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = silu((W.x) / div) elementwise; otherwise as gemv()."""
    nb, in_dim = _dims(x, "x")
    out_dim = _dims(w, "w")[0]
    out = _empty((nb, out_dim), torch.float32, x) if out is None else out
    py, pw, ps, pb, px = _ptrs((out, "y", _F32, (nb, out_dim)), *_mat(w, s, b, out_dim, in_dim), (x, "x", _F16, None))
    _check("q4a_gemv_silu", _lib.q4a_gemv_silu(py, pw, ps, pb, px, float(div), nb, out_dim, in_dim, _stream(stream)))
    return out


def gemv_gate_up_silu(w, s, b, x, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """h = fp16(silu(W_gate x) * (W_up x)); w holds the gate rows, then the up rows."""
    nb, in_dim = _dims(x, "x")
    inter = _dims(w, "w")[0] // 2
    out = _empty((nb, inter), torch.float16, x) if out is None else out
    ph, pw, ps, pb, px = _ptrs((out, "h", _F16, (nb, inter)), *_mat(w, s, b, 2 * inter, in_dim), (x, "x", _F16, None))
    _check("q4a_gemv_gate_up_silu", _lib.q4a_gemv_gate_up_silu(ph, pw, ps, pb, px, nb, inter, in_dim,
                                                               _stream(stream)))
    return out


def gemv_rmsnorm_gate_up_silu(w, s, b, x_raw, norm_w, eps: float = 1e-6, shift: float = 0.0,
                              out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """gemv_gate_up_silu on RMS-normalised fp32 activations (one normalisation group)."""
    nb, in_dim = _dims(x_raw, "x_raw")
    inter = _dims(w, "w")[0] // 2
    out = _empty((nb, inter), torch.float16, x_raw) if out is None else out
    ph, pw, ps, pb, px, pn = _ptrs((out, "h", _F16, (nb, inter)), *_mat(w, s, b, 2 * inter, in_dim),
                                   (x_raw, "x_raw", _F32, None), (norm_w, "norm_w", _BF16, (in_dim,)))
    _check("q4a_gemv_rmsnorm_gate_up_silu", _lib.q4a_gemv_rmsnorm_gate_up_silu(
        ph, pw, ps, pb, px, pn, float(eps), float(shift), nb, inter, in_dim, _stream(stream)))
    return out


def decode_mlp(w_gu, s_gu, b_gu, x_raw, norm_w, w_dn, s_dn, b_dn, eps: float = 1e-6, shift: float = 0.0,
               out: torch.Tensor | None = None, h: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One decode layer's MLP: h = fp16(silu(W_gate xn) * (W_up xn)) with xn the RMS-normalised
    x_raw, then y = W_down h (fp32 [nb][hidden]). w_gu holds the gate rows, then the up rows."""
    nb, hidden = _dims(x_raw, "x_raw")
    inter = _dims(w_gu, "w_gu")[0] // 2
    out = _empty((nb, hidden), torch.float32, x_raw) if out is None else out
    h = _empty((nb, inter), torch.float16, x_raw) if h is None else h
    py, ph, pgw, pgs, pgb, px, pn, pdw, pds, pdb = _ptrs(
        (out, "y", _F32, (nb, hidden)), (h, "h", _F16, (nb, inter)),
        *_mat(w_gu, s_gu, b_gu, 2 * inter, hidden, "w_gu", "s_gu", "b_gu"),
        (x_raw, "x_raw", _F32, None), (norm_w, "norm_w", _BF16, (hidden,)),
        *_mat(w_dn, s_dn, b_dn, hidden, inter, "w_dn", "s_dn", "b_dn"))
    _check("q4a_decode_mlp", _lib.q4a_decode_mlp(py, ph, pgw, pgs, pgb, px, pn, float(eps), float(shift), pdw, pds,
                                                 pdb, nb, hidden, inter, _stream(stream)))
    return out


def gemv_rmsnorm(w, s, b, x_raw, norm_w, eps: float = 1e-6, shift: float = 0.0,
                 out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    out_dim = _dims(w, "w")[0]
    nb, in_dim = _dims(x_raw, "x_raw")
    out = _empty((nb, out_dim), torch.float32, x_raw) if out is None else out
    py, pw, ps, pb, px, pn = _ptrs((out, "y", _F32, (nb, out_dim)), *_mat(w, s, b, out_dim, in_dim),
                                   (x_raw, "x_raw", _F32, None), (norm_w, "norm_w", _BF16, (in_dim,)))
    _check("q4a_gemv_rmsnorm", _lib.q4a_gemv_rmsnorm(py, pw, ps, pb, px, pn, float(eps), float(shift), nb, out_dim,
                                                     in_dim, _stream(stream)))
    return out


def gemv_rmsnorm_grouped(w, s, b, x_raw, norm_w, norm_groups: int, eps: float = 1e-6, shift: float = 0.0,
                         out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """gemv_rmsnorm with norm_groups equal segments per row, each normalised on its own."""
    nb, in_dim = _dims(x_raw, "x_raw")
    out_dim = _dims(w, "w")[0]
    out = _empty((nb, out_dim), torch.float32, x_raw) if out is None else out
    py, pw, ps, pb, px, pn = _ptrs((out, "y", _F32, (nb, out_dim)), *_mat(w, s, b, out_dim, in_dim),
                                   (x_raw, "x_raw", _F32, None), (norm_w, "norm_w", _BF16, (in_dim,)))
    _check("q4a_gemv_rmsnorm_grouped", _lib.q4a_gemv_rmsnorm_grouped(
        py, pw, ps, pb, px, pn, float(eps), float(shift), int(norm_groups), nb, out_dim, in_dim, _stream(stream)))
    return out


def gemv_inject_rmsnorm_grouped(w, s, b, x_raw, out, logit, norm_w, norm_groups: int, eps: float = 1e-6,
                                shift: float = 0.0, y: torch.Tensor | None = None, x_new: torch.Tensor | None = None,
                                want_x_new: bool = True, stream=None):
    """Inject out [nb][n] into each of the norm_groups streams of x_raw [nb][n * norm_groups]
    with weight 2 sigmoid(logit[r][g] / norm_groups), then the grouped RMSNorm and y = W.xn.
    Returns (y, x_new): x_new is the injected stream (None when want_x_new is False)."""
    nb, in_dim = _dims(x_raw, "x_raw")
    out_dim = _dims(w, "w")[0]
    if norm_groups < 1 or in_dim % norm_groups != 0:
        raise ValueError(f"in_dim {in_dim} does not split into {norm_groups} streams")
    y = _empty((nb, out_dim), torch.float32, x_raw) if y is None else y
    if x_new is None and want_x_new:
        x_new = _empty((nb, in_dim), torch.float32, x_raw)
    py, pxn, pw, ps, pb, px, po, pl, pn = _ptrs(
        (y, "y", _F32, (nb, out_dim)), None if x_new is None else (x_new, "x_new", _F32, (nb, in_dim)),
        *_mat(w, s, b, out_dim, in_dim), (x_raw, "x_raw", _F32, None), (out, "out", _F32, (nb, in_dim // norm_groups)),
        (logit, "logit", _F32, (nb, norm_groups)), (norm_w, "norm_w", _BF16, (in_dim,)))
    _check("q4a_gemv_inject_rmsnorm_grouped", _lib.q4a_gemv_inject_rmsnorm_grouped(
        py, pxn, pw, ps, pb, px, po, pl, pn, float(eps), float(shift), int(norm_groups), nb, out_dim, in_dim,
        _stream(stream)))
    return y, x_new


def quantize(w: torch.Tensor, stream=None):
    """4-bit min/max quantisation of fp32 weights [rows][in]: (packed codes, s bf16, b bf16)."""
    rows, in_dim = _dims(w, "w")
    packed = _empty((rows, in_dim // 2), torch.uint8, w)
    s = _empty((rows, in_dim // 64), torch.bfloat16, w)
    b = _empty((rows, in_dim // 64), torch.bfloat16, w)
    pp, ps, pb, pw = _ptrs((packed, "w_packed", _U8, None), (s, "s", _BF16, None), (b, "b", _BF16, None),
                           (w, "w", _F32, None))
    _check("q4a_quantize", _lib.q4a_quantize(pp, ps, pb, pw, rows, in_dim, _stream(stream)))
    return packed, s, b


def gemv_f32x(w, s, b, x, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = W x from fp32 activations (narrow projections of prefill)."""
    nb, in_dim = _dims(x, "x")
    out_dim = _dims(w, "w")[0]
    out = _empty((nb, out_dim), torch.float32, x) if out is None else out
    py, pw, ps, pb, px = _ptrs((out, "y", _F32, (nb, out_dim)), *_mat(w, s, b, out_dim, in_dim), (x, "x", _F32, None))
    _check("q4a_gemv_f32x", _lib.q4a_gemv_f32x(py, pw, ps, pb, px, nb, out_dim, in_dim, _stream(stream)))
    return out


def lowbit_pack(w_packed: torch.Tensor, with_lowest: bool = True, stream=None):
    """Derived low-bit codes of a packed 4-bit matrix: (w_up [rows][in/4], w_lo [rows][in/8]
    or None). w_up alone is the 2-bit matrix; w_up with w_lo the 3-bit one."""
    rows, half = _dims(w_packed, "w_packed")
    in_dim = 2 * half
    w_up = _empty((rows, in_dim // 4), torch.uint8, w_packed)
    w_lo = _empty((rows, in_dim // 8), torch.uint8, w_packed) if with_lowest else None
    pu, pl, pp = _ptrs((w_up, "w_up", _U8, None), None if w_lo is None else (w_lo, "w_lo", _U8, None),
                       (w_packed, "w_packed", _U8, None))
    _check("q4a_lowbit_pack", _lib.q4a_lowbit_pack(pu, pl, pp, rows, in_dim, _stream(stream)))
    return w_up, w_lo


def gemv_lowbit(bits: int, w_up, w_lo, s, b, x, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = W.x with W from derived 2-bit (bits=2, w_lo unused) or 3-bit codes."""
    out_dim = _dims(w_up, "w_up")[0]
    nb, in_dim = _dims(x, "x")
    out = _empty((nb, out_dim), torch.float32, x) if out is None else out
    lo = None if (w_lo is None or bits == 2) else (w_lo, "w_lo", _U8, (out_dim, in_dim // 8))
    py, pw, ps, pb, pl, px = _ptrs((out, "y", _F32, (nb, out_dim)),
                                   *_mat(w_up, s, b, out_dim, in_dim, "w_up", code_cols=in_dim // 4), lo,
                                   (x, "x", _F16, None))
    _check("q4a_gemv_lowbit", _lib.q4a_gemv_lowbit(py, int(bits), pw, pl, ps, pb, px, nb, out_dim, in_dim,
                                                   _stream(stream)))
    return out


def gemv_experts(w_bank, s_bank, b_bank, x, x_rows, expert_ids, token_offsets, n_experts: int,
                 out_dim: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """expert_ids / token_offsets are HOST int32 arrays (numpy or lists); x_rows is a
    CUDA int32 tensor or None."""
    expert_ids = np.ascontiguousarray(expert_ids, dtype=np.int32)
    token_offsets = np.ascontiguousarray(token_offsets, dtype=np.int32)
    if token_offsets.ndim != 1 or expert_ids.ndim != 1 or token_offsets.shape[0] != expert_ids.shape[0] + 1:
        raise ValueError("token_offsets must have one entry more than expert_ids")
    n_rows = int(token_offsets[-1])
    x_n, in_dim = _dims(x, "x")
    out = _empty((max(n_rows, 0), out_dim), torch.float32, x) if out is None else out
    if x_rows is None and x_n < n_rows:
        raise ValueError(f"x has {x_n} rows; without x_rows it needs token_offsets[-1] = {n_rows}")
    xr = None if x_rows is None else (x_rows, "x_rows", _I32, (n_rows,))
    py, pw, ps, pb, px, pr = _ptrs(
        (out, "y", _F32, (n_rows, out_dim)),
        *_mat(w_bank, s_bank, b_bank, int(n_experts) * int(out_dim), in_dim, "w_bank", "s_bank", "b_bank"),
        (x, "x", _F16, None), xr)
    _check("q4a_gemv_experts", _lib.q4a_gemv_experts(
        py, pw, ps, pb, px, pr, ctypes.c_void_p(expert_ids.ctypes.data), ctypes.c_void_p(token_offsets.ctypes.data),
        int(expert_ids.shape[0]), int(n_experts), n_rows, int(out_dim), int(in_dim), _stream(stream)))
    return out


def gemv_experts_gate_up_silu(w_bank, s_bank, b_bank, x, x_rows, expert_ids, token_offsets, n_experts: int,
                              inter: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """h = fp16(silu(gate) * up) [n_rows][inter] over a bank of fused gate|up experts (expert e:
    gate rows e*2*inter .., then its up rows). expert_ids / token_offsets are HOST int32 arrays;
    x_rows is a CUDA int32 tensor or None."""
    expert_ids = np.ascontiguousarray(expert_ids, dtype=np.int32)
    token_offsets = np.ascontiguousarray(token_offsets, dtype=np.int32)
    if token_offsets.ndim != 1 or expert_ids.ndim != 1 or token_offsets.shape[0] != expert_ids.shape[0] + 1:
        raise ValueError("token_offsets must have one entry more than expert_ids")
    n_rows = int(token_offsets[-1])
    x_n, in_dim = _dims(x, "x")
    out = _empty((max(n_rows, 0), inter), torch.float16, x) if out is None else out
    if x_rows is None and x_n < n_rows:
        raise ValueError(f"x has {x_n} rows; without x_rows it needs token_offsets[-1] = {n_rows}")
    xr = None if x_rows is None else (x_rows, "x_rows", _I32, (n_rows,))
    ph, pw, ps, pb, px, pr = _ptrs(
        (out, "h", _F16, (n_rows, inter)),
        *_mat(w_bank, s_bank, b_bank, int(n_experts) * 2 * int(inter), in_dim, "w_bank", "s_bank", "b_bank"),
        (x, "x", _F16, None), xr)
    _check("q4a_gemv_experts_gate_up_silu", _lib.q4a_gemv_experts_gate_up_silu(
        ph, pw, ps, pb, px, pr, ctypes.c_void_p(expert_ids.ctypes.data), ctypes.c_void_p(token_offsets.ctypes.data),
        int(expert_ids.shape[0]), int(n_experts), n_rows, int(inter), int(in_dim), _stream(stream)))
    return out


def gemv_experts_lowbit(bits: int, w_up_bank, w_lo_bank, s_bank, b_bank, x, x_rows, expert_ids, token_offsets,
                        n_experts: int, out_dim: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Routed experts with derived 2-bit (w_lo_bank unused) or 3-bit codes; x is a float16 or
    float32 CUDA tensor (fp32 rows are rounded to binary16 when staged). expert_ids and
    token_offsets are HOST int32 arrays; x_rows a CUDA int32 tensor or None."""
    expert_ids = np.ascontiguousarray(expert_ids, dtype=np.int32)
    token_offsets = np.ascontiguousarray(token_offsets, dtype=np.int32)
    if token_offsets.ndim != 1 or expert_ids.ndim != 1 or token_offsets.shape[0] != expert_ids.shape[0] + 1:
        raise ValueError("token_offsets must have one entry more than expert_ids")
    n_rows = int(token_offsets[-1])
    x_n, in_dim = _dims(x, "x")
    rows = int(n_experts) * int(out_dim)
    out = _empty((max(n_rows, 0), out_dim), torch.float32, x) if out is None else out
    if x_rows is None and x_n < n_rows:
        raise ValueError(f"x has {x_n} rows; without x_rows it needs token_offsets[-1] = {n_rows}")
    f32 = isinstance(x, torch.Tensor) and x.dtype == torch.float32
    lo = None if (w_lo_bank is None or bits == 2) else (w_lo_bank, "w_lo_bank", _U8, (rows, in_dim // 8))
    xr = None if x_rows is None else (x_rows, "x_rows", _I32, (n_rows,))
    py, pw, ps, pb, pl, px, pr = _ptrs(
        (out, "y", _F32, (n_rows, out_dim)),
        *_mat(w_up_bank, s_bank, b_bank, rows, in_dim, "w_up_bank", "s_bank", "b_bank", code_cols=in_dim // 4), lo,
        (x, "x", _F32 if f32 else _F16, None), xr)
    _check("q4a_gemv_experts_lowbit", _lib.q4a_gemv_experts_lowbit(
        py, int(bits), pw, pl, ps, pb, px, 1 if f32 else 0, pr, ctypes.c_void_p(expert_ids.ctypes.data),
        ctypes.c_void_p(token_offsets.ctypes.data), int(expert_ids.shape[0]), int(n_experts), n_rows, int(out_dim),
        int(in_dim), _stream(stream)))
    return out


def silu_mul_xsum(gate_up: torch.Tensor, h: torch.Tensor | None = None,
                  hsum: torch.Tensor | None = None, stream=None, want_hsum: bool = True):
    rows, two_inter = _dims(gate_up, "gate_up")
    inter = two_inter // 2
    h = _empty((rows, inter), torch.float16, gate_up) if h is None else h
    if hsum is None and want_hsum:
        hsum = _empty((rows, inter // 64), torch.float32, gate_up)
    ph, phs, pg = _ptrs((h, "h", _F16, (rows, inter)),
                        None if hsum is None else (hsum, "hsum", _F32, (rows, inter // 64)),
                        (gate_up, "gate_up", _F32, None))
    _check("q4a_silu_mul_xsum", _lib.q4a_silu_mul_xsum(ph, phs, pg, rows, inter, _stream(stream)))
    return h, hsum


def moe_combine(y: torch.Tensor, slot: torch.Tensor, w: torch.Tensor, y_shared: torch.Tensor | None = None,
                gate: torch.Tensor | None = None, x: torch.Tensor | None = None,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[t] = sum_k w[t][k] * y[slot[t][k]] (+ sigmoid(gate . x[t]) * y_shared[t]).
    y fp32 [n_slots][hidden]; slot int32 [n_tok][k]; w fp32 [n_tok][k]; y_shared fp32
    [n_tok][hidden] or None; gate bf16 [hidden]; x fp32 [n_tok][hidden]."""
    n_slots, hidden = _dims(y, "y")
    n_tok, top_k = _dims(slot, "slot")
    out = _empty((n_tok, hidden), torch.float32, y) if out is None else out
    shared = y_shared is not None
    po, py, ps, pw, pys, pg, px = _ptrs(
        (out, "out", _F32, (n_tok, hidden)), (y, "y", _F32, None), (slot, "slot", _I32, None),
        (w, "w", _F32, (n_tok, top_k)), (y_shared, "y_shared", _F32, (n_tok, hidden)) if shared else None,
        (gate, "gate", _BF16, (hidden,)) if shared else None, (x, "x", _F32, (n_tok, hidden)) if shared else None)
    _check("q4a_moe_combine", _lib.q4a_moe_combine(po, py, ps, pw, int(n_tok), int(top_k), int(n_slots), int(hidden),
                                                   pys, pg, px, _stream(stream)))
    return out


def check_device_error(stream=None) -> None:
    _check("q4a_check_device_error", _lib.q4a_check_device_error(_stream(stream)))


def gemv_kernel_choice(s, b, nb: int, out_dim: int, in_dim: int) -> str:
    """The kernel gemv() launches for these arguments, without launching: "tcgen05" or "gemv".
    s and b are the scale and bias tensors (only their addresses matter) or raw addresses."""
    ps, pb = (ctypes.c_void_p(t.data_ptr() if isinstance(t, torch.Tensor) else int(t)) for t in (s, b))
    return "tcgen05" if _lib.q4a_gemv_kernel_choice(ps, pb, int(nb), int(out_dim), int(in_dim)) == 1 else "gemv"


def debug_withhold_stage(stage: int) -> None:
    """Failure-path testing: the next GEMV-kernel launch from this thread never loads weight
    stage `stage` of each CTA, so its bounded wait gives up (check_device_error then raises
    ERR_TIMEOUT). -1 clears the request."""
    _check("q4a_debug_withhold_stage", _lib.q4a_debug_withhold_stage(int(stage)))
