"""CPU oracle for the affine-4-bit dequantising GEMV -- TEST INFRASTRUCTURE.

Only the test-suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package. The product path (the CUDA library and
its Python binding) never loads it and never falls back to it.

The arithmetic lives in ``q4a_oracle.c`` (plain single-threaded C, IEEE double
precision, no code shared with the CUDA path). This module compiles it with
gcc on first use (or through ``build()``) and wraps it with ctypes for numpy
arrays.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4a_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_q4a.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle_q4a.so`` (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11",
                               "-fno-fast-math", "-ffp-contract=off", "-fvisibility=hidden",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int64
        D = ctypes.c_double
        sig = {
            "q4o_half_value": (D, [ctypes.c_uint16]),
            "q4o_bf16_value": (D, [ctypes.c_uint16]),
            "q4o_half_round": (ctypes.c_uint16, [D]),
            "q4o_pack": (None, [P, P, I, I]),
            "q4o_unpack": (None, [P, P, I, I]),
            "q4o_dequant": (None, [P, P, P, P, I, I]),
            "q4o_xsum": (None, [P, P, I, I]),
            "q4o_gemv": (None, [P, P, P, P, P, P, I, I, I]),
            "q4o_gemv_factored": (None, [P, P, P, P, P, I, I, I]),
            "q4o_gemv_entries": (None, [P, P, P, P, I, P, P, P, P, I]),
            "q4o_gemv_experts": (None, [P, P, P, P, P, P, P, P, P, I, I, I, I]),
            "q4o_rmsnorm_f16": (None, [P, P, P, P, D, D, I, I]),
            "q4o_silu_mul_f16": (None, [P, P, I, I]),
            "q4o_route_topk": (None, [P, P, P, I, I, I]),
            "q4o_moe_combine": (None, [P, P, P, P, P, P, P, P, P, I, I, I, I]),
            "q4o_gemv_silu": (None, [P, P, P, P, P, P, P, D, I, I, I]),
            "q4o_rmsnorm_groups_f16": (None, [P, P, P, P, D, D, I, I, I]),
            "q4o_inject_rmsnorm_groups_f16": (None, [P, P, P, P, P, P, D, D, I, I, I]),
            "q4o_lowbit_pack2": (None, [P, P, I, I]),
            "q4o_lowbit_pack3lo": (None, [P, P, I, I]),
            "q4o_lowbit_codes": (None, [P, P, P, I, I]),
            "q4o_gemv_lowbit": (None, [P, P, P, P, P, P, P, I, I, I]),
            "q4o_experts_lowbit": (None, [P, P, P, P, P, P, P, P, P, P, P, I, I, I, I]),
            "q4o_gemv_f32x": (None, [P, P, P, P, P, P, I, I, I]),
            "q4o_quantize": (None, [P, P, P, P, I, I]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a) -> ctypes.c_void_p:
    return ctypes.c_void_p(0) if a is None else ctypes.c_void_p(a.ctypes.data)


# ---- scalar format helpers ----------------------------------------------------

def half_value(bits: int) -> float:
    return _load().q4o_half_value(int(bits))


def bf16_value(bits: int) -> float:
    return _load().q4o_bf16_value(int(bits))


def half_round(v: float) -> int:
    return int(_load().q4o_half_round(float(v)))


# ---- array functions -------------------------------------------------------------

def pack(codes: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.uint8)
    rows, in_dim = codes.shape
    out = np.empty((rows, in_dim // 2), np.uint8)
    _load().q4o_pack(_p(out), _p(codes), rows, in_dim)
    return out


def unpack(packed: np.ndarray, in_dim: int) -> np.ndarray:
    packed = _c(packed, np.uint8)
    rows = packed.shape[0]
    out = np.empty((rows, in_dim), np.uint8)
    _load().q4o_unpack(_p(out), _p(packed), rows, in_dim)
    return out


def dequant(packed, s, b, in_dim: int) -> np.ndarray:
    packed, s, b = _c(packed, np.uint8), _c(s, np.uint16), _c(b, np.uint16)
    rows = packed.shape[0]
    out = np.empty((rows, in_dim), np.float64)
    _load().q4o_dequant(_p(out), _p(packed), _p(s), _p(b), rows, in_dim)
    return out


def xsum(x_bits: np.ndarray) -> np.ndarray:
    x_bits = _c(x_bits, np.uint16)
    nb, in_dim = x_bits.shape
    out = np.empty((nb, in_dim // 64), np.float64)
    _load().q4o_xsum(_p(out), _p(x_bits), nb, in_dim)
    return out


def gemv(packed, s, b, x_bits, out_dim: int | None = None):
    """Returns (y [nb][out], bound [nb][out]) in float64."""
    packed, s, b, x_bits = (_c(packed, np.uint8), _c(s, np.uint16), _c(b, np.uint16),
                            _c(x_bits, np.uint16))
    nb, in_dim = x_bits.shape
    out_dim = packed.shape[0] if out_dim is None else out_dim
    y = np.empty((nb, out_dim), np.float64)
    bound = np.empty((nb, out_dim), np.float64)
    _load().q4o_gemv(_p(y), _p(bound), _p(packed), _p(s), _p(b), _p(x_bits), nb, out_dim, in_dim)
    return y, bound


def gemv_factored(packed, s, b, x_bits) -> np.ndarray:
    packed, s, b, x_bits = (_c(packed, np.uint8), _c(s, np.uint16), _c(b, np.uint16),
                            _c(x_bits, np.uint16))
    nb, in_dim = x_bits.shape
    out_dim = packed.shape[0]
    y = np.empty((nb, out_dim), np.float64)
    _load().q4o_gemv_factored(_p(y), _p(packed), _p(s), _p(b), _p(x_bits), nb, out_dim, in_dim)
    return y


def gemv_entries(packed, s, b, x_bits, r_idx, o_idx):
    """y[k] = (W x)[r_idx[k]][o_idx[k]] and its bound, one dot product each."""
    packed, s, b, x_bits = (_c(packed, np.uint8), _c(s, np.uint16), _c(b, np.uint16),
                            _c(x_bits, np.uint16))
    r_idx, o_idx = _c(r_idx, np.int64), _c(o_idx, np.int64)
    n = r_idx.shape[0]
    in_dim = x_bits.shape[1]
    y = np.empty(n, np.float64)
    bound = np.empty(n, np.float64)
    _load().q4o_gemv_entries(_p(y), _p(bound), _p(r_idx), _p(o_idx), n, _p(packed), _p(s),
                             _p(b), _p(x_bits), in_dim)
    return y, bound


def gemv_experts(w_bank, s_bank, b_bank, x_bits, x_rows, expert_ids, token_offsets,
                 n_experts: int, out_dim: int):
    w_bank, s_bank, b_bank = _c(w_bank, np.uint8), _c(s_bank, np.uint16), _c(b_bank, np.uint16)
    x_bits = _c(x_bits, np.uint16)
    expert_ids = _c(expert_ids, np.int32)
    token_offsets = _c(token_offsets, np.int32)
    xr = None if x_rows is None else _c(x_rows, np.int32)
    in_dim = x_bits.shape[1]
    n_active = expert_ids.shape[0]
    n_rows = int(token_offsets[-1])
    y = np.empty((n_rows, out_dim), np.float64)
    bound = np.empty((n_rows, out_dim), np.float64)
    _load().q4o_gemv_experts(_p(y), _p(bound), _p(w_bank), _p(s_bank), _p(b_bank), _p(x_bits),
                             _p(xr), _p(expert_ids), _p(token_offsets), n_active, n_experts,
                             out_dim, in_dim)
    return y, bound


def rmsnorm_f16(x_raw, norm_w, eps: float = 1e-6, shift: float = 0.0):
    """Returns (xn fp16 bits [nb][n], inv_rms [nb])."""
    x_raw, norm_w = _c(x_raw, np.float32), _c(norm_w, np.uint16)
    nb, n = x_raw.shape
    xn = np.empty((nb, n), np.uint16)
    inv = np.empty(nb, np.float64)
    _load().q4o_rmsnorm_f16(_p(xn), _p(inv), _p(x_raw), _p(norm_w), float(eps), float(shift), nb, n)
    return xn, inv


def silu_mul_f16(gate_up) -> np.ndarray:
    gate_up = _c(gate_up, np.float32)
    rows, two_inter = gate_up.shape
    inter = two_inter // 2
    h = np.empty((rows, inter), np.uint16)
    _load().q4o_silu_mul_f16(_p(h), _p(gate_up), rows, inter)
    return h


def route_topk(logits, top_k: int):
    """Returns (idx int32 [n_tok][k], weights float64 [n_tok][k])."""
    logits = _c(logits, np.float32)
    n_tok, n_exp = logits.shape
    idx = np.empty((n_tok, top_k), np.int32)
    wts = np.empty((n_tok, top_k), np.float64)
    _load().q4o_route_topk(_p(idx), _p(wts), _p(logits), n_tok, n_exp, top_k)
    return idx, wts


def moe_combine(y, slot, w, y_shared=None, gate=None, x=None):
    """Routing-weighted sum of the expert outputs of each token, plus the gated shared
    expert output. y: float32 [n_slots][hidden]; slot: int32 [n_tok][k]; w: float32
    [n_tok][k]; y_shared: float32 [n_tok][hidden] or None; gate: bf16 bits [hidden];
    x: float32 [n_tok][hidden]. Returns (out float64, abs-sum float64 [n_tok][hidden],
    gate-dot abs-sum float64 [n_tok])."""
    y = _c(y, np.float32)
    slot = _c(slot, np.int32)
    w = _c(w, np.float32)
    n_slots, hidden = y.shape
    n_tok, k = slot.shape
    out = np.empty((n_tok, hidden), np.float64)
    bound = np.empty((n_tok, hidden), np.float64)
    gabs = np.empty((n_tok,), np.float64)
    if y_shared is not None:
        y_shared = _c(y_shared, np.float32)
        gate = _c(gate, np.uint16)
        x = _c(x, np.float32)
    _load().q4o_moe_combine(_p(out), _p(bound), _p(gabs), _p(y), _p(slot), _p(w),
                            _p(y_shared) if y_shared is not None else None,
                            _p(gate) if y_shared is not None else None,
                            _p(x) if y_shared is not None else None, n_tok, k, n_slots, hidden)
    return out, bound, gabs


def gemv_silu(packed, s, b, x_bits, div: float):
    """silu(y / div) of the plain product. Returns (out, y, bound) in float64; bound is the
    product's acceptance bound (the epilogue's own tolerance follows from it)."""
    packed, s, b, x_bits = (_c(packed, np.uint8), _c(s, np.uint16), _c(b, np.uint16),
                            _c(x_bits, np.uint16))
    nb, in_dim = x_bits.shape
    out_dim = packed.shape[0]
    out = np.empty((nb, out_dim), np.float64)
    y = np.empty((nb, out_dim), np.float64)
    bound = np.empty((nb, out_dim), np.float64)
    _load().q4o_gemv_silu(_p(out), _p(y), _p(bound), _p(packed), _p(s), _p(b), _p(x_bits), float(div),
                          nb, out_dim, in_dim)
    return out, y, bound


def rmsnorm_groups_f16(x_raw, norm_w, groups: int, eps: float = 1e-6, shift: float = 0.0):
    """Grouped RMSNorm: each of `groups` equal segments of a row normalised on its own.
    Returns (xn fp16 bits [nb][in_dim], inv_rms [nb][groups])."""
    x_raw, norm_w = _c(x_raw, np.float32), _c(norm_w, np.uint16)
    nb, n = x_raw.shape
    xn = np.empty((nb, n), np.uint16)
    inv = np.empty((nb, groups), np.float64)
    _load().q4o_rmsnorm_groups_f16(_p(xn), _p(inv), _p(x_raw), _p(norm_w), float(eps), float(shift), nb, n,
                                   int(groups))
    return xn, inv


def inject_rmsnorm_groups_f16(x_raw, out, logit, norm_w, groups: int, eps: float = 1e-6, shift: float = 0.0):
    """Hyper-connection injection, then the grouped RMSNorm ([BATCH_MSL] hyperconnection.metal
    fn_inject_b; fn_norm_prep_b with inject = 1): stream g of row r (inputs g*n .. g*n+n-1,
    n = in_dim / groups) becomes x + out[r] * 2 sigmoid(logit[r][g] / groups), then each stream
    is normalised on its own. x_raw fp32 [nb][in_dim], out fp32 [nb][n], logit fp32
    [nb][groups]. Returns (xn fp16 bits [nb][in_dim], x_new float64 [nb][in_dim])."""
    x_raw, out, logit, norm_w = (_c(x_raw, np.float32), _c(out, np.float32), _c(logit, np.float32),
                                 _c(norm_w, np.uint16))
    nb, in_dim = x_raw.shape
    assert out.shape == (nb, in_dim // groups) and logit.shape == (nb, groups)
    xn = np.empty((nb, in_dim), np.uint16)
    x_new = np.empty((nb, in_dim), np.float64)
    _load().q4o_inject_rmsnorm_groups_f16(_p(xn), _p(x_new), _p(x_raw), _p(out), _p(logit), _p(norm_w), float(eps),
                                          float(shift), nb, in_dim, int(groups))
    return xn, x_new


# ---- derived low-bit codes ([BATCH_MSL] fn_q2_rows_h, fn_q3_rows_h) ------------------------


def lowbit_pack2(codes):
    """4-bit codes [rows][in] (one per byte) -> 2-bit packed rows [rows][in/4] of q4 >> 2."""
    codes = _c(codes, np.uint8)
    rows, in_dim = codes.shape
    out = np.empty((rows, in_dim // 4), np.uint8)
    _load().q4o_lowbit_pack2(_p(out), _p(codes), rows, in_dim)
    return out


def lowbit_pack3lo(codes):
    """4-bit codes [rows][in] -> the lowest-bit plane [rows][in/8] of the 3-bit codes q4 >> 1."""
    codes = _c(codes, np.uint8)
    rows, in_dim = codes.shape
    out = np.empty((rows, in_dim // 8), np.uint8)
    _load().q4o_lowbit_pack3lo(_p(out), _p(codes), rows, in_dim)
    return out


def lowbit_codes(w2, wlo=None):
    """The derived codes read back from the packed layout: q2 (wlo None) or q3."""
    w2 = _c(w2, np.uint8)
    rows, in_dim = w2.shape[0], w2.shape[1] * 4
    wlo = None if wlo is None else _c(wlo, np.uint8)
    out = np.empty((rows, in_dim), np.uint8)
    _load().q4o_lowbit_codes(_p(out), _p(w2), _p(wlo), rows, in_dim)
    return out


def gemv_lowbit(w2, wlo, s, b, x_bits):
    """y = W x with W from derived 2-bit (wlo None) or 3-bit codes. Returns (y, bound)."""
    w2, s, b, x_bits = _c(w2, np.uint8), _c(s, np.uint16), _c(b, np.uint16), _c(x_bits, np.uint16)
    wlo = None if wlo is None else _c(wlo, np.uint8)
    nb, in_dim = x_bits.shape
    out_dim = w2.shape[0]
    y = np.empty((nb, out_dim), np.float64)
    bound = np.empty((nb, out_dim), np.float64)
    _load().q4o_gemv_lowbit(_p(y), _p(bound), _p(w2), _p(wlo), _p(s), _p(b), _p(x_bits), nb, out_dim, in_dim)
    return y, bound


def experts_lowbit(w2_bank, wlo_bank, s_bank, b_bank, x, x_rows, expert_ids, token_offsets, n_experts: int,
                   out_dim: int):
    """Routed low-bit experts ([BATCH_MSL] expert_gemm.metal fn_expert_qmm; the routed form of
    fn_q2_rows_h / fn_q3_rows_h): 2-bit codes (wlo_bank None) or 3-bit codes, activations fp32
    (a float32 array) or binary16 bits (a uint16 array). Returns (y, bound) in float64."""
    w2_bank, s_bank, b_bank = _c(w2_bank, np.uint8), _c(s_bank, np.uint16), _c(b_bank, np.uint16)
    wlo_bank = None if wlo_bank is None else _c(wlo_bank, np.uint8)
    x32 = _c(x, np.float32) if np.asarray(x).dtype == np.float32 else None
    x16 = None if x32 is not None else _c(x, np.uint16)
    expert_ids, token_offsets = _c(expert_ids, np.int32), _c(token_offsets, np.int32)
    xr = None if x_rows is None else _c(x_rows, np.int32)
    in_dim = (x32 if x32 is not None else x16).shape[1]
    n_rows = int(token_offsets[-1])
    y = np.empty((n_rows, out_dim), np.float64)
    bound = np.empty((n_rows, out_dim), np.float64)
    _load().q4o_experts_lowbit(_p(y), _p(bound), _p(w2_bank), _p(wlo_bank), _p(s_bank), _p(b_bank), _p(x32), _p(x16),
                               _p(xr), _p(expert_ids), _p(token_offsets), expert_ids.shape[0], n_experts, out_dim,
                               in_dim)
    return y, bound


# ---- prefill helpers ------------------------------------------------------------------------


def gemv_f32x(packed, s, b, x_f32):
    """y = W x with fp32 activations as given ([BATCH_MSL] fn_qmv_small_b). Returns (y, bound)."""
    packed, s, b, x = _c(packed, np.uint8), _c(s, np.uint16), _c(b, np.uint16), _c(x_f32, np.float32)
    nb, in_dim = x.shape
    out_dim = packed.shape[0]
    y = np.empty((nb, out_dim), np.float64)
    bound = np.empty((nb, out_dim), np.float64)
    _load().q4o_gemv_f32x(_p(y), _p(bound), _p(packed), _p(s), _p(b), _p(x), nb, out_dim, in_dim)
    return y, bound


def quantize(w_f32):
    """4-bit affine min/max quantiser (binary32 steps). Returns (packed, s bits, b bits)."""
    w = _c(w_f32, np.float32)
    rows, in_dim = w.shape
    packed = np.empty((rows, in_dim // 2), np.uint8)
    s = np.empty((rows, in_dim // 64), np.uint16)
    b = np.empty((rows, in_dim // 64), np.uint16)
    _load().q4o_quantize(_p(packed), _p(s), _p(b), _p(w), rows, in_dim)
    return packed, s, b

