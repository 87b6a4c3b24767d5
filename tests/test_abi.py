"""The C ABI without a GPU: libq4a.so loads, exports every entry point that
include/q4a.h declares, and rejects invalid arguments on the host (before any
CUDA call) with the documented status codes."""

import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q4a.h")

OK, NULL, SHAPE, ALIGN, UNSUP, CUDA, TIMEOUT = range(7)


def _builder():
    import __graft_entry__

    return __graft_entry__._build_module()


@pytest.fixture(scope="module")
def lib():
    path = _builder().build()
    lib = ctypes.CDLL(path)
    P, I64, I32, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.q4a_status_string.restype = ctypes.c_char_p
    lib.q4a_status_string.argtypes = [I32]
    lib.q4a_pack.argtypes = [P, P, I64, I64, P]
    lib.q4a_xsum.argtypes = [P, P, I32, I64, P]
    lib.q4a_gemv.argtypes = [P, P, P, P, P, I32, I64, I64, P]
    lib.q4a_gemv_experts.argtypes = [P, P, P, P, P, P, P, P, I32, I32, I64, I64, I64, P]
    lib.q4a_gemv_rmsnorm.argtypes = [P, P, P, P, P, P, F, F, I32, I64, I64, P]
    lib.q4a_silu_mul_xsum.argtypes = [P, P, P, I64, I64, P]
    lib.q4a_moe_combine.argtypes = [P, P, P, P, I32, I32, I64, I64, P, P, P, P]
    lib.q4a_gemv_silu.argtypes = [P, P, P, P, P, F, I32, I64, I64, P]
    lib.q4a_gemv_rmsnorm_grouped.argtypes = [P, P, P, P, P, P, F, F, I32, I32, I64, I64, P]
    lib.q4a_lowbit_pack.argtypes = [P, P, P, I64, I64, P]
    lib.q4a_gemv_lowbit.argtypes = [P, I32, P, P, P, P, P, I32, I64, I64, P]
    lib.q4a_gemv_gate_up_silu.argtypes = [P, P, P, P, P, I32, I64, I64, P]
    lib.q4a_quantize.argtypes = [P, P, P, P, I64, I64, P]
    lib.q4a_gemv_f32x.argtypes = [P, P, P, P, P, I32, I64, I64, P]
    lib.q4a_gemv_rmsnorm_gate_up_silu.argtypes = [P, P, P, P, P, P, F, F, I32, I64, I64, P]
    return lib


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"Q4A_API\s+[\w\s\*]+?\b(q4a_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("q4a_pack", "q4a_xsum", "q4a_gemv", "q4a_gemv_experts", "q4a_gemv_rmsnorm",
                     "q4a_silu_mul_xsum", "q4a_status_string", "q4a_check_device_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_exports_nothing_else():
    import subprocess

    out = subprocess.run(["nm", "-D", "--defined-only", _builder().build()], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(declared_functions())


def test_status_strings(lib):
    for code in range(7):
        assert lib.q4a_status_string(code)
    assert lib.q4a_status_string(99) == b"unknown status"


A = 0x10000        # a fake, aligned "device" address (never dereferenced on rejection)


def test_pack_rejections(lib):
    assert lib.q4a_pack(None, A, 4, 64, None) == NULL
    assert lib.q4a_pack(A, A, 0, 64, None) == SHAPE
    assert lib.q4a_pack(A, A, 4, 96, None) == SHAPE
    assert lib.q4a_pack(A + 8, A, 4, 64, None) == ALIGN


def test_xsum_rejections(lib):
    assert lib.q4a_xsum(A, None, 1, 64, None) == NULL
    assert lib.q4a_xsum(A, A, 0, 64, None) == SHAPE
    assert lib.q4a_xsum(A, A, 1, 100, None) == SHAPE
    assert lib.q4a_xsum(A, A + 2, 1, 64, None) == ALIGN


def test_gemv_rejections(lib):
    g = lib.q4a_gemv
    assert g(A, A, A, None, A, 1, 8, 64, None) == NULL
    assert g(A, A, A, A, A, 0, 8, 64, None) == SHAPE
    assert g(A, A, A, A, A, 1, 0, 64, None) == SHAPE
    assert g(A, A, A, A, A, 1, 8, 32, None) == SHAPE
    assert g(A, A, A, A, A, 1, 8, 65, None) == SHAPE
    assert g(A, A + 4, A, A, A, 1, 8, 64, None) == ALIGN      # w not 16-byte aligned
    assert g(A, A, A, A, A + 8, 1, 8, 64, None) == ALIGN      # x not 16-byte aligned
    assert g(A, A, A + 1, A, A, 1, 8, 64, None) == ALIGN      # s not 2-byte aligned
    assert g(A, A, A, A, A, 300, 8, 64, None) == UNSUP        # more than 8 token chunks


def test_rmsnorm_rejections(lib):
    r = lib.q4a_gemv_rmsnorm
    assert r(A, A, A, A, A, None, 1e-6, 0.0, 1, 8, 64, None) == NULL
    assert r(A, A, A, A, A, A, -1.0, 0.0, 1, 8, 64, None) == SHAPE
    assert r(A, A, A, A, A, A, float("nan"), 0.0, 1, 8, 64, None) == SHAPE
    assert r(A, A, A, A, A + 4, A, 1e-6, 0.0, 1, 8, 64, None) == ALIGN
    assert r(A, A, A, A, A, A, 1e-6, 0.0, 33, 8, 64, None) == UNSUP


def test_experts_rejections(lib):
    e = lib.q4a_gemv_experts
    ids = np.array([0, 1], np.int32)
    offs = np.array([0, 2, 3], np.int32)
    pi = ctypes.c_void_p(ids.ctypes.data)
    po = ctypes.c_void_p(offs.ctypes.data)
    assert e(A, A, A, A, A, None, None, po, 2, 4, 3, 8, 64, None) == NULL
    assert e(A, A, A, A, A, None, pi, po, 0, 4, 3, 8, 64, None) == SHAPE
    assert e(A, A, A, A, A, None, pi, po, 513, 4, 3, 8, 64, None) == SHAPE
    assert e(A, A, A, A, A, None, pi, po, 2, 4, 4, 8, 64, None) == SHAPE   # offsets end != n_rows
    bad = np.array([0, 3, 2], np.int32)                                     # decreasing
    assert e(A, A, A, A, A, None, pi, ctypes.c_void_p(bad.ctypes.data), 2, 4, 2, 8, 64, None) == SHAPE
    first = np.array([1, 2, 3], np.int32)                                   # offsets[0] != 0
    assert e(A, A, A, A, A, None, pi, ctypes.c_void_p(first.ctypes.data), 2, 4, 3, 8, 64, None) == SHAPE
    assert e(A, A, A, A, A + 2, None, pi, po, 2, 4, 3, 8, 64, None) == ALIGN
    assert e(A, A, A, A, A, A + 2, pi, po, 2, 4, 3, 8, 64, None) == ALIGN    # x_rows


def test_silu_rejections(lib):
    s = lib.q4a_silu_mul_xsum
    assert s(None, A, A, 1, 64, None) == NULL
    assert s(A, A, A, 1, 96, None) == SHAPE
    assert s(A, A, A, 0, 64, None) == SHAPE
    assert s(A + 2, A, A, 1, 64, None) == ALIGN
    assert s(A, A + 2, A, 1, 64, None) == ALIGN


def test_moe_combine_rejections(lib):
    A = 0x1000    # a 16-byte aligned stand-in address; nothing is dereferenced on rejection
    f = lib.q4a_moe_combine
    assert f(None, A, A, A, 2, 8, 16, 2048, None, None, None, None) == NULL
    assert f(A, A, A, A, 2, 8, 16, 2048, A, None, A, None) == NULL          # shared term without gate
    assert f(A, A, A, A, 0, 8, 16, 2048, None, None, None, None) == SHAPE
    assert f(A, A, A, A, 2, 0, 16, 2048, None, None, None, None) == SHAPE
    assert f(A, A, A, A, 2, 8, 16, 2050, None, None, None, None) == SHAPE   # hidden % 4
    assert f(A, A, A, A, 2, 65, 16, 2048, None, None, None, None) == UNSUP  # top_k > 64
    assert f(A + 4, A, A, A, 2, 8, 16, 2048, None, None, None, None) == ALIGN
    assert f(A, A, A + 2, A, 2, 8, 16, 2048, None, None, None, None) == ALIGN
    assert f(A, A, A, A, 2, 8, 16, 2048, A + 8, A, A, None) == ALIGN        # y_shared


def test_gemv_silu_rejections(lib):
    A = 0x1000
    f = lib.q4a_gemv_silu
    assert f(A, A, A, A, A, 0.0, 1, 64, 64, None) == SHAPE              # div = 0
    assert f(A, A, A, A, A, float("inf"), 1, 64, 64, None) == SHAPE
    assert f(A, A, A, A, A, float("nan"), 1, 64, 64, None) == SHAPE
    assert f(None, A, A, A, A, 2.0, 1, 64, 64, None) == NULL
    assert f(A, A, A, A, A, 2.0, 1, 64, 96, None) == SHAPE              # in_dim % 64
    assert f(A, A + 1, A, A, A, 2.0, 1, 64, 64, None) == ALIGN


def test_rmsnorm_grouped_rejections(lib):
    A = 0x1000
    f = lib.q4a_gemv_rmsnorm_grouped
    assert f(A, A, A, A, A, A, 1e-6, 0.0, 0, 1, 64, 512, None) == SHAPE      # groups < 1
    assert f(A, A, A, A, A, A, 1e-6, 0.0, 3, 1, 64, 512, None) == SHAPE      # 512 % (64*3)
    assert f(A, A, A, A, A, A, 1e-6, 0.0, 16, 1, 64, 1024, None) == UNSUP    # groups > 8
    assert f(A, A, A, A, A, A, 1e-6, 0.0, 2, 33, 64, 512, None) == UNSUP     # nb > 32
    assert f(A, A, A, A, A, A, -1.0, 0.0, 2, 1, 64, 512, None) == SHAPE      # eps < 0
    assert f(A, A, A, A, A + 4, A, 1e-6, 0.0, 2, 1, 64, 512, None) == ALIGN  # x_raw


def test_lowbit_rejections(lib):
    A = 0x1000
    f = lib.q4a_lowbit_pack
    assert f(None, None, A, 4, 64, None) == NULL
    assert f(A, None, A, 0, 64, None) == SHAPE
    assert f(A, None, A, 4, 96, None) == SHAPE
    assert f(A + 8, None, A, 4, 64, None) == ALIGN
    assert f(A, A + 4, A, 4, 64, None) == ALIGN
    g = lib.q4a_gemv_lowbit
    assert g(A, 4, A, A, A, A, A, 1, 64, 512, None) == UNSUP    # bits
    assert g(A, 3, A, None, A, A, A, 1, 64, 512, None) == NULL  # 3-bit needs the lowest bits
    assert g(A, 2, A, None, A, A, A, 0, 64, 512, None) == SHAPE
    assert g(A, 3, A, A, A, A, A, 1, 64, 576, None) == SHAPE    # 3-bit: in_dim % 128
    assert g(A, 2, A, None, A, A, A, 257, 64, 512, None) == UNSUP
    assert g(A, 2, A + 4, None, A, A, A, 1, 64, 512, None) == ALIGN


def test_gate_up_silu_rejections(lib):
    A = 0x1000
    f = lib.q4a_gemv_gate_up_silu
    assert f(None, A, A, A, A, 1, 64, 512, None) == NULL
    assert f(A, A, A, A, A, 0, 64, 512, None) == SHAPE
    assert f(A, A, A, A, A, 1, 40, 512, None) == SHAPE      # inter % 16
    assert f(A, A, A, A, A, 1, 64, 500, None) == SHAPE      # in_dim % 64
    assert f(A, A, A, A, A, 257, 64, 512, None) == UNSUP
    assert f(A + 1, A, A, A, A, 1, 64, 512, None) == ALIGN
    assert f(A, A, A, A, A, 1, 64, 576, None) == UNSUP       # 9 groups: no 2D scale boxes
    assert f(A, A, A + 2, A, A, 1, 64, 512, None) == UNSUP   # scales not 16-byte aligned
    g = lib.q4a_gemv_rmsnorm_gate_up_silu
    assert g(A, A, A, A, A, A, 1e-6, 0.0, 33, 64, 512, None) == UNSUP
    assert g(A, A, A, A, A, A, -1.0, 0.0, 1, 64, 512, None) == SHAPE
    assert g(A, A, A, A, A + 4, A, 1e-6, 0.0, 1, 64, 512, None) == ALIGN
    assert g(A, A, A, A, A, A, 1e-6, 0.0, 1, 64, 640, None) == UNSUP


def test_prefill_rejections(lib):
    A = 0x1000
    q = lib.q4a_quantize
    assert q(None, A, A, A, 4, 64, None) == NULL
    assert q(A, A, A, A, 0, 64, None) == SHAPE
    assert q(A, A, A, A, 4, 100, None) == SHAPE
    assert q(A, A, A, A + 4, 4, 64, None) == ALIGN
    f = lib.q4a_gemv_f32x
    assert f(A, A, A, A, None, 1, 8, 64, None) == NULL
    assert f(A, A, A, A, A, 0, 8, 64, None) == SHAPE
    assert f(A, A, A, A, A, 1, 8, 96, None) == SHAPE
    assert f(A, A, A, A, A + 8, 1, 8, 64, None) == ALIGN


def test_gemv_batch_limits(lib):
    A = 0x1000
    # 9 groups are not tensor-core eligible: the GEMV kernel takes at most 256 rows
    assert lib.q4a_gemv(A, A, A, A, A, 257, 64, 576, None) == UNSUP
    assert lib.q4a_gemv(A, A, A, A, A, 0, 64, 576, None) == SHAPE

