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
    lib.q4a_decode_mlp.argtypes = [P, P, P, P, P, P, P, F, F, P, P, P, I32, I64, I64, P]
    lib.q4a_gemv_inject_rmsnorm_grouped.argtypes = [P, P, P, P, P, P, P, P, P, F, F, I32, I32, I64, I64, P]
    lib.q4a_debug_withhold_stage.argtypes = [I32]
    lib.q4a_gemv_kernel_choice.argtypes = [P, P, I32, I64, I64]
    lib.q4a_gemv_experts_gate_up_silu.argtypes = [P, P, P, P, P, P, P, P, I32, I32, I64, I64, I64, P]
    lib.q4a_gemv_experts_lowbit.argtypes = [P, I32, P, P, P, P, P, I32, P, P, P, I32, I32, I64, I64, I64, P]
    lib.q4a_check_device_error.argtypes = [P]
    lib.q4a_last_cuda_error.restype = I32
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



def test_decode_mlp_rejections(lib):
    A = 0x1000
    f = lib.q4a_decode_mlp

    def call(y=A, h=A, wg=A, sg=A, bg=A, x=A, nw=A, eps=1e-6, wd=A, sd=A, bd=A, nb=1, hidden=512, inter=128):
        return f(y, h, wg, sg, bg, x, nw, eps, 0.0, wd, sd, bd, nb, hidden, inter, None)

    assert call(y=None) == NULL
    assert call(wd=None) == NULL
    assert call(nb=0) == SHAPE
    assert call(eps=-1.0) == SHAPE
    assert call(inter=96) == SHAPE                      # the down projection's in_dim % 64
    assert call(hidden=500) == SHAPE
    assert call(nb=33) == UNSUP
    assert call(h=A + 8) == ALIGN                       # h is the down projection's x: 16 bytes
    assert call(wd=A + 4) == ALIGN
    assert call(hidden=576) == UNSUP                    # 9 groups: no 2D scale boxes
    assert call(sg=A + 2) == UNSUP


def test_inject_rejections(lib):
    A = 0x100000
    f = lib.q4a_gemv_inject_rmsnorm_grouped

    def call(y=A, xn=0x200000, x=A, o=0x300000, lg=0x400000, nw=A, eps=1e-6, groups=2, nb=2, out_dim=64,
             in_dim=512):
        return f(y, xn, A, A, A, x, o, lg, nw, eps, 0.0, groups, nb, out_dim, in_dim, None)

    assert call(o=None) == NULL
    assert call(lg=None) == NULL
    assert call(groups=3) == SHAPE                 # 512 % (64 * 3)
    assert call(eps=-1.0) == SHAPE
    assert call(xn=A) == SHAPE                     # x_new overlaps x_raw
    assert call(xn=A + 2048) == SHAPE              # partial overlap (x_raw is 2 x 512 fp32)
    assert call(xn=0x300000 + 256) == SHAPE        # overlaps out (2 x 256 fp32)
    assert call(nb=33) == UNSUP
    assert call(groups=16, in_dim=1024) == UNSUP
    assert call(o=0x300000 + 4) == ALIGN
    assert call(xn=0x200000 + 8) == ALIGN
    assert call(lg=0x400000 + 2) == ALIGN


# ---- the Python binding refuses mis-shaped buffers before anything launches -------------

@pytest.fixture(scope="module")
def q4a():
    torch = pytest.importorskip("torch")
    _builder().build()
    import affine_q4_dequant_gb300 as mod

    return mod, torch


def test_binding_kernel_choice(q4a):
    mod, _ = q4a
    assert mod.gemv_kernel_choice(0x10000, 0x10000, 16, 151936, 4096) == "tcgen05"
    assert mod.gemv_kernel_choice(0x10000, 0x10000, 16, 12288, 4096) == "gemv"


def _bad(fn, what):
    with pytest.raises(ValueError, match=what):
        fn()


def test_binding_checks_matrix_shapes(q4a):
    mod, torch = q4a
    u8, bf, f16, f32 = torch.uint8, torch.bfloat16, torch.float16, torch.float32
    w = torch.zeros(16, 256, dtype=u8)
    s = torch.zeros(16, 8, dtype=bf)
    x = torch.zeros(2, 512, dtype=f16)
    _bad(lambda: mod.gemv(torch.zeros(16, 255, dtype=u8), s, s, x), "w: shape")
    _bad(lambda: mod.gemv(w, torch.zeros(8, 8, dtype=bf), s, x), "s: shape")
    _bad(lambda: mod.gemv(w, s, torch.zeros(16, 4, dtype=bf), x), "b: shape")
    _bad(lambda: mod.gemv(w, s, s, x, out=torch.zeros(1, 16, dtype=f32)), "y: shape")
    _bad(lambda: mod.gemv(w, s, s, torch.zeros(2, 500, dtype=f16)), "multiple of 64")
    _bad(lambda: mod.gemv_silu(w, s, s, x, 2.0, out=torch.zeros(2, 17, dtype=f32)), "y: shape")
    _bad(lambda: mod.gemv_f32x(w, s, s, torch.zeros(2, 512, dtype=f32), out=torch.zeros(3, 16, dtype=f32)),
         "y: shape")
    with pytest.raises(TypeError, match="CUDA"):
        mod.gemv(w, s, s, x)                            # right shapes, but host memory


def test_binding_checks_fused_and_norm_shapes(q4a):
    mod, torch = q4a
    u8, bf, f16, f32 = torch.uint8, torch.bfloat16, torch.float16, torch.float32
    w = torch.zeros(32, 256, dtype=u8)                  # 16 gate rows + 16 up rows
    s = torch.zeros(32, 8, dtype=bf)
    x = torch.zeros(2, 512, dtype=f16)
    a = torch.zeros(2, 512, dtype=f32)
    nw = torch.zeros(512, dtype=bf)
    _bad(lambda: mod.gemv_gate_up_silu(w, s, s, x, out=torch.zeros(2, 32, dtype=f16)), "h: shape")
    _bad(lambda: mod.gemv_rmsnorm_gate_up_silu(w, s, s, a, torch.zeros(256, dtype=bf)), "norm_w: shape")
    _bad(lambda: mod.gemv_rmsnorm(w, s, s, a, nw, out=torch.zeros(2, 16, dtype=f32)), "y: shape")
    _bad(lambda: mod.gemv_rmsnorm_grouped(w, torch.zeros(32, 4, dtype=bf), s, a, nw, 2), "s: shape")
    o = torch.zeros(2, 256, dtype=f32)
    lg = torch.zeros(2, 2, dtype=f32)
    _bad(lambda: mod.gemv_inject_rmsnorm_grouped(w, s, s, a, torch.zeros(2, 512, dtype=f32), lg, nw, 2), "out: shape")
    _bad(lambda: mod.gemv_inject_rmsnorm_grouped(w, s, s, a, o, torch.zeros(2, 3, dtype=f32), nw, 2), "logit: shape")
    _bad(lambda: mod.gemv_inject_rmsnorm_grouped(w, s, s, a, o, lg, nw, 2, x_new=torch.zeros(2, 256, dtype=f32)),
         "x_new: shape")
    _bad(lambda: mod.gemv_inject_rmsnorm_grouped(w, s, s, a, o, lg, nw, 3), "streams")
    # 16 gate + 16 up rows make inter = 16: the down projection's rows are too short
    _bad(lambda: mod.decode_mlp(w, s, s, a, nw, torch.zeros(512, 8, dtype=u8), torch.zeros(512, 0, dtype=bf),
                                torch.zeros(512, 0, dtype=bf)), "multiple of 64")
    w2 = torch.zeros(128, 256, dtype=u8)                # inter 64: down 64 -> 512
    s2 = torch.zeros(128, 8, dtype=bf)
    wd2 = torch.zeros(512, 32, dtype=u8)
    sd2 = torch.zeros(512, 1, dtype=bf)
    _bad(lambda: mod.decode_mlp(w2, s2, s2, a, nw, torch.zeros(511, 32, dtype=u8), sd2, sd2), "w_dn: shape")
    _bad(lambda: mod.decode_mlp(w2, s2, s2, a, nw, wd2, sd2, sd2, h=torch.zeros(2, 32, dtype=f16)), "h: shape")
    _bad(lambda: mod.decode_mlp(w2, s2, s2, a, nw, wd2, sd2, sd2, out=torch.zeros(2, 64, dtype=f32)), "y: shape")


def test_binding_checks_expert_and_helper_shapes(q4a):
    mod, torch = q4a
    u8, bf, f16, f32, i32 = torch.uint8, torch.bfloat16, torch.float16, torch.float32, torch.int32
    # a bank of 2 experts x 16 rows, 512 inputs
    wb = torch.zeros(32, 256, dtype=u8)
    sb = torch.zeros(32, 8, dtype=bf)
    x = torch.zeros(3, 512, dtype=f16)
    _bad(lambda: mod.gemv_experts(torch.zeros(31, 256, dtype=u8), sb, sb, x, None, [0, 1], [0, 2, 3], 2, 16),
         "w_bank: shape")
    _bad(lambda: mod.gemv_experts(wb, sb, sb, x, None, [0, 1], [0, 2, 4], 2, 16), "without x_rows")
    _bad(lambda: mod.gemv_experts(wb, sb, sb, x, torch.zeros(2, dtype=i32), [0, 1], [0, 2, 3], 2, 16),
         "x_rows: shape")
    _bad(lambda: mod.gemv_experts(wb, sb, sb, x, None, [0, 1], [0, 3], 2, 16), "one entry more")
    _bad(lambda: mod.silu_mul_xsum(torch.zeros(2, 256, dtype=f32), h=torch.zeros(2, 64, dtype=f16)), "h: shape")
    _bad(lambda: mod.xsum(x, out=torch.zeros(3, 4, dtype=f32)), "out: shape")
    _bad(lambda: mod.pack(torch.zeros(4, 64, dtype=u8), out=torch.zeros(4, 64, dtype=u8)), "out: shape")
    y = torch.zeros(6, 8, dtype=f32)
    _bad(lambda: mod.moe_combine(y, torch.zeros(3, 2, dtype=i32), torch.zeros(3, 1, dtype=f32)), "w: shape")
    _bad(lambda: mod.moe_combine(y, torch.zeros(3, 2, dtype=i32), torch.zeros(3, 2, dtype=f32),
                                 y_shared=torch.zeros(3, 8, dtype=f32), gate=torch.zeros(4, dtype=bf),
                                 x=torch.zeros(3, 8, dtype=f32)), "gate: shape")
    _bad(lambda: mod.gemv_lowbit(3, torch.zeros(16, 128, dtype=u8), torch.zeros(16, 63, dtype=u8),
                                 torch.zeros(16, 8, dtype=bf), torch.zeros(16, 8, dtype=bf), x[:2]), "w_lo: shape")


def _has_gpu():
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False


def test_cuda_failure_is_reported(lib):
    """A valid call on a machine with no usable CUDA device reaches the runtime, which fails:
    the call returns Q4A_ERR_CUDA and q4a_last_cuda_error holds the runtime's error code (the
    launchers' error path, made to fail on the host; no GPU is faulted)."""
    if _has_gpu():
        pytest.skip("a CUDA device is present: the runtime does not fail here")
    A = 0x1000
    assert lib.q4a_gemv(A, A, A, A, A, 1, 64, 512, None) == CUDA
    assert lib.q4a_last_cuda_error() != 0
    assert b"CUDA" in lib.q4a_status_string(CUDA)
    assert lib.q4a_check_device_error(None) == CUDA


def test_gemv_kernel_choice_rule(lib):
    """q4a_gemv's routing (host logic, no launch): the tensor-core path from NB 64, from NB 9
    on matrices of >= 38912 rows (152 units of 256 rows) and from NB 17 on matrices of >= 12288
    rows (48 units), when in_dim % 512 == 0 and the scales and biases are 16-byte aligned; the
    GEMV kernel otherwise."""
    A = 0x10000
    k = lib.q4a_gemv_kernel_choice
    assert [k(A, A, nb, 151936, 4096) for nb in (1, 8, 9, 12, 13, 16, 17, 32, 63, 64, 128, 300)] == \
        [0, 0, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1]
    assert [k(A, A, nb, 38911, 4096) for nb in (9, 16, 17, 32, 63, 64)] == [0, 0, 1, 1, 1, 1]
    assert [k(A, A, nb, 38912, 4096) for nb in (8, 9)] == [0, 1]
    assert [k(A, A, nb, 12288, 4096) for nb in (1, 9, 16, 17, 32, 64)] == [0, 0, 0, 1, 1, 1]
    assert [k(A, A, nb, 12287, 4096) for nb in (17, 63, 64)] == [0, 0, 1]
    assert [k(A, A, nb, 4096, 12288) for nb in (16, 32, 63, 64)] == [0, 0, 0, 1]
    assert k(A + 2, A, 64, 4096, 4096) == 0        # scales not 16-byte aligned
    assert k(A, A + 8, 64, 4096, 4096) == 0        # biases not 16-byte aligned
    assert k(A, A, 64, 4096, 4096 + 64) == 0       # 65 groups: not a multiple of 8
    assert k(A, A, 64, 4096, 512) == 1
    assert k(None, A, 64, 4096, 4096) == 0 and k(A, A, 0, 4096, 4096) == 0 and k(A, A, 64, 4096, 100) == 0


def test_withhold_stage_hook_arguments(lib):
    assert lib.q4a_debug_withhold_stage(-2) == SHAPE
    assert lib.q4a_debug_withhold_stage(3) == OK
    assert lib.q4a_debug_withhold_stage(-1) == OK     # clears the request


def test_experts_gate_up_silu_rejections(lib):
    A = 0x1000
    f = lib.q4a_gemv_experts_gate_up_silu
    ids = np.array([0, 1], np.int32)
    offs = np.array([0, 2, 3], np.int32)
    pi, po = ctypes.c_void_p(ids.ctypes.data), ctypes.c_void_p(offs.ctypes.data)
    ok = dict(h=A, w=A, s=A, b=A, x=A, xr=None, ids=pi, offs=po, na=2, ne=4, nr=3, inter=640, ind=2048)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["h"], a["w"], a["s"], a["b"], a["x"], a["xr"], a["ids"], a["offs"], a["na"], a["ne"], a["nr"],
                 a["inter"], a["ind"], None)

    assert call(h=None) == NULL and call(ids=None) == NULL
    assert call(inter=8) == SHAPE                  # inter % 16
    assert call(inter=648) == SHAPE
    assert call(nr=4) == SHAPE                     # token_offsets[-1] != n_rows
    assert call(h=A + 8) == ALIGN                  # h 16-byte aligned
    assert call(ind=2048 + 64) == UNSUP            # in_dim % 512
    assert call(s=A + 2) == UNSUP                  # scales must be 16-byte aligned for the fused form


def test_experts_lowbit_rejections(lib):
    A = 0x1000
    f = lib.q4a_gemv_experts_lowbit
    ids = np.array([0, 1], np.int32)
    offs = np.array([0, 2, 3], np.int32)
    pi, po = ctypes.c_void_p(ids.ctypes.data), ctypes.c_void_p(offs.ctypes.data)

    def call(y=A, bits=2, w=A, lo=None, s=A, b=A, x=A, f32=1, xr=None, ids_=pi, offs_=po, n_active=2, n_exp=4,
             n_rows=3, out_dim=8, in_dim=128):
        return f(y, bits, w, lo, s, b, x, f32, xr, ids_, offs_, n_active, n_exp, n_rows, out_dim, in_dim, None)

    assert call(bits=4) == UNSUP
    assert call(bits=3) == NULL                     # 3-bit codes need the lowest-bit plane
    assert call(x=None) == NULL
    assert call(ids_=None) == NULL
    assert call(n_active=0) == SHAPE
    assert call(n_rows=4) == SHAPE                  # offsets end != n_rows
    assert call(bits=3, lo=A, in_dim=192) == SHAPE  # 3-bit: in_dim % 128
    assert call(in_dim=100) == SHAPE
    assert call(w=A + 4) == ALIGN
    assert call(bits=3, lo=A + 8) == ALIGN
    assert call(x=A + 8) == ALIGN
