"""Property checks of the CPU oracle on random inputs (hypothesis; CPU only).

Each property follows from the definitions on the pages and pins the oracle independently
of its own arithmetic: packing is a bijection on 4-bit codes, the derived low-bit codes are
the shifted 4-bit codes, the product is linear in the activations and additive in the
weight rows, and the quantiser reconstructs every weight within half a step of its group.
"""

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle  # noqa: E402
import q4a_workloads as wl  # noqa: E402

SETTINGS = settings(max_examples=40, deadline=None)


def _case(seed, rows, groups, nb):
    rng = np.random.default_rng(seed)
    in_dim = 64 * groups
    codes = rng.integers(0, 16, (rows, in_dim), dtype=np.uint8)
    s = wl.f32_to_bf16_bits(np.abs(rng.normal(0, 0.02, (rows, groups))).astype(np.float32))
    b = wl.f32_to_bf16_bits((-8 * rng.normal(0, 0.01, (rows, groups))).astype(np.float32))
    x = wl.f16_bits(rng.normal(0, 1, (nb, in_dim)))
    return codes, s, b, x


@SETTINGS
@given(seed=st.integers(0, 2 ** 31), rows=st.integers(1, 9), groups=st.integers(1, 4))
def test_pack_is_a_bijection(seed, rows, groups):
    codes = np.random.default_rng(seed).integers(0, 256, (rows, 64 * groups), dtype=np.uint8)
    packed = oracle.pack(codes)
    assert np.array_equal(oracle.unpack(packed, 64 * groups), codes & 15)
    assert np.array_equal(oracle.pack(oracle.unpack(packed, 64 * groups)), packed)


@SETTINGS
@given(seed=st.integers(0, 2 ** 31), rows=st.integers(1, 7), chunks=st.integers(1, 6))
def test_lowbit_codes_round_trip(seed, rows, chunks):
    in_dim = 64 * chunks
    codes = np.random.default_rng(seed).integers(0, 16, (rows, in_dim), dtype=np.uint8)
    w2, lo = oracle.lowbit_pack2(codes), oracle.lowbit_pack3lo(codes)
    assert np.array_equal(oracle.lowbit_codes(w2), codes >> 2)
    assert np.array_equal(oracle.lowbit_codes(w2, lo), codes >> 1)
    # every byte of the 2-bit plane carries exactly four codes: repacking its read-back is exact
    assert np.array_equal(oracle.lowbit_pack2(oracle.lowbit_codes(w2) << 2), w2)


@SETTINGS
@given(seed=st.integers(0, 2 ** 31), rows=st.integers(1, 6), groups=st.integers(1, 3),
       alpha=st.sampled_from([0.5, 2.0, -1.0, 0.25]))
def test_gemv_is_linear_in_x(seed, rows, groups, alpha):
    codes, s, b, x = _case(seed, rows, groups, 2)
    packed = oracle.pack(codes)
    # scaling by 1/2 or 1/4 is exact in binary16 only away from the subnormal range: inputs
    # that would leave the normal range are zeroed, so alpha * x is representable exactly
    xf = x.view(np.float16).astype(np.float32)
    xf[np.abs(xf) < 2.0 ** -12] = 0.0
    x = wl.f16_bits(xf.astype(np.float64))
    y1, _ = oracle.gemv(packed, s, b, x)
    ya, _ = oracle.gemv(packed, s, b, wl.f16_bits((alpha * xf).astype(np.float64)))
    np.testing.assert_allclose(ya, alpha * y1, rtol=1e-12, atol=1e-12)
    # additivity over activation rows: the sum of two rows' products is the product of the sum
    # (the f32x product takes the fp32 sum exactly)
    y2, _ = oracle.gemv_f32x(packed, s, b, (xf[:1] + xf[1:]).astype(np.float32))
    np.testing.assert_allclose(y2[0], y1[0] + y1[1], rtol=1e-9, atol=1e-9)


@SETTINGS
@given(seed=st.integers(0, 2 ** 31), rows=st.integers(1, 6), groups=st.integers(1, 3),
       scale=st.sampled_from([1e-3, 0.05, 3.0, 400.0]))
def test_quantize_reconstructs_within_half_a_step(seed, rows, groups, scale):
    rng = np.random.default_rng(seed)
    w = (rng.normal(0, scale, (rows, 64 * groups))).astype(np.float32)
    packed, s, b = oracle.quantize(w)
    q = oracle.unpack(packed, 64 * groups).astype(np.float64)
    sf = np.repeat(wl.bf16_bits_to_f32(s).astype(np.float64), 64, axis=1)
    bf = np.repeat(wl.bf16_bits_to_f32(b).astype(np.float64), 64, axis=1)
    gmin = np.repeat(w.reshape(rows, groups, 64).min(axis=2), 64, axis=1).astype(np.float64)
    err = np.abs(sf * q + bf - w)
    assert np.all(err <= 0.5 * sf + np.abs(bf - gmin) + 16 * sf * 2.0 ** -8 + 1e-30)
