"""Pins for the CPU oracle: it is checked here against things other than itself.

Hand-worked examples (tests/golden/), closed forms, invariants, exact rational
arithmetic, numpy/math library routines and brute force on tiny inputs. Each
pin is chosen so that a plausible slip in the oracle (swapped nibbles, a wrong
group index, scale and bias exchanged, a dropped bias term, transposed rows and
tokens, a wrong tie rule) fails at least one of them.
"""

import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import q4a_workloads as wl

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def ramp_codes():
    i = np.arange(64)
    return np.stack([i % 16, 15 - (i % 16)]).astype(np.uint8)


def bf16(vals):
    return wl.f32_to_bf16_bits(np.asarray(vals, np.float32))


# ---- storage-format decoders ------------------------------------------------------

def test_half_decoder_matches_numpy_on_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_value(int(b)) for b in bits[::7]])
    r = ref[::7]
    both_nan = np.isnan(got) & np.isnan(r)
    assert np.all(both_nan | (got == r))


def test_bf16_decoder_matches_fp32_upper_half():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 65536, size=5000).astype(np.uint16)
    ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16_value(int(b)) for b in bits])
    assert np.all((got == ref) | (np.isnan(got) & np.isnan(ref)))


def test_half_round_matches_numpy_round_to_nearest_even():
    rng = np.random.default_rng(2)
    vals = np.concatenate([
        rng.normal(0, 1, 3000), rng.normal(0, 1e-5, 1000), rng.normal(0, 3e4, 500),
        # exact ties between neighbouring binary16 values
        (np.arange(1024, 1100) + 0.5) / 1024.0, (np.arange(0, 40) + 0.5) * 2.0 ** -24,
        [65504.0, 65519.99, 65520.0, -65520.0, 1e9, 0.0, -0.0, 2.0 ** -25, 3 * 2.0 ** -26],
    ])
    ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.half_round(v) for v in vals], np.uint16)
    assert np.array_equal(got, ref)


# ---- A1 packing ---------------------------------------------------------------------

def test_pack_matches_hand_worked_bytes(golden):
    g = golden("pack_ramp.txt")
    packed = oracle.pack(ramp_codes())
    for row, key in ((0, "row0_period_bytes"), (1, "row1_period_bytes")):
        period = bytes(int(h, 16) for h in g[key])
        assert bytes(packed[row]) == period * 4
    words = packed.view("<u4")
    assert [int(w) for w in words[0, :2]] == [int(v, 16) for v in g["row0_words"]]
    assert [int(w) for w in words[1, :2]] == [int(v, 16) for v in g["row1_words"]]


def test_pack_unpack_round_trip_and_mask():
    codes = wl.codes(99, 0, 7, 192)
    assert np.array_equal(oracle.unpack(oracle.pack(codes), 192), codes)
    wide = np.random.default_rng(3).integers(0, 256, size=(3, 64), dtype=np.uint8)
    assert np.array_equal(oracle.unpack(oracle.pack(wide), 64), wide & 0x0F)


# ---- A4 GEMV --------------------------------------------------------------------------

def test_gemv_hand_worked_2x64(golden):
    g = golden("gemv_2x64.txt")
    packed = oracle.pack(ramp_codes())
    s = bf16([[float(v)] for v in g["scale"]])
    b = bf16([[float(v)] for v in g["bias"]])
    x1 = wl.f16_bits(np.ones((1, 64)))
    x2 = wl.f16_bits(((-1.0) ** np.arange(64))[None, :])
    y1, _ = oracle.gemv(packed, s, b, x1)
    y2, _ = oracle.gemv(packed, s, b, x2)
    assert list(y1[0]) == [float(v) for v in g["x_ones_y"]]
    assert list(y2[0]) == [float(v) for v in g["x_alternating_y"]]


def _brute_force(codes, s_bits, b_bits, x_bits):
    """Dense float64 product from the UNPACKED codes (never the packed bytes)."""
    s = wl.bf16_bits_to_f32(s_bits).astype(np.float64)
    b = wl.bf16_bits_to_f32(b_bits).astype(np.float64)
    w = codes.astype(np.float64) * np.repeat(s, 64, axis=1) + np.repeat(b, 64, axis=1)
    x = x_bits.view(np.float16).astype(np.float64)
    return x @ w.T, np.abs(x) @ np.abs(w).T


@pytest.mark.parametrize("out_dim,in_dim,nb", [(1, 64, 1), (3, 128, 2), (8, 64, 3), (5, 192, 3), (2, 128, 1)])
def test_gemv_brute_force_tiny(out_dim, in_dim, nb):
    rng = np.random.default_rng(out_dim * 1000 + in_dim + nb)
    codes = rng.integers(0, 16, size=(out_dim, in_dim), dtype=np.uint8)
    codes[0, :16] = np.arange(16)            # every code value appears
    s = bf16(np.abs(rng.normal(0, 0.5, (out_dim, in_dim // 64))))
    b = bf16(rng.normal(0, 1.0, (out_dim, in_dim // 64)))
    x = wl.f16_bits(rng.normal(0, 1, (nb, in_dim)))
    y, bound = oracle.gemv(oracle.pack(codes), s, b, x)
    ref, mag = _brute_force(codes, s, b, x)
    assert y.shape == (nb, out_dim)
    assert np.all(np.abs(y - ref) <= 1e-12 * mag + 1e-300)
    assert np.allclose(bound, 2e-3 * mag + 1e-5, rtol=1e-12, atol=0)


def test_gemv_exact_rational():
    """Power-of-two scales, integer biases and integer x: every product and sum is
    exact in double, so the oracle must equal the rational result exactly."""
    rng = np.random.default_rng(5)
    out_dim, in_dim, nb = 4, 128, 2
    codes = rng.integers(0, 16, size=(out_dim, in_dim), dtype=np.uint8)
    s_val = 2.0 ** rng.integers(-6, 2, size=(out_dim, 2))
    b_val = rng.integers(-5, 6, size=(out_dim, 2)).astype(np.float64)
    x_val = rng.integers(-8, 9, size=(nb, in_dim)).astype(np.float64)
    y, _ = oracle.gemv(oracle.pack(codes), bf16(s_val), bf16(b_val), wl.f16_bits(x_val))
    for r in range(nb):
        for o in range(out_dim):
            exact = sum(Fraction(s_val[o, i // 64]) * int(codes[o, i]) * int(x_val[r, i])
                        + Fraction(b_val[o, i // 64]) * int(x_val[r, i]) for i in range(in_dim))
            assert Fraction(y[r, o]) == exact


def _case(seed, out_dim=6, in_dim=256, nb=3):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(out_dim, in_dim), dtype=np.uint8)
    s = bf16(np.abs(rng.normal(0, 0.02, (out_dim, in_dim // 64))))
    b = bf16(-8 * rng.normal(0, 0.01, (out_dim, in_dim // 64)))
    x = wl.f16_bits(rng.normal(0, 1, (nb, in_dim)))
    return codes, s, b, x


def test_closed_forms_codes_zero_and_fifteen_and_scale_zero():
    codes, s, b, x = _case(6)
    xs = oracle.xsum(x)                                   # [nb][G]
    sv = wl.bf16_bits_to_f32(s).astype(np.float64)
    bv = wl.bf16_bits_to_f32(b).astype(np.float64)
    zero = np.zeros_like(codes)
    y0, _ = oracle.gemv(oracle.pack(zero), s, b, x)
    assert np.allclose(y0, xs @ bv.T, rtol=1e-12, atol=1e-12)
    fifteen = np.full_like(codes, 15)
    y15, _ = oracle.gemv(oracle.pack(fifteen), s, bf16(np.zeros_like(bv)), x)
    assert np.allclose(y15, 15 * (xs @ sv.T), rtol=1e-12, atol=1e-12)
    ys0, _ = oracle.gemv(oracle.pack(codes), bf16(np.zeros_like(sv)), b, x)
    assert np.allclose(ys0, xs @ bv.T, rtol=1e-12, atol=1e-12)


def test_linearity_in_x():
    codes, s, b, x = _case(7)
    p = oracle.pack(codes)
    y, _ = oracle.gemv(p, s, b, x)
    neg = wl.f16_bits(-x.view(np.float16).astype(np.float32))
    dbl = wl.f16_bits(2 * x.view(np.float16).astype(np.float32))
    yn, _ = oracle.gemv(p, s, b, neg)
    yd, _ = oracle.gemv(p, s, b, dbl)
    assert np.array_equal(yn, -y)
    assert np.array_equal(yd, 2 * y)
    # additivity on integer activations (sums stay exact in binary16)
    rng = np.random.default_rng(8)
    x1 = rng.integers(-20, 21, size=x.shape).astype(np.float32)
    x2 = rng.integers(-20, 21, size=x.shape).astype(np.float32)
    ya, _ = oracle.gemv(p, s, b, wl.f16_bits(x1))
    yb, _ = oracle.gemv(p, s, b, wl.f16_bits(x2))
    yab, _ = oracle.gemv(p, s, b, wl.f16_bits(x1 + x2))
    assert np.allclose(yab, ya + yb, rtol=1e-12, atol=1e-9)


def test_explicit_equals_factored_form():
    codes, s, b, x = _case(9, out_dim=5, in_dim=320, nb=4)
    p = oracle.pack(codes)
    y, bound = oracle.gemv(p, s, b, x)
    yf = oracle.gemv_factored(p, s, b, x)
    assert np.all(np.abs(y - yf) <= 1e-9 * bound)


def test_rows_and_tokens_are_not_transposed():
    codes, s, b, x = _case(10, out_dim=3, in_dim=128, nb=2)
    y, _ = oracle.gemv(oracle.pack(codes), s, b, x)
    ref, _ = _brute_force(codes, s, b, x)
    assert y.shape == (2, 3)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    # moving one token row moves only that output row
    x2 = x.copy()
    x2[1] = x[0]
    y2, _ = oracle.gemv(oracle.pack(codes), s, b, x2)
    assert np.array_equal(y2[0], y[0]) and np.array_equal(y2[1], y[0])


def test_entries_match_full_product():
    codes, s, b, x = _case(11, out_dim=9, in_dim=192, nb=3)
    p = oracle.pack(codes)
    y, bound = oracle.gemv(p, s, b, x)
    r = np.array([0, 2, 1, 2]); o = np.array([8, 0, 4, 3])
    ye, be = oracle.gemv_entries(p, s, b, x, r, o)
    assert np.array_equal(ye, y[r, o]) and np.array_equal(be, bound[r, o])


def test_adversarial_scales_propagate():
    codes, s, b, x = _case(12, out_dim=4, in_dim=128, nb=1)
    s = s.copy()
    s[0, 0] = 0x7FC0    # NaN
    s[1, 1] = 0x7F80    # +inf
    s[2, 0] = 0x0001    # smallest bf16 subnormal
    y, _ = oracle.gemv(oracle.pack(codes), s, b, x)
    assert math.isnan(y[0, 0])
    assert math.isinf(y[0, 1]) or math.isnan(y[0, 1])
    assert np.isfinite(y[0, 2:]).all()


# ---- A2 xsum -------------------------------------------------------------------------

def test_xsum_groups_and_library_sum():
    x = np.zeros((2, 192), np.float32)
    x[0, 63] = 1.0
    x[0, 64] = 2.0
    x[1, 191] = -3.0
    xs = oracle.xsum(wl.f16_bits(x))
    assert xs.tolist() == [[1.0, 2.0, 0.0], [0.0, 0.0, -3.0]]
    xr = wl.normal_f16(98, 0, (3, 256))
    ref = xr.view(np.float16).astype(np.float64).reshape(3, 4, 64).sum(axis=2)
    assert np.allclose(oracle.xsum(xr), ref, rtol=1e-14, atol=1e-14)


# ---- A3 RMSNorm ------------------------------------------------------------------------

def test_rmsnorm_closed_form_and_invariants():
    x = np.array([[3.0, 4.0, 0.0, 0.0]], np.float32)
    w = bf16([1.0, 1.0, 1.0, 1.0])
    xn, inv = oracle.rmsnorm_f16(x, w, eps=0.0)
    assert inv[0] == pytest.approx(1 / math.sqrt(25 / 4), rel=1e-15)
    assert xn[0].view(np.float16).tolist() == [float(np.float16(3 * 0.4)), float(np.float16(4 * 0.4)), 0.0, 0.0]
    a = wl.normal_f32(97, 0, (3, 512))
    ones = bf16(np.ones(512))
    xn, _ = oracle.rmsnorm_f16(a, ones, eps=0.0)
    rms = np.sqrt((xn.view(np.float16).astype(np.float64) ** 2).mean(axis=1))
    assert np.allclose(rms, 1.0, atol=2e-3)
    # scale invariance (power-of-two scaling is exact; eps = 0)
    xn8, _ = oracle.rmsnorm_f16(8 * a, ones, eps=0.0)
    assert np.array_equal(xn8, xn)
    # w + shift: (w = 0, shift = 1) equals (w = 1, shift = 0)
    xs1, _ = oracle.rmsnorm_f16(a, bf16(np.zeros(512)), eps=0.0, shift=1.0)
    assert np.array_equal(xs1, xn)
    # weight applies per column
    wv = wl.norm_weight(97, 1, 512)
    xw, inv = oracle.rmsnorm_f16(a, wv, eps=1e-6)
    ref = (a.astype(np.float64) * inv[:, None] * wl.bf16_bits_to_f32(wv).astype(np.float64))
    assert np.array_equal(xw, wl.f16_bits(ref))


# ---- A7 SiLU * up ---------------------------------------------------------------------

def test_silu_mul_special_values_and_library():
    gu = np.array([[0.0, 1.0, 30.0, -30.0, 2.0, 3.0, -1.5, 7.0]], np.float32)
    h = oracle.silu_mul_f16(gu).view(np.float16).astype(np.float64)[0]
    assert h[0] == 0.0
    assert h[1] == np.float16(1 / (1 + math.exp(-1)) * 3.0)
    assert h[2] == np.float16(30.0 * -1.5)
    assert abs(h[3]) < 1e-10
    rng = np.random.default_rng(13)
    gu = rng.normal(0, 2, (3, 128)).astype(np.float32)
    got = oracle.silu_mul_f16(gu)
    g = gu[:, :64].astype(np.float64)
    u = gu[:, 64:].astype(np.float64)
    ref = np.vectorize(lambda a, c: a / (1 + math.exp(-a)) * c)(g, u)
    assert np.array_equal(got, wl.f16_bits(ref))


# ---- routing ----------------------------------------------------------------------------

def test_route_topk_brute_force_and_ties():
    logits = wl.moe_logits()
    idx, w = oracle.route_topk(logits, 8)
    for t in range(logits.shape[0]):
        l = logits[t].astype(np.float64)
        p = np.exp(l - l.max())
        p /= p.sum()
        order = sorted(range(64), key=lambda e: (-p[e], e))[:8]
        assert idx[t].tolist() == order
        assert np.allclose(w[t], p[order] / p[order].sum(), rtol=1e-12)
        assert w[t].sum() == pytest.approx(1.0, rel=1e-12)
    ties = np.zeros((1, 6), np.float32)
    ties[0, 4] = 1.0
    idx, _ = oracle.route_topk(ties, 3)
    assert idx[0].tolist() == [4, 0, 1]
    # the workload generator picks the same experts as the oracle's router
    r = wl.route_by_logits(logits, 8)
    oidx, _ = oracle.route_topk(logits, 8)
    assert np.array_equal(r.chosen, oidx)


def test_route_denominator_floor():
    logits = np.zeros((1, 100000), np.float32)
    _, w = oracle.route_topk(logits, 1)
    assert w[0, 0] == pytest.approx(1e-5 / 6.1035156e-5, rel=1e-9)


# ---- A6 expert banks -------------------------------------------------------------------

def _bank(seed, n_exp=4, out_dim=6, in_dim=128):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(n_exp * out_dim, in_dim), dtype=np.uint8)
    s = bf16(np.abs(rng.normal(0, 0.02, (n_exp * out_dim, in_dim // 64))))
    b = bf16(-8 * rng.normal(0, 0.01, (n_exp * out_dim, in_dim // 64)))
    return codes, s, b


def test_experts_equal_per_expert_dense_product():
    codes, s, b = _bank(14)
    x = wl.normal_f16(96, 0, (5, 128))
    experts = np.array([3, 0, 2], np.int32)
    offsets = np.array([0, 2, 3, 6], np.int32)
    x_rows = np.array([4, 1, 0, 2, 3, 1], np.int32)
    y, _ = oracle.gemv_experts(oracle.pack(codes), s, b, x, x_rows, experts, offsets, 4, 6)
    for a, e in enumerate(experts):
        sl = slice(e * 6, (e + 1) * 6)
        for r in range(offsets[a], offsets[a + 1]):
            ref, _ = _brute_force(codes[sl], s[sl], b[sl], x[x_rows[r]][None])
            assert np.allclose(y[r], ref[0], rtol=1e-12, atol=1e-12)


def test_experts_permutation_and_invalid_id():
    codes, s, b = _bank(15)
    p = oracle.pack(codes)
    x = wl.normal_f16(95, 0, (4, 128))
    y, _ = oracle.gemv_experts(p, s, b, x, None, np.array([1, 3], np.int32),
                               np.array([0, 2, 4], np.int32), 4, 6)
    # swap the two segments (and their x rows): outputs swap accordingly
    xs = x[[2, 3, 0, 1]]
    y2, _ = oracle.gemv_experts(p, s, b, xs, None, np.array([3, 1], np.int32),
                                np.array([0, 2, 4], np.int32), 4, 6)
    assert np.array_equal(y2, y[[2, 3, 0, 1]])
    # x_rows indirection equals a gathered x
    y3, _ = oracle.gemv_experts(p, s, b, x, np.array([2, 3, 0, 1], np.int32),
                                np.array([3, 1], np.int32), np.array([0, 2, 4], np.int32), 4, 6)
    assert np.array_equal(y3, y2)
    y4, _ = oracle.gemv_experts(p, s, b, x, None, np.array([7, 0], np.int32),
                                np.array([0, 1, 4], np.int32), 4, 6)
    assert np.isnan(y4[0]).all() and np.isfinite(y4[1:]).all()


# ---- MoE combine ("BATCH_MSL" page, experts.metal fn_moe_combine_b / fn_shared_add_rows) ----

def test_moe_combine_hand_worked(golden):
    g = golden("moe_combine_2x2.txt")
    y = np.array([[float(v) for v in g[f"y{i}"]] for i in range(3)], np.float32)
    slot = np.array([[int(v) for v in g[f"slot{t}"]] for t in range(2)], np.int32)
    w = np.array([[float(v) for v in g[f"w{t}"]] for t in range(2)], np.float32)
    out, bound, _ = oracle.moe_combine(y, slot, w)
    want = np.array([[float(v) for v in g[f"out{t}"]] for t in range(2)])
    assert np.array_equal(out, want)
    assert np.array_equal(bound, want)      # all terms positive


def test_moe_combine_identity_routing():
    rng = np.random.default_rng(21)
    y = rng.normal(size=(7, 33)).astype(np.float32)
    perm = rng.permutation(7).astype(np.int32)
    out, _, _ = oracle.moe_combine(y, perm[:, None], np.ones((7, 1), np.float32))
    assert np.array_equal(out, y[perm].astype(np.float64))


def test_moe_combine_shared_gate_at_zero_is_half():
    """gate = 0 -> sigmoid(0) = 1/2 exactly."""
    rng = np.random.default_rng(22)
    y = rng.integers(-8, 8, size=(4, 16)).astype(np.float32)
    ysh = rng.integers(-8, 8, size=(2, 16)).astype(np.float32)
    slot = np.array([[0, 3], [2, 1]], np.int32)
    w = np.array([[0.5, 0.5], [0.25, 0.75]], np.float32)
    x = rng.normal(size=(2, 16)).astype(np.float32)
    out, _, gabs = oracle.moe_combine(y, slot, w, ysh, np.zeros(16, np.uint16), x)
    plain, _, _ = oracle.moe_combine(y, slot, w)
    assert np.array_equal(out, plain + 0.5 * ysh)
    assert np.all(gabs == 0.0)


def test_moe_combine_sigmoid_symmetry():
    """sigmoid(-d) = 1 - sigmoid(d): the shared parts for gate and -gate add up to y_shared."""
    rng = np.random.default_rng(23)
    y = rng.normal(size=(5, 24)).astype(np.float32)
    ysh = rng.normal(size=(3, 24)).astype(np.float32)
    slot = rng.integers(0, 5, size=(3, 2)).astype(np.int32)
    w = rng.random((3, 2)).astype(np.float32)
    x = rng.normal(size=(3, 24)).astype(np.float32)
    gate = wl.f32_to_bf16_bits(rng.normal(0, 0.2, 24).astype(np.float32))
    plain, _, _ = oracle.moe_combine(y, slot, w)
    a, _, _ = oracle.moe_combine(y, slot, w, ysh, gate, x)
    b, _, _ = oracle.moe_combine(y, slot, w, ysh, gate ^ np.uint16(0x8000), x)
    assert np.allclose((a - plain) + (b - plain), ysh, rtol=0, atol=1e-12)


def test_moe_combine_saturated_gate_and_linearity():
    rng = np.random.default_rng(24)
    y = rng.normal(size=(6, 8)).astype(np.float32)
    ysh = rng.normal(size=(2, 8)).astype(np.float32)
    slot = np.array([[0, 5, 2], [4, 4, 1]], np.int32)
    w = rng.random((2, 3)).astype(np.float32)
    x = np.full((2, 8), 8.0, np.float32)
    gate = wl.f32_to_bf16_bits(np.full(8, 1.0, np.float32))     # dot = 64: sigmoid = 1 - 1.6e-28
    plain, _, _ = oracle.moe_combine(y, slot, w)
    out, _, gabs = oracle.moe_combine(y, slot, w, ysh, gate, x)
    assert np.allclose(out - plain, ysh, rtol=0, atol=1e-15) and np.all(gabs == 64.0)
    out2, _, _ = oracle.moe_combine(y, slot, 2 * w)               # exact: doubling a float32
    assert np.array_equal(out2, 2 * plain)


def test_moe_combine_invalid_slot_gives_nan_row():
    y = np.ones((3, 4), np.float32)
    out, _, _ = oracle.moe_combine(y, np.array([[0, 3], [1, 2]], np.int32), np.ones((2, 2), np.float32))
    assert np.isnan(out[0]).all() and np.array_equal(out[1], np.full(4, 2.0))


# ---- GEMV with the SiLU epilogue ("BATCH_MSL" page, hyperconnection.metal fn_qmv_silu_b) ----

def _silu_case(seed, out_dim=9, in_dim=128, nb=2):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(out_dim, in_dim), dtype=np.uint8)
    s = wl.f32_to_bf16_bits(np.abs(rng.normal(0, 0.02, (out_dim, in_dim // 64))).astype(np.float32))
    b = wl.f32_to_bf16_bits((-8 * rng.normal(0, 0.01, (out_dim, in_dim // 64))).astype(np.float32))
    x = wl.f16_bits(rng.normal(0, 1, (nb, in_dim)))
    return oracle.pack(codes), s, b, x


def test_gemv_silu_zero_weights_give_zero():
    """q = 0, b = 0 -> y = 0 -> silu(0) = 0 exactly."""
    _, s, _, x = _silu_case(41)
    packed = oracle.pack(np.zeros((9, 128), np.uint8))
    out, y, _ = oracle.gemv_silu(packed, s, np.zeros_like(s), x, 3.0)
    assert np.all(y == 0.0) and np.all(out == 0.0)


def test_gemv_silu_odd_part_identity():
    """silu(v) - silu(-v) = v: the outputs for div and -div differ by y / div."""
    packed, s, b, x = _silu_case(42)
    a, y, _ = oracle.gemv_silu(packed, s, b, x, 0.75)
    c, _, _ = oracle.gemv_silu(packed, s, b, x, -0.75)
    assert np.allclose(a - c, y / 0.75, rtol=1e-13, atol=1e-15)


def test_gemv_silu_matches_the_plain_product_and_limits():
    packed, s, b, x = _silu_case(43)
    out, y, bound = oracle.gemv_silu(packed, s, b, x, 1.0)
    y2, bound2 = oracle.gemv(packed, s, b, x)
    assert np.array_equal(y, y2) and np.array_equal(bound, bound2)
    big, _, _ = oracle.gemv_silu(packed, s, b, x, 1e-4)           # |v| large: silu -> max(v, 0)
    v = y / 1e-4
    pos = v > 50
    assert np.allclose(big[pos], v[pos], rtol=1e-15) and np.all(np.abs(big[v < -50]) < 1e-15)


# ---- grouped RMSNorm ("BATCH_MSL" page, hyperconnection.metal fn_group_norm_b, groups > 1) ----

def test_rmsnorm_groups_one_group_is_the_row_norm():
    rng = np.random.default_rng(51)
    x = rng.normal(0, 2, (3, 256)).astype(np.float32)
    w = wl.norm_weight(0, 0, 256)
    a, ia = oracle.rmsnorm_groups_f16(x, w, 1, eps=1e-6, shift=0.25)
    b, ib = oracle.rmsnorm_f16(x, w, eps=1e-6, shift=0.25)
    assert np.array_equal(a, b) and np.array_equal(ia[:, 0], ib)


def test_rmsnorm_groups_are_independent_segments():
    """Each segment equals the one-group norm of that segment alone (weight slice g*n..)."""
    rng = np.random.default_rng(52)
    x = rng.normal(0, 1, (2, 512)).astype(np.float32)
    x[:, 128:256] *= 40.0                  # one loud segment: the others must not notice
    w = wl.norm_weight(0, 1, 512)
    xn, inv = oracle.rmsnorm_groups_f16(x, w, 4)
    for g in range(4):
        seg, iseg = oracle.rmsnorm_f16(x[:, 128 * g:128 * (g + 1)], w[128 * g:128 * (g + 1)])
        assert np.array_equal(xn[:, 128 * g:128 * (g + 1)], seg) and np.array_equal(inv[:, g], iseg)


def test_rmsnorm_groups_unit_rms_per_segment():
    """w = 1, shift = 0, eps = 0: every segment of the output has RMS 1 (up to fp16 rounding)."""
    rng = np.random.default_rng(53)
    x = rng.normal(0, 1, (2, 384)).astype(np.float32) * np.repeat([0.01, 1.0, 100.0], 128)
    w = wl.f32_to_bf16_bits(np.ones(384, np.float32))
    xn, _ = oracle.rmsnorm_groups_f16(x, w, 3, eps=0.0)
    v = xn.view(np.float16).astype(np.float64).reshape(2, 3, 128)
    assert np.allclose(np.sqrt((v ** 2).mean(axis=2)), 1.0, rtol=2e-3)


# ---- NEXT-3 injection ("BATCH_MSL" hyperconnection.metal fn_inject_b, fn_norm_prep_b inject = 1) ----

def test_inject_zero_logit_adds_out_once():
    """2 sigmoid(0) = 1 exactly: every stream receives out itself. With small integers x + out is
    exact in binary32, so the normalisation equals the pinned grouped RMSNorm of x + out."""
    rng = np.random.default_rng(61)
    nb, groups, n = 3, 4, 64
    x = rng.integers(-8, 9, (nb, groups * n)).astype(np.float32)
    out = rng.integers(-8, 9, (nb, n)).astype(np.float32)
    w = wl.norm_weight(0, 2, groups * n)
    xn, x_new = oracle.inject_rmsnorm_groups_f16(x, out, np.zeros((nb, groups), np.float32), w, groups, eps=1e-6,
                                                 shift=0.25)
    summed = x + np.tile(out, (1, groups))
    assert np.array_equal(x_new, summed.astype(np.float64))
    ref, _ = oracle.rmsnorm_groups_f16(summed, w, groups, eps=1e-6, shift=0.25)
    assert np.array_equal(xn, ref)


def test_inject_zero_out_is_the_grouped_norm():
    rng = np.random.default_rng(62)
    x = rng.normal(0, 2, (2, 384)).astype(np.float32)
    logit = rng.normal(0, 3, (2, 3)).astype(np.float32)
    w = wl.norm_weight(0, 3, 384)
    xn, x_new = oracle.inject_rmsnorm_groups_f16(x, np.zeros((2, 128), np.float32), logit, w, 3)
    ref, _ = oracle.rmsnorm_groups_f16(x, w, 3)
    assert np.array_equal(x_new, x.astype(np.float64)) and np.array_equal(xn, ref)


def test_inject_weight_closed_forms_per_stream():
    """Stream g of row r takes the logit of (r, g), divided by the stream count: with
    logit = groups * ln 3 the weight is 2 * 3/4 = 1.5; a large positive logit saturates at 2 and
    a large negative one at 0. Rows and streams get different logits (nb != groups), so a
    transposed index or a sign slip fails."""
    nb, groups, n = 2, 3, 64
    x = np.ones((nb, groups * n), np.float32)
    out = np.full((nb, n), 2.0, np.float32)
    out[1] = -4.0
    logit = np.array([[groups * math.log(3.0), 1e4, -1e4],
                      [0.0, groups * math.log(3.0), 1e4]], np.float32)
    _, x_new = oracle.inject_rmsnorm_groups_f16(x, out, logit, wl.f32_to_bf16_bits(np.ones(groups * n, np.float32)),
                                                groups)
    expect_w = [[2.0 / (1.0 + math.exp(-float(logit[0, 0]) / groups)), 2.0, 0.0],
                [1.0, 2.0 / (1.0 + math.exp(-float(logit[1, 1]) / groups)), 2.0]]
    assert expect_w[0][0] == pytest.approx(1.5, rel=1e-6)
    for r in range(nb):
        for g in range(groups):
            seg = x_new[r, g * n:(g + 1) * n]
            assert np.allclose(seg, 1.0 + float(out[r, 0]) * expect_w[r][g], rtol=1e-12, atol=1e-300), (r, g)
    # a positive logit weighs the output above 1, a negative one below
    _, hi = oracle.inject_rmsnorm_groups_f16(x[:1, :n], out[:1], np.array([[0.5]], np.float32),
                                             wl.f32_to_bf16_bits(np.ones(n, np.float32)), 1)
    assert hi[0, 0] > 1.0 + 2.0


def test_inject_is_linear_in_out_before_the_norm():
    rng = np.random.default_rng(63)
    nb, groups, n = 2, 2, 128
    x = rng.normal(0, 1, (nb, groups * n)).astype(np.float32)
    o1 = rng.integers(-4, 5, (nb, n)).astype(np.float32)
    logit = rng.normal(0, 2, (nb, groups)).astype(np.float32)
    w = wl.norm_weight(0, 4, groups * n)
    _, a = oracle.inject_rmsnorm_groups_f16(x, o1, logit, w, groups)
    _, b2 = oracle.inject_rmsnorm_groups_f16(x, 2 * o1, logit, w, groups)
    assert np.allclose(b2 - x, 2 * (a - x), rtol=1e-12, atol=1e-12)


# ---- derived low-bit codes ([BATCH_MSL] fn_q2_rows_h, fn_q3_rows_h) ----------------------


def _golden_lowbit_row(golden):
    g = golden("lowbit_layout.txt")
    codes = np.zeros((1, 64), np.uint8)
    for item in g["codes"]:
        e, v = item.split("=")
        codes[0, int(e)] = int(v)
    w2 = np.array([int(v, 16) for v in g["w2_words"]], np.uint32)
    lo = np.array([int(v, 16) for v in g["lo_words"]], np.uint32)
    return codes, w2, lo


def test_lowbit_layout_hand_worked(golden):
    codes, w2_words, lo_words = _golden_lowbit_row(golden)
    w2 = oracle.lowbit_pack2(codes)
    lo = oracle.lowbit_pack3lo(codes)
    assert np.array_equal(w2.view("<u4").ravel(), w2_words)
    assert np.array_equal(lo.view("<u4").ravel(), lo_words)
    assert np.array_equal(oracle.lowbit_codes(w2), codes >> 2)
    assert np.array_equal(oracle.lowbit_codes(w2, lo), codes >> 1)


def test_lowbit_codes_are_the_shifted_4bit_codes():
    rng = np.random.default_rng(41)
    codes = rng.integers(0, 16, (7, 192), dtype=np.uint8)
    w2, lo = oracle.lowbit_pack2(codes), oracle.lowbit_pack3lo(codes)
    assert np.array_equal(oracle.lowbit_codes(w2), codes >> 2)
    assert np.array_equal(oracle.lowbit_codes(w2, lo), codes >> 1)
    # every code lands in exactly one field: packing a single nonzero code sets one field
    one = np.zeros((1, 64), np.uint8)
    for e in range(64):
        one[:] = 0
        one[0, e] = 12
        bits = np.unpackbits(oracle.lowbit_pack2(one)).sum()
        assert bits == 2 and np.unpackbits(oracle.lowbit_pack3lo(one)).sum() == 0


def _lowbit_case(seed, rows, in_dim, nb):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, (rows, in_dim), dtype=np.uint8)
    s = wl.f32_to_bf16_bits(np.abs(rng.normal(0, 0.02, (rows, in_dim // 64))).astype(np.float32))
    b = wl.f32_to_bf16_bits((-8 * rng.normal(0, 0.01, (rows, in_dim // 64))).astype(np.float32))
    x = wl.f16_bits(rng.normal(0, 1, (nb, in_dim)))
    return codes, s, b, x


def test_lowbit_gemv_is_the_quad_midpoint_of_the_4bit_product():
    """w2 = (4 q2 + 1.5) s + b is the mean of the four 4-bit weights s q4 + b sharing q2,
    and w3 = (2 q3 + 0.5) s + b the mean of the two sharing q3: the low-bit products are the
    means of 4-bit products (the pinned 4-bit oracle) over the codes of each quad / pair."""
    codes, s, b, x = _lowbit_case(42, 9, 128, 3)
    y2, _ = oracle.gemv_lowbit(oracle.lowbit_pack2(codes), None, s, b, x)
    quads = [oracle.gemv(oracle.pack(((codes >> 2) << 2) + k), s, b, x)[0] for k in range(4)]
    np.testing.assert_allclose(y2, sum(quads) / 4, rtol=1e-12, atol=1e-12)
    y3, _ = oracle.gemv_lowbit(oracle.lowbit_pack2(codes), oracle.lowbit_pack3lo(codes), s, b, x)
    pairs = [oracle.gemv(oracle.pack(((codes >> 1) << 1) + k), s, b, x)[0] for k in range(2)]
    np.testing.assert_allclose(y3, sum(pairs) / 2, rtol=1e-12, atol=1e-12)


def test_lowbit_gemv_brute_force_tiny():
    codes, s, b, x = _lowbit_case(43, 3, 64, 2)
    sf, bf = wl.bf16_bits_to_f32(s).astype(float), wl.bf16_bits_to_f32(b).astype(float)
    xf = x.view(np.float16).astype(float)
    for bits in (2, 3):
        w2 = oracle.lowbit_pack2(codes)
        lo = oracle.lowbit_pack3lo(codes) if bits == 3 else None
        y, bound = oracle.gemv_lowbit(w2, lo, s, b, x)
        for r in range(2):
            for o in range(3):
                acc = 0.0
                for i in range(64):
                    q = int(codes[o, i])
                    w = (4 * (q >> 2) + 1.5) * sf[o, 0] + bf[o, 0] if bits == 2 else \
                        (2 * (q >> 1) + 0.5) * sf[o, 0] + bf[o, 0]
                    acc += w * xf[r, i]
                assert abs(y[r, o] - acc) <= 1e-12 * (1 + abs(acc))
        assert np.all(bound > 0)


def _lowbit_bank(seed, n_exp, out_dim, in_dim):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(n_exp * out_dim, in_dim), dtype=np.uint8)
    s = wl.f32_to_bf16_bits(np.abs(rng.normal(0, 0.02, (n_exp * out_dim, in_dim // 64))).astype(np.float32))
    b = wl.f32_to_bf16_bits((-8 * rng.normal(0, 0.01, (n_exp * out_dim, in_dim // 64))).astype(np.float32))
    return codes, s, b


def test_experts_lowbit_equal_the_dense_lowbit_product_per_expert():
    """Routed low-bit experts (fn_expert_qmm's contraction, routed) reduce to the pinned dense
    low-bit product of each expert's matrix over its rows (identical arithmetic), for 2- and
    3-bit codes, with a token map, an empty segment and a repeated expert."""
    n_exp, out_dim, in_dim = 3, 5, 128
    codes, s, b = _lowbit_bank(71, n_exp, out_dim, in_dim)
    x = wl.f16_bits(np.random.default_rng(72).normal(0, 1, (4, in_dim)))
    ids = np.array([2, 0, 1, 2], np.int32)
    offs = np.array([0, 2, 2, 5, 6], np.int32)
    x_rows = np.array([3, 0, 1, 1, 2, 0], np.int32)
    for bits in (2, 3):
        w2 = oracle.lowbit_pack2(codes)
        lo = oracle.lowbit_pack3lo(codes) if bits == 3 else None
        y, bound = oracle.experts_lowbit(w2, lo, s, b, x, x_rows, ids, offs, n_exp, out_dim)
        for a, e in enumerate(ids):
            rows = slice(e * out_dim, (e + 1) * out_dim)
            r0, r1 = offs[a], offs[a + 1]
            if r0 == r1:
                continue
            ref, rb = oracle.gemv_lowbit(w2[rows], None if lo is None else lo[rows], s[rows], b[rows],
                                         x[x_rows[r0:r1]])
            assert np.array_equal(y[r0:r1], ref) and np.array_equal(bound[r0:r1], rb), (bits, a)


def test_experts_lowbit_fp32_activations_as_given():
    """fp32 activations that binary16 represents exactly give the same products as their
    binary16 bits; values binary16 cannot hold enter exactly (checked against numpy)."""
    n_exp, out_dim, in_dim = 2, 4, 192
    codes, s, b = _lowbit_bank(73, n_exp, out_dim, in_dim)
    xh = wl.f16_bits(np.random.default_rng(74).normal(0, 1, (3, in_dim)))
    x32 = xh.view(np.float16).astype(np.float32)
    ids, offs = np.array([1, 0], np.int32), np.array([0, 1, 3], np.int32)
    w2, lo = oracle.lowbit_pack2(codes), oracle.lowbit_pack3lo(codes)
    for low in (None, lo):
        a, _ = oracle.experts_lowbit(w2, low, s, b, x32, None, ids, offs, n_exp, out_dim)
        h, _ = oracle.experts_lowbit(w2, low, s, b, xh, None, ids, offs, n_exp, out_dim)
        assert np.array_equal(a, h)
    xf = (np.random.default_rng(75).normal(0, 1, (3, in_dim)) * 1.000001).astype(np.float32)
    y, _ = oracle.experts_lowbit(w2, None, s, b, xf, None, ids, offs, n_exp, out_dim)
    q2 = oracle.lowbit_codes(w2).astype(np.float64)
    sf = np.repeat(wl.bf16_bits_to_f32(s).astype(np.float64), 64, axis=1)
    bf = np.repeat(wl.bf16_bits_to_f32(b).astype(np.float64), 64, axis=1)
    w = sf * (4.0 * q2 + 1.5) + bf
    ref = np.vstack([xf[0:1].astype(np.float64) @ w[4:8].T, xf[1:3].astype(np.float64) @ w[0:4].T])
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_experts_lowbit_brute_force_and_invalid_id():
    n_exp, out_dim, in_dim = 2, 2, 64
    codes, s, b = _lowbit_bank(76, n_exp, out_dim, in_dim)
    xf = np.random.default_rng(77).normal(0, 1, (2, in_dim)).astype(np.float32)
    sf, bfv = wl.bf16_bits_to_f32(s).astype(float), wl.bf16_bits_to_f32(b).astype(float)
    w2, lo = oracle.lowbit_pack2(codes), oracle.lowbit_pack3lo(codes)
    ids, offs = np.array([1, 5], np.int32), np.array([0, 1, 2], np.int32)   # expert 5 does not exist
    y, bound = oracle.experts_lowbit(w2, lo, s, b, xf, None, ids, offs, n_exp, out_dim)
    for o in range(out_dim):
        row = out_dim + o
        acc = sum(((2 * (int(codes[row, i]) >> 1) + 0.5) * sf[row, 0] + bfv[row, 0]) * float(xf[0, i])
                  for i in range(in_dim))
        assert abs(y[0, o] - acc) <= 1e-12 * (1 + abs(acc))
    assert np.all(np.isnan(y[1])) and np.all(np.isnan(bound[1]))


# ---- prefill helpers ([BATCH_MSL] fn_qmv_small_b; the min/max quantiser) -------------------


def test_quantize_hand_worked(golden):
    g = golden("quantize_ramp.txt")
    w = (np.arange(64, dtype=np.float32) * 0.25).reshape(1, 64)
    packed, s, b = oracle.quantize(w)
    assert int(s[0, 0]) == int(g["s"][0], 16) and int(b[0, 0]) == int(g["b"][0], 16)
    codes = oracle.unpack(packed, 64)[0]
    for item in g["codes"]:
        i, q = item.split("=")
        assert int(codes[int(i)]) == int(q), i


def test_quantize_exact_grid_and_constant_groups():
    k = np.tile(np.arange(16), 4)
    w = np.stack([-1.0 + 0.125 * k, np.full(64, 2.0), 3.0 + 0.5 * k[::-1]]).astype(np.float32)
    packed, s, b = oracle.quantize(w)
    codes = oracle.unpack(packed, 64)
    assert np.array_equal(codes[0], k) and s[0, 0] == 0x3E00 and b[0, 0] == 0xBF80   # 0.125, -1
    assert s[1, 0] == 0 and b[1, 0] == 0x4000 and not codes[1].any()                 # constant 2.0
    assert np.array_equal(codes[2], k[::-1]) and s[2, 0] == 0x3F00 and b[2, 0] == 0x4040


def test_quantize_reconstruction_error():
    rng = np.random.default_rng(51)
    w = rng.normal(0, 0.05, (9, 256)).astype(np.float32)
    packed, s, b = oracle.quantize(w)
    codes = oracle.unpack(packed, 256).astype(np.float64)
    sf = np.repeat(wl.bf16_bits_to_f32(s).astype(np.float64), 64, axis=1)
    bf = np.repeat(wl.bf16_bits_to_f32(b).astype(np.float64), 64, axis=1)
    err = np.abs(sf * codes + bf - w)
    # half a step, plus the bf16 rounding of the bias (below the minimum) and of the step
    gmin = np.repeat(w.reshape(9, 4, 64).min(axis=2), 64, axis=1)
    assert np.all(err <= 0.5 * sf + np.abs(bf - gmin) + 15 * sf * 2.0 ** -8 + 1e-7)
    assert np.all(codes[codes > 0] <= 15)


def test_gemv_f32x_matches_the_fp16_product_on_fp16_values():
    rng = np.random.default_rng(52)
    codes = rng.integers(0, 16, (5, 128), dtype=np.uint8)
    s = wl.f32_to_bf16_bits(np.abs(rng.normal(0, 0.02, (5, 2))).astype(np.float32))
    b = wl.f32_to_bf16_bits((-8 * rng.normal(0, 0.01, (5, 2))).astype(np.float32))
    x16 = wl.f16_bits(rng.normal(0, 1, (3, 128)))
    packed = oracle.pack(codes)
    y16, _ = oracle.gemv(packed, s, b, x16)
    y32, bound = oracle.gemv_f32x(packed, s, b, x16.view(np.float16).astype(np.float32))
    np.testing.assert_allclose(y32, y16, rtol=0, atol=1e-12)
    # brute force with fp32 activations that fp16 cannot hold
    x = rng.normal(0, 1, (2, 128)).astype(np.float32) * np.float32(1 + 2 ** -20)
    y, _ = oracle.gemv_f32x(packed, s, b, x)
    sf, bf = wl.bf16_bits_to_f32(s).astype(float), wl.bf16_bits_to_f32(b).astype(float)
    for r in range(2):
        for o in range(5):
            ref = sum((sf[o, i // 64] * codes[o, i] + bf[o, i // 64]) * float(x[r, i]) for i in range(128))
            assert abs(y[r, o] - ref) <= 1e-12 * (1 + abs(ref))


def test_quantize_zero_minimum_is_positive_zero():
    w = np.zeros((2, 64), np.float32)
    w[0, 5] = 1.5
    w[1, :] = -0.0
    w[1, 7] = 3.0
    _, s, b = oracle.quantize(w)
    assert b[0, 0] == 0 and b[1, 0] == 0 and s[0, 0] == 0x3DCD and s[1, 0] == 0x3E4D

