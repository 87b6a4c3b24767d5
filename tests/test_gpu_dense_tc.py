"""GPU parity of the wide-batch dense path of q4a_gemv (NB >= 64: binary16 weights in TMEM,
tcgen05.mma with TMEM accumulators) against the CPU oracle, through the C ABI.

Bar: every element within the oracle's bound |y - y_ref| <= 2e-3 * sum_i |w_oi x_ri| + 1e-5,
every output written (NaN sentinel). The path rounds each weight once to binary16 after a
per-row power-of-two rescale, so its error is at most 2^-11 * sum_i |w_oi x_ri| plus fp32
accumulation: a quarter of the bound.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import affine_q4_dequant_gb300 as q4a  # noqa: E402
import oracle  # noqa: E402
import q4a_workloads as wl  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(DEV)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def case(out_dim, in_dim, nb, seed):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(out_dim, in_dim), dtype=np.uint8)
    s = wl.f32_to_bf16_bits(np.abs(rng.normal(0, 0.02, (out_dim, in_dim // 64))).astype(np.float32))
    b = wl.f32_to_bf16_bits((-8 * rng.normal(0, 0.01, (out_dim, in_dim // 64))).astype(np.float32))
    x = wl.f16_bits(rng.normal(0, 1, (nb, in_dim)))
    return oracle.pack(codes), s, b, x


def gemv(packed, s, b, x, out_dim, s_dev=None, b_dev=None):
    y = torch.full((x.shape[0], out_dim), float("nan"), dtype=torch.float32, device=DEV)
    q4a.gemv(dev(packed), dev(s) if s_dev is None else s_dev, dev(b) if b_dev is None else b_dev, dev(x), out=y)
    torch.cuda.synchronize()
    q4a.check_device_error()
    return host(y)


def check(y, y_ref, bound, what):
    assert y.shape == y_ref.shape, what
    assert np.isfinite(y).all(), f"{what}: non-finite output (unwritten or overflow)"
    ratio = np.abs(y.astype(np.float64) - y_ref) / bound
    worst = float(ratio.max())
    assert worst <= 1.0, f"{what}: worst err/bound {worst:.3g} at {np.unravel_index(ratio.argmax(), ratio.shape)}"
    return worst


TC_CASES = [
    (256, 512, 64),      # one work unit, N 64
    (300, 512, 65),      # ragged rows (second 128-row tile partly outside), N padded to 80
    (129, 512, 100),     # second tile holds one row
    (513, 1024, 128),    # three units, N 128
    (1000, 4096, 80),    # long K (64 groups, 16 code stages)
    (256, 1024, 256),    # two launches of 128 activation rows
    (70, 512, 300),      # three launches: 128, 128, then 44 rows
    (40000, 512, 64),    # 157 units: CTAs take a second unit
    (1100, 512, 64),     # last unit's second tile starts beyond out_dim (its y box is not stored)
    (384, 2048, 96),     # one accumulator set: y boxes of 32 columns, 96 = 3 x 32
]


@pytest.mark.parametrize("out_dim,in_dim,nb", TC_CASES)
def test_dense_tc_matches_oracle(out_dim, in_dim, nb):
    packed, s, b, x = case(out_dim, in_dim, nb, out_dim * 3 + in_dim + nb)
    y = gemv(packed, s, b, x, out_dim)
    y_ref, bound = oracle.gemv(packed, s, b, x)
    check(y, y_ref, bound, f"dense_tc {out_dim}x{in_dim} nb={nb}")


def test_dense_tc_row_scale_range():
    """Rows whose scales and biases span 2^-40 .. 2^40 (a per-row rescale keeps every
    binary16 weight normal), all-zero rows, and a row with one dominant group."""
    packed, s, b, x = case(300, 1024, 64, 11)
    sf, bf = wl.bf16_bits_to_f32(s).astype(np.float64), wl.bf16_bits_to_f32(b).astype(np.float64)
    k = np.linspace(-40, 40, 300).round()[:, None]
    sf, bf = sf * 2.0 ** k, bf * 2.0 ** k
    sf[7], bf[7] = 0.0, 0.0
    sf[8, 3] *= 2.0 ** 12
    s2 = wl.f32_to_bf16_bits(sf.astype(np.float32))
    b2 = wl.f32_to_bf16_bits(bf.astype(np.float32))
    y = gemv(packed, s2, b2, x, 300)
    y_ref, bound = oracle.gemv(packed, s2, b2, x)
    check(y, y_ref, bound, "row scale range")
    assert np.all(y[:, 7] == 0.0)


def test_dense_tc_nonfinite_scales_are_loud():
    packed, s, b, x = case(256, 512, 64, 12)
    s = s.copy()
    s[3, 2] = 0x7FC0    # NaN
    s[9, 0] = 0x7F80    # +inf
    y = torch.zeros((64, 256), dtype=torch.float32, device=DEV)
    q4a.gemv(dev(packed), dev(s), dev(b), dev(x), out=y)
    y = host(y)
    assert not np.isfinite(y[:, 3]).any() and not np.isfinite(y[:, 9]).any()
    y_ref, bound = oracle.gemv(packed, s, b, x)
    keep = np.ones(256, bool)
    keep[[3, 9]] = False
    check(y[:, keep], y_ref[:, keep], bound[:, keep], "finite rows next to non-finite ones")


def test_dense_tc_is_deterministic():
    packed, s, b, x = case(513, 1024, 96, 13)
    y1 = gemv(packed, s, b, x, 513)
    y2 = gemv(packed, s, b, x, 513)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_wide_batch_falls_back_when_ineligible():
    """Scales not 16-byte aligned, or a group count that is not a multiple of 8: the
    wide batch runs on the mma.sync GEMV kernel instead, with the same bar."""
    packed, s, b, x = case(200, 512, 64, 14)
    buf_s = torch.empty(s.size + 8, dtype=torch.int16, device=DEV)
    buf_b = torch.empty(b.size + 8, dtype=torch.int16, device=DEV)
    s_dev = buf_s[1:1 + s.size].view(s.shape)
    b_dev = buf_b[1:1 + b.size].view(b.shape)
    s_dev.copy_(dev(s))
    b_dev.copy_(dev(b))
    y = gemv(packed, s, b, x, 200, s_dev=s_dev, b_dev=b_dev)
    y_ref, bound = oracle.gemv(packed, s, b, x)
    check(y, y_ref, bound, "misaligned scales")
    packed, s, b, x = case(100, 576, 64, 15)   # 9 groups
    y = gemv(packed, s, b, x, 100)
    y_ref, bound = oracle.gemv(packed, s, b, x)
    check(y, y_ref, bound, "9 groups")


def test_wide_batch_runs_on_the_tensor_core_kernel():
    """The routing a call takes (q4a_gemv_kernel_choice, the function the dispatch itself calls):
    NB 64 on a short matrix and NB 9 on a tall one run the tcgen05 kernel, NB 16 on a short
    matrix and NB 8 on a tall one the GEMV kernel; each result meets the oracle's bar."""
    packed, s, b, x = case(256, 512, 64, 16)
    sd, bd = dev(s), dev(b)
    assert q4a.gemv_kernel_choice(sd, bd, 64, 256, 512) == "tcgen05"
    assert q4a.gemv_kernel_choice(sd, bd, 16, 256, 512) == "gemv"
    y_ref, bound = oracle.gemv(packed, s, b, x)
    check(gemv(packed, s, b, x, 256, s_dev=sd, b_dev=bd), y_ref, bound, "NB 64 (tcgen05)")
    check(gemv(packed, s, b, x[:16], 256, s_dev=sd, b_dev=bd), y_ref[:16], bound[:16], "NB 16 (GEMV)")
    out_dim = 152 * 256
    packed, s, b, x = case(out_dim, 512, 9, 17)
    sd, bd = dev(s), dev(b)
    assert q4a.gemv_kernel_choice(sd, bd, 9, out_dim, 512) == "tcgen05"
    assert q4a.gemv_kernel_choice(sd, bd, 8, out_dim, 512) == "gemv"
    y_ref, bound = oracle.gemv(packed, s, b, x)
    check(gemv(packed, s, b, x, out_dim, s_dev=sd, b_dev=bd), y_ref, bound, "tall NB 9 (tcgen05)")
    check(gemv(packed, s, b, x[:8], out_dim, s_dev=sd, b_dev=bd), y_ref[:8], bound[:8], "tall NB 8 (GEMV)")
    # 48 units: from NB 17
    out_dim = 48 * 256
    packed, s, b, x = case(out_dim, 512, 17, 18)
    sd, bd = dev(s), dev(b)
    assert q4a.gemv_kernel_choice(sd, bd, 17, out_dim, 512) == "tcgen05"
    assert q4a.gemv_kernel_choice(sd, bd, 16, out_dim, 512) == "gemv"
    y_ref, bound = oracle.gemv(packed, s, b, x)
    check(gemv(packed, s, b, x, out_dim, s_dev=sd, b_dev=bd), y_ref, bound, "NB 17 on 48 units (tcgen05)")
    check(gemv(packed, s, b, x[:16], out_dim, s_dev=sd, b_dev=bd), y_ref[:16], bound[:16], "NB 16 on 48 units (GEMV)")
