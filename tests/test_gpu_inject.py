"""GPU parity of the hyper-connection injection prologue (q4a_gemv_inject_rmsnorm_grouped)
against the CPU oracle ("BATCH_MSL" constant page, hyperconnection.metal fn_inject_b and
fn_norm_prep_b with inject = 1), through the C ABI.

Bars:
  * y: the GEMV bound 2e-3 * sum|w x| + 1e-5 per element against the oracle's product of its
    own normalised input (as the grouped-RMSNorm tests: a binary16 rounding that lands on the
    other side of a boundary is far inside the bound);
  * x_new: the kernel forms x + out * wgt with one fp32 fused multiply-add and wgt from fp32
    expf (a few ulp), so |x_new - x'| <= 2^-20 * (|x| + |out * wgt|) + 2^-126 against the
    oracle's double x'.
"""

import math

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


def case(out_dim, in_dim, nb, groups, seed):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(out_dim, in_dim), dtype=np.uint8)
    s = wl.f32_to_bf16_bits(np.abs(rng.normal(0, 0.02, (out_dim, in_dim // 64))).astype(np.float32))
    b = wl.f32_to_bf16_bits((-8 * rng.normal(0, 0.01, (out_dim, in_dim // 64))).astype(np.float32))
    n = in_dim // groups
    x = (rng.normal(0, 1, (nb, in_dim)) * 2.0).astype(np.float32)
    x[:, :n] *= 30.0                                   # one loud stream
    out = rng.normal(0, 3, (nb, n)).astype(np.float32)
    logit = rng.normal(0, 4, (nb, groups)).astype(np.float32)
    nw = wl.norm_weight(79, seed % 5, in_dim)
    return oracle.pack(codes), s, b, x, out, logit, nw


def run(out_dim, in_dim, nb, groups, seed, want_x_new=True):
    packed, s, b, x, out, logit, nw = case(out_dim, in_dim, nb, groups, seed)
    y = torch.full((nb, out_dim), float("nan"), device=DEV)
    x_new = torch.full((nb, in_dim), float("nan"), device=DEV) if want_x_new else None
    q4a.gemv_inject_rmsnorm_grouped(dev(packed), dev(s), dev(b), dev(x), dev(out), dev(logit), dev(nw), groups,
                                    eps=1e-6, y=y, x_new=x_new, want_x_new=want_x_new)
    torch.cuda.synchronize()
    q4a.check_device_error()
    xn, xr = oracle.inject_rmsnorm_groups_f16(x, out, logit, nw, groups, eps=1e-6)
    y_ref, bound = oracle.gemv(packed, s, b, xn)
    what = f"inject {out_dim}x{in_dim} nb={nb} groups={groups}"
    yh = y.cpu().numpy().astype(np.float64)
    assert np.isfinite(yh).all(), f"{what}: non-finite y"
    worst = float((np.abs(yh - y_ref) / bound).max())
    assert worst <= 1.0, f"{what}: y worst err/bound {worst:.3g}"
    if want_x_new:
        n = in_dim // groups
        wgt = 2.0 / (1.0 + np.exp(-logit.astype(np.float64) / groups))
        term = np.abs(np.repeat(wgt, n, axis=1) * np.tile(out.astype(np.float64), (1, groups)))
        tol = 2.0 ** -20 * (np.abs(x) + term) + 2.0 ** -126
        xg = x_new.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(xg - xr) <= tol), f"{what}: x_new off by {np.abs(xg - xr).max():.3g}"
    return y


@pytest.mark.parametrize("out_dim,in_dim,nb,groups", [(256, 512, 1, 2), (300, 1024, 4, 2), (77, 4096, 16, 4),
                                                      (40, 512, 1, 8), (33, 12288, 3, 3), (129, 2048, 9, 1),
                                                      (64, 1024, 32, 4)])
def test_inject_matches_oracle(out_dim, in_dim, nb, groups):
    """Single-CTA and cluster K-split layouts (12288 inputs), ragged row counts, 1..8 streams."""
    run(out_dim, in_dim, nb, groups, out_dim + in_dim + nb + groups)


def test_inject_without_x_new_gives_the_same_y():
    a = run(300, 1024, 4, 2, 5, want_x_new=True)
    b = run(300, 1024, 4, 2, 5, want_x_new=False)
    assert torch.equal(a, b)


def test_zero_logit_injection_equals_grouped_norm_of_the_sum():
    """2 sigmoid(0) = 1: the same y as q4a_gemv_rmsnorm_grouped on x + out (exact in fp32 for
    these small integers), bit for bit."""
    out_dim, in_dim, nb, groups = 128, 1024, 2, 4
    rng = np.random.default_rng(9)
    packed = oracle.pack(rng.integers(0, 16, (out_dim, in_dim), dtype=np.uint8))
    s = wl.f32_to_bf16_bits(np.abs(rng.normal(0, 0.02, (out_dim, in_dim // 64))).astype(np.float32))
    b = wl.f32_to_bf16_bits((-8 * rng.normal(0, 0.01, (out_dim, in_dim // 64))).astype(np.float32))
    x = rng.integers(-8, 9, (nb, in_dim)).astype(np.float32)
    out = rng.integers(-8, 9, (nb, in_dim // groups)).astype(np.float32)
    nw = wl.norm_weight(80, 0, in_dim)
    y1, xn1 = q4a.gemv_inject_rmsnorm_grouped(dev(packed), dev(s), dev(b), dev(x), dev(out),
                                              torch.zeros((nb, groups), device=DEV), dev(nw), groups)
    y2 = q4a.gemv_rmsnorm_grouped(dev(packed), dev(s), dev(b), dev(x + np.tile(out, (1, groups))), dev(nw), groups)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert np.array_equal(xn1.cpu().numpy(), x + np.tile(out, (1, groups)))
    assert math.isclose(float(2.0 / (1.0 + math.exp(0.0))), 1.0)
