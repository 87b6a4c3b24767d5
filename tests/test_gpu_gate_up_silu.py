"""GPU parity of the fused gate|up projection with the SiLU*up epilogue ("BATCH_MSL" constant
page, experts.metal fn_moe_gate_up_b then fn_moe_act_b) against the CPU oracle, through the
C ABI: h = fp16(silu(g) * u) with g, u the gate and up rows of one product.

Bar, from the oracle's bounds bg, bu on g and u (2e-3 * sum|w x| + 1e-5 each): silu has
slope at most 1.1, so
    |h - h_ref| <= 1.1 (|u| + bu) bg + (|silu(g)| + 1.1 bg) bu + 2^-11 |h_ref| + 2^-24,
the last two terms the single rounding to binary16 (normal and subnormal range).
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


def case(inter, in_dim, seed):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(2 * inter, in_dim), dtype=np.uint8)
    s = wl.f32_to_bf16_bits(np.abs(rng.normal(0, 0.02, (2 * inter, in_dim // 64))).astype(np.float32))
    b = wl.f32_to_bf16_bits((-8 * rng.normal(0, 0.01, (2 * inter, in_dim // 64))).astype(np.float32))
    return oracle.pack(codes), s, b


def check(h_dev, packed, s, b, xn, inter, what):
    h = h_dev.cpu().numpy().astype(np.float64)
    y, bound = oracle.gemv(packed, s, b, xn)
    g, u = y[:, :inter], y[:, inter:]
    bg, bu = bound[:, :inter], bound[:, inter:]
    sg = g / (1.0 + np.exp(-g))
    ref = sg * u
    tol = 1.1 * (np.abs(u) + bu) * bg + (np.abs(sg) + 1.1 * bg) * bu + 2.0 ** -11 * np.abs(ref) + 2.0 ** -24
    assert np.isfinite(h).all(), f"{what}: non-finite output"
    worst = float((np.abs(h - ref) / tol).max())
    assert worst <= 1.0, f"{what}: worst err/bound {worst:.3g}"


@pytest.mark.parametrize("inter,in_dim,nb", [(128, 512, 1), (1024, 4096, 4), (640, 2048, 16), (48, 12288, 3),
                                             (256, 1024, 32), (64, 512, 40)])
def test_gate_up_silu_matches_oracle(inter, in_dim, nb):
    packed, s, b = case(inter, in_dim, inter + in_dim + nb)
    x = wl.f16_bits(np.random.default_rng(nb).normal(0, 1, (nb, in_dim)))
    h = torch.full((nb, inter), float("nan"), dtype=torch.float16, device=DEV)
    q4a.gemv_gate_up_silu(dev(packed), dev(s), dev(b), dev(x), out=h)
    torch.cuda.synchronize()
    q4a.check_device_error()
    check(h, packed, s, b, x, inter, f"gate_up_silu {inter}x{in_dim} nb={nb}")


@pytest.mark.parametrize("inter,in_dim,nb", [(1024, 4096, 1), (512, 4096, 8), (96, 12288, 16), (640, 2048, 32)])
def test_rmsnorm_gate_up_silu_matches_oracle(inter, in_dim, nb):
    packed, s, b = case(inter, in_dim, 3 * inter + in_dim + nb)
    a = wl.normal_f32(91, 0, (nb, in_dim)) * 3.0
    nw = wl.norm_weight(91, 1, in_dim)
    h = torch.full((nb, inter), float("nan"), dtype=torch.float16, device=DEV)
    q4a.gemv_rmsnorm_gate_up_silu(dev(packed), dev(s), dev(b), dev(a), dev(nw), eps=1e-6, out=h)
    torch.cuda.synchronize()
    q4a.check_device_error()
    xn, _ = oracle.rmsnorm_f16(a, nw, eps=1e-6)
    check(h, packed, s, b, xn, inter, f"rmsnorm_gate_up_silu {inter}x{in_dim} nb={nb}")


def test_gate_up_silu_equals_the_unfused_layer():
    """Same inputs through q4a_gemv + q4a_silu_mul_xsum: within the same bar."""
    inter, in_dim, nb = 512, 2048, 5
    packed, s, b = case(inter, in_dim, 5)
    x = wl.f16_bits(np.random.default_rng(6).normal(0, 1, (nb, in_dim)))
    h = q4a.gemv_gate_up_silu(dev(packed), dev(s), dev(b), dev(x))
    gu = q4a.gemv(dev(packed), dev(s), dev(b), dev(x))
    h2, _ = q4a.silu_mul_xsum(gu)
    torch.cuda.synchronize()
    d = (h.float() - h2.float()).abs().max().item()
    assert d <= 2e-3 * max(1.0, h2.float().abs().max().item())
    check(h, packed, s, b, x, inter, "fused")
