"""GPU parity of q4a_gemv_silu (the GEMV with the silu(y / div) epilogue) against the CPU
oracle, on both kernels (NB < 64: mma.sync GEMV; NB >= 64: tensor-core path).

Bar: the product is within the GEMV bound B = 2e-3 sum|w x| + 1e-5; silu is 1.0999-Lipschitz,
so silu(y/div) moves by at most 1.1 B / |div|; the fp32 evaluation (one division, expf, one
more division) adds a few ulp: |out - ref| <= 1.1 B / |div| + 2^-21 |ref| + 1e-30.
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


@pytest.mark.parametrize("out_dim,in_dim,nb,div", [(256, 512, 1, 1.0), (300, 1024, 9, -0.5), (129, 4096, 33, 3.7),
                                                   (513, 1024, 64, 0.25), (200, 512, 100, -2.0),
                                                   (40, 12288, 4, 1.5),
                                                   (300, 512, 128, 0.5),      # tensor cores, 32-column y boxes
                                                   (152 * 256, 512, 9, 2.0)])  # tall: tensor cores from NB 9
def test_gemv_silu_matches_oracle(out_dim, in_dim, nb, div):
    rng = np.random.default_rng(out_dim + nb)
    codes = rng.integers(0, 16, size=(out_dim, in_dim), dtype=np.uint8)
    s = wl.f32_to_bf16_bits(np.abs(rng.normal(0, 0.02, (out_dim, in_dim // 64))).astype(np.float32))
    b = wl.f32_to_bf16_bits((-8 * rng.normal(0, 0.01, (out_dim, in_dim // 64))).astype(np.float32))
    x = wl.f16_bits(rng.normal(0, 1, (nb, in_dim)))
    packed = oracle.pack(codes)
    y = torch.full((nb, out_dim), float("nan"), dtype=torch.float32, device=DEV)
    q4a.gemv_silu(dev(packed), dev(s), dev(b), dev(x), div, out=y)
    torch.cuda.synchronize()
    q4a.check_device_error()
    got = y.cpu().numpy().astype(np.float64)
    ref, _, bound = oracle.gemv_silu(packed, s, b, x, div)
    assert np.isfinite(got).all()
    tol = 1.1 * bound / abs(div) + 2.0 ** -21 * np.abs(ref) + 1e-30
    worst = float((np.abs(got - ref) / tol).max())
    assert worst <= 1.0, f"worst err/bound {worst:.3g}"
