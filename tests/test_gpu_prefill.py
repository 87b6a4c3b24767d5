"""GPU parity of the prefill helpers against the CPU oracle, through the C ABI.

q4a_quantize is integer work decided in binary32 on both sides: bit-exact codes, scales and
biases. q4a_gemv_f32x ("BATCH_MSL" constant page, hyperconnection.metal fn_qmv_small_b):
every element within the oracle's bound |y - y_ref| <= 2e-3 * sum_i |w_oi x_ri| + 1e-5
(fp32 accumulation of exact products is far inside it), every output written.
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


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("rows,in_dim", [(3, 64), (100, 4096), (7, 640)])
def test_quantize_bit_exact(rows, in_dim):
    rng = np.random.default_rng(rows + in_dim)
    w = (rng.normal(0, 1, (rows, in_dim)) * np.exp(rng.normal(0, 2, (rows, 1)))).astype(np.float32)
    w[0, :64] = 2.0                       # a constant group (s = 0)
    w[-1, -64:] = -0.3                    # a constant group whose bias rounds (s > 0, tiny)
    packed, s, b = q4a.quantize(dev(w))
    torch.cuda.synchronize()
    p_ref, s_ref, b_ref = oracle.quantize(w)
    assert np.array_equal(packed.cpu().numpy(), p_ref)
    assert np.array_equal(bits16(s), s_ref)
    assert np.array_equal(bits16(b), b_ref)


def test_quantize_signed_zero_minimum():
    w = np.abs(np.random.default_rng(3).normal(0, 1, (3, 128))).astype(np.float32)
    w[0, :64:2] = -0.0                    # minimum -0 and +0 in one group
    w[1, 64:] = 0.0
    w[2, 3] = -0.0
    packed, s, b = q4a.quantize(dev(w))
    p_ref, s_ref, b_ref = oracle.quantize(w)
    assert np.array_equal(packed.cpu().numpy(), p_ref)
    assert np.array_equal(bits16(s), s_ref) and np.array_equal(bits16(b), b_ref)


@pytest.mark.parametrize("out_dim,in_dim,nb", [(64, 4096, 1), (16, 2048, 7), (3, 640, 33), (256, 512, 128),
                                               (5, 12288, 2)])
def test_gemv_f32x_matches_oracle(out_dim, in_dim, nb):
    rng = np.random.default_rng(out_dim * 7 + nb)
    codes = rng.integers(0, 16, (out_dim, in_dim), dtype=np.uint8)
    s = wl.f32_to_bf16_bits(np.abs(rng.normal(0, 0.02, (out_dim, in_dim // 64))).astype(np.float32))
    b = wl.f32_to_bf16_bits((-8 * rng.normal(0, 0.01, (out_dim, in_dim // 64))).astype(np.float32))
    x = rng.normal(0, 1, (nb, in_dim)).astype(np.float32)
    packed = oracle.pack(codes)
    y = torch.full((nb, out_dim), float("nan"), dtype=torch.float32, device=DEV)
    q4a.gemv_f32x(dev(packed), dev(s), dev(b), dev(x), out=y)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    ref, bound = oracle.gemv_f32x(packed, s, b, x)
    assert np.isfinite(got).all()
    worst = float((np.abs(got - ref) / bound).max())
    assert worst <= 1.0, f"f32x {out_dim}x{in_dim} nb={nb}: worst err/bound {worst:.3g}"


def test_quantize_then_project():
    """Float weights quantised on the device, then the fp32-activation projection; both
    against the oracle, and bitwise repeatable."""
    rng = np.random.default_rng(77)
    w = rng.normal(0, 0.05, (40, 1024)).astype(np.float32)
    x = rng.normal(0, 1, (9, 1024)).astype(np.float32)
    packed, s, b = q4a.quantize(dev(w))
    y1 = q4a.gemv_f32x(packed, s, b, dev(x))
    y2 = q4a.gemv_f32x(packed, s, b, dev(x))
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    p_ref, s_ref, b_ref = oracle.quantize(w)
    ref, bound = oracle.gemv_f32x(p_ref, s_ref, b_ref, x)
    assert float((np.abs(y1.cpu().numpy() - ref) / bound).max()) <= 1.0
