"""GPU parity of the derived low-bit codes ("BATCH_MSL" constant page, quantized_rows.metal
fn_q2_rows_h and fn_q3_rows_h) against the CPU oracle, through the C ABI.

q4a_lowbit_pack is integer work: bit-exact. q4a_gemv_lowbit: every element within the
oracle's bound |y - y_ref| <= 2e-3 * sum_i |w_oi x_ri| + 1e-5, every output written (NaN
sentinel). The kernel reads each code exactly (binary16 subnormals), scales activations by
powers of two, and carries the bias and reconstruction-offset terms with ~16-bit hi/lo sums:
its error is fp32 accumulation plus ~2^-16 of the offset terms, far inside the bound.
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


def case(out_dim, in_dim, nb, seed):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(out_dim, in_dim), dtype=np.uint8)
    s = wl.f32_to_bf16_bits(np.abs(rng.normal(0, 0.02, (out_dim, in_dim // 64))).astype(np.float32))
    b = wl.f32_to_bf16_bits((-8 * rng.normal(0, 0.01, (out_dim, in_dim // 64))).astype(np.float32))
    x = wl.f16_bits(rng.normal(0, 1, (nb, in_dim)))
    return codes, s, b, x


@pytest.mark.parametrize("rows,in_dim", [(1, 64), (300, 4096), (7, 640), (33, 12288)])
def test_lowbit_pack_bit_exact(rows, in_dim):
    codes, _, _, _ = case(rows, in_dim, 1, rows + in_dim)
    w4 = q4a.pack(dev(codes))
    w_up, w_lo = q4a.lowbit_pack(w4)
    torch.cuda.synchronize()
    assert np.array_equal(w_up.cpu().numpy(), oracle.lowbit_pack2(codes))
    assert np.array_equal(w_lo.cpu().numpy(), oracle.lowbit_pack3lo(codes))
    w_up2, none = q4a.lowbit_pack(w4, with_lowest=False)
    assert none is None and torch.equal(w_up2, w_up)


LOWBIT_CASES = [
    (256, 512, 1),      # the small single-GEMV shape
    (300, 1024, 4),     # ragged rows
    (77, 4096, 8),
    (33, 12288, 3),     # long rows: K split across a cluster
    (129, 2048, 16),    # NT = 2
    (40, 640, 2),       # 10 groups: scales fetched row block by row block
    (1000, 4096, 32),   # NT = 4
    (200, 512, 40),     # two activation segments
]


@pytest.mark.parametrize("bits", [2, 3])
@pytest.mark.parametrize("out_dim,in_dim,nb", LOWBIT_CASES)
def test_gemv_lowbit_matches_oracle(bits, out_dim, in_dim, nb):
    codes, s, b, x = case(out_dim, in_dim, nb, 7 * out_dim + in_dim + nb + bits)
    w_up = oracle.lowbit_pack2(codes)
    w_lo = oracle.lowbit_pack3lo(codes) if bits == 3 else None
    y = torch.full((nb, out_dim), float("nan"), dtype=torch.float32, device=DEV)
    q4a.gemv_lowbit(bits, dev(w_up), None if w_lo is None else dev(w_lo), dev(s), dev(b), dev(x), out=y)
    torch.cuda.synchronize()
    q4a.check_device_error()
    got = y.cpu().numpy().astype(np.float64)
    ref, bound = oracle.gemv_lowbit(w_up, w_lo, s, b, x)
    assert np.isfinite(got).all(), "non-finite output (unwritten or overflow)"
    worst = float((np.abs(got - ref) / bound).max())
    assert worst <= 1.0, f"{bits}-bit {out_dim}x{in_dim} nb={nb}: worst err/bound {worst:.3g}"


def test_gemv_lowbit_from_device_pack_and_determinism():
    """The full path: 4-bit codes packed, derived codes packed, both products, twice."""
    codes, s, b, x = case(513, 4096, 5, 91)
    w_up, w_lo = q4a.lowbit_pack(q4a.pack(dev(codes)))
    for bits in (2, 3):
        y1 = q4a.gemv_lowbit(bits, w_up, w_lo, dev(s), dev(b), dev(x))
        y2 = q4a.gemv_lowbit(bits, w_up, w_lo, dev(s), dev(b), dev(x))
        torch.cuda.synchronize()
        assert torch.equal(y1, y2)
        ref, bound = oracle.gemv_lowbit(oracle.lowbit_pack2(codes),
                                        oracle.lowbit_pack3lo(codes) if bits == 3 else None, s, b, x)
        assert float((np.abs(y1.cpu().numpy() - ref) / bound).max()) <= 1.0
