"""GPU parity of the decode-layer MLP entry point (q4a_decode_mlp) against the CPU oracle, and
of weight-writing kernels followed at once by a GEMV on the same stream.

q4a_decode_mlp chains RMSNorm -> gate|up with h = fp16(silu(g) * u) -> the down projection of
h ("BATCH_MSL" constant page, hyperconnection.metal fn_norm_prep_b, experts.metal
fn_moe_gate_up_b, fn_moe_act_b, fn_moe_down_b). Bars:
  * h against the oracle's gate|up products on the oracle's normalised input, with the bound
    of the fused gate|up tests (silu' <= 1.1 plus one rounding to binary16);
  * y against the oracle's down projection of the h the GPU produced (h is checked on its
    own above), with the GEMV bound 2e-3 * sum|w x| + 1e-5 per element.
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


def quant(rows, in_dim, seed):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(rows, in_dim), dtype=np.uint8)
    s = wl.f32_to_bf16_bits(np.abs(rng.normal(0, 0.02, (rows, in_dim // 64))).astype(np.float32))
    b = wl.f32_to_bf16_bits((-8 * rng.normal(0, 0.01, (rows, in_dim // 64))).astype(np.float32))
    return oracle.pack(codes), s, b


def check_h(h, gu, xn, inter, what):
    packed, s, b = gu
    y, bound = oracle.gemv(packed, s, b, xn)
    g, u, bg, bu = y[:, :inter], y[:, inter:], bound[:, :inter], bound[:, inter:]
    sg = g / (1.0 + np.exp(-g))
    ref = sg * u
    tol = 1.1 * (np.abs(u) + bu) * bg + (np.abs(sg) + 1.1 * bg) * bu + 2.0 ** -11 * np.abs(ref) + 2.0 ** -24
    assert np.isfinite(h).all(), f"{what}: non-finite h"
    worst = float((np.abs(h.astype(np.float64) - ref) / tol).max())
    assert worst <= 1.0, f"{what}: h worst err/bound {worst:.3g}"


def check_y(y, dn, h_bits, what):
    packed, s, b = dn
    ref, bound = oracle.gemv(packed, s, b, h_bits)
    assert np.isfinite(y).all(), f"{what}: non-finite y"
    worst = float((np.abs(y.astype(np.float64) - ref) / bound).max())
    assert worst <= 1.0, f"{what}: y worst err/bound {worst:.3g}"


def run_layer(hidden, inter, nb, seed, repeat=1):
    """One decode layer through q4a_decode_mlp, checked against the oracle."""
    gu = quant(2 * inter, hidden, seed)
    dn = quant(hidden, inter, seed + 1)
    a = wl.normal_f32(93, seed % 7, (nb, hidden)) * 2.0
    nw = wl.norm_weight(93, 1, hidden)
    args = [dev(t) for t in gu] + [dev(a), dev(nw)] + [dev(t) for t in dn]
    for _ in range(repeat):
        y = torch.full((nb, hidden), float("nan"), device=DEV)
        h = torch.full((nb, inter), float("nan"), dtype=torch.float16, device=DEV)
        q4a.decode_mlp(*args, eps=1e-6, out=y, h=h)
    torch.cuda.synchronize()
    q4a.check_device_error()
    xn, _ = oracle.rmsnorm_f16(a, nw, eps=1e-6)
    h_np = h.cpu().numpy()
    what = f"decode_mlp hidden={hidden} inter={inter} nb={nb}"
    check_h(h_np, gu, xn, inter, what)
    check_y(y.cpu().numpy(), dn, h_np.view(np.uint16), what)
    return y, h


@pytest.mark.parametrize("hidden,inter,nb", [(512, 128, 1), (1024, 640, 3), (2048, 1024, 8), (4096, 1024, 16),
                                             (512, 256, 32), (1024, 512, 5), (512, 1536, 2)])
def test_decode_mlp_matches_oracle(hidden, inter, nb):
    """Shapes from 512 to 4096 inputs, 1 to 32 activation rows."""
    run_layer(hidden, inter, nb, hidden + inter + nb)


def test_decode_mlp_full_size():
    """The dense decode layer of the workloads: 4096 -> 2 x 6144 -> 4096 at NB 1, 8 and 16."""
    for nb in (1, 8, 16):
        run_layer(4096, 6144, nb, 7 + nb)


def test_decode_mlp_back_to_back():
    """Several calls on one stream with no sync between them (each launch overlaps the tail of
    the one before under programmatic dependent launch)."""
    run_layer(2048, 1024, 4, 21, repeat=6)


def test_pack_then_gemv_without_a_sync():
    """q4a_pack writes the weights and q4a_gemv reads them right behind it on the same stream
    (the GEMV starts under programmatic dependent launch; its weight loads wait for the
    previous kernel to complete)."""
    c = wl.DENSE_GATE_UP_CASE
    qm = wl.quant_matrix(c.config_id, c.out_dim, c.in_dim)
    x = wl.dense_x(c, 2)
    codes, s, b, xd = dev(qm.codes), dev(qm.scale), dev(qm.bias), dev(x)
    w = torch.zeros((c.out_dim, c.in_dim // 2), dtype=torch.uint8, device=DEV)
    torch.cuda.synchronize()
    ys = []
    for _ in range(3):
        w.zero_()
        q4a.pack(codes, out=w)
        ys.append(q4a.gemv(w, s, b, xd))
    torch.cuda.synchronize()
    q4a.check_device_error()
    ref, bound = oracle.gemv(oracle.pack(qm.codes), qm.scale, qm.bias, x)
    for y in ys:
        worst = float((np.abs(y.cpu().numpy().astype(np.float64) - ref) / bound).max())
        assert worst <= 1.0, f"pack -> gemv: worst err/bound {worst:.3g}"


def test_quantize_then_gemv_without_a_sync():
    """q4a_quantize writes codes, scales and biases; q4a_gemv (and the tensor-core path at a
    wide batch) reads them right behind it on the same stream."""
    rows, in_dim = 4096, 4096
    wf = (np.random.default_rng(5).normal(0, 0.05, (rows, in_dim))).astype(np.float32)
    packed_ref, s_ref, b_ref = oracle.quantize(wf)
    wd = dev(wf)
    for nb in (4, 64):
        x = wl.f16_bits(np.random.default_rng(nb).normal(0, 1, (nb, in_dim)))
        xd = dev(x)
        torch.cuda.synchronize()
        packed, s, b = q4a.quantize(wd)
        y = q4a.gemv(packed, s, b, xd)
        torch.cuda.synchronize()
        q4a.check_device_error()
        ref, bound = oracle.gemv(packed_ref, s_ref, b_ref, x)
        worst = float((np.abs(y.cpu().numpy().astype(np.float64) - ref) / bound).max())
        assert worst <= 1.0, f"quantize -> gemv nb={nb}: worst err/bound {worst:.3g}"
