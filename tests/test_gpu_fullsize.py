"""GPU parity at the full workload sizes, in the launch configurations bench.py uses.

Inputs come from q4a_workloads (the seeded generators); every expected value comes
from the CPU oracle on the same inputs. Where the oracle cannot afford the whole
output (the LM head at large NB), it computes sampled entries one dot product each.
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


def host(t):
    return t.detach().cpu().numpy()


def check(y, y_ref, bound, what):
    assert y.shape == y_ref.shape, what
    assert np.isfinite(y).all(), f"{what}: non-finite output"
    ratio = np.abs(y.astype(np.float64) - y_ref) / bound
    worst = float(ratio.max())
    assert worst <= 1.0, f"{what}: worst err/bound {worst:.3g}"
    return worst


class Dense:
    """A packed matrix on the device, packed by q4a_pack and checked bit-exact."""

    def __init__(self, qm: wl.QuantMatrix):
        self.qm = qm
        self.packed = oracle.pack(qm.codes)
        self.w = q4a.pack(dev(qm.codes))
        assert np.array_equal(host(self.w), self.packed), "q4a_pack differs from the oracle"
        self.s = dev(qm.scale)
        self.b = dev(qm.bias)


@pytest.fixture(scope="module")
def gate_up():
    c = wl.DENSE_GATE_UP_CASE
    return Dense(wl.quant_matrix(c.config_id, c.out_dim, c.in_dim))


@pytest.fixture(scope="module")
def down():
    c = wl.DENSE_DOWN_CASE
    return Dense(wl.quant_matrix(c.config_id, c.out_dim, c.in_dim))


@pytest.mark.parametrize("nb", wl.DENSE_GATE_UP_CASE.nbs)
def test_gate_up_4096x12288(gate_up, nb):
    """x = fp16(RMSNorm(a)) with a ~ N(0,1), norm weight bf16(1 + N(0, 0.05)), eps 1e-6:
    the unfused GEMV on the oracle's normalised x, and the fused RMSNorm variant on a."""
    c = wl.DENSE_GATE_UP_CASE
    a = wl.normal_f32(c.config_id, wl.T_A, (nb, c.in_dim))
    nw = wl.norm_weight(c.config_id, wl.T_NORM_W, c.in_dim)
    xn, _ = oracle.rmsnorm_f16(a, nw, eps=1e-6)
    y_ref, bound = oracle.gemv(gate_up.packed, gate_up.qm.scale, gate_up.qm.bias, xn)
    y = host(q4a.gemv(gate_up.w, gate_up.s, gate_up.b, dev(xn)))
    check(y, y_ref, bound, f"gate_up nb={nb}")
    yf = host(q4a.gemv_rmsnorm(gate_up.w, gate_up.s, gate_up.b, dev(a), dev(nw), eps=1e-6))
    check(yf, y_ref, bound, f"gate_up fused rmsnorm nb={nb}")
    # the decode layer's first half as bench.py runs it: RMSNorm prologue, silu(gate) * up
    # epilogue (rows [0, 6144) gate, [6144, 12288) up); bar as in test_gpu_gate_up_silu.py
    inter = c.out_dim // 2
    h = host(q4a.gemv_rmsnorm_gate_up_silu(gate_up.w, gate_up.s, gate_up.b, dev(a), dev(nw), eps=1e-6))
    g, u = y_ref[:, :inter], y_ref[:, inter:]
    bg, bu = bound[:, :inter], bound[:, inter:]
    sg = g / (1.0 + np.exp(-g))
    tol = 1.1 * (np.abs(u) + bu) * bg + (np.abs(sg) + 1.1 * bg) * bu + 2.0 ** -11 * np.abs(sg * u) + 2.0 ** -24
    check(h.astype(np.float64), sg * u, tol, f"gate_up fused rmsnorm + silu*up nb={nb}")
    q4a.check_device_error()


@pytest.mark.parametrize("nb,bits", [(1, 2), (8, 2), (1, 3), (8, 3)])
def test_gate_up_4096x12288_lowbit(gate_up, nb, bits):
    """The derived 2/3-bit codes of the gate|up weights (packed on the device from the 4-bit
    ones, bit-exact), the product against the oracle's."""
    c = wl.DENSE_GATE_UP_CASE
    x = wl.normal_f16(c.config_id, wl.T_X, (nb, c.in_dim))
    w_up, w_lo = q4a.lowbit_pack(gate_up.w)
    ref_up = oracle.lowbit_pack2(gate_up.qm.codes)
    ref_lo = oracle.lowbit_pack3lo(gate_up.qm.codes) if bits == 3 else None
    assert np.array_equal(host(w_up), ref_up)
    if bits == 3:
        assert np.array_equal(host(w_lo), ref_lo)
    y = host(q4a.gemv_lowbit(bits, w_up, w_lo, gate_up.s, gate_up.b, dev(x)))
    y_ref, bound = oracle.gemv_lowbit(ref_up, ref_lo, gate_up.qm.scale, gate_up.qm.bias, x)
    check(y, y_ref, bound, f"gate_up {bits}-bit nb={nb}")
    q4a.check_device_error()


@pytest.mark.parametrize("nb", wl.DENSE_DOWN_CASE.nbs)
def test_down_12288x4096(down, nb):
    """x = fp16(silu(a) * b) with a, b ~ N(0,1) (the oracle's activation step)."""
    c = wl.DENSE_DOWN_CASE
    a = wl.normal_f32(c.config_id, wl.T_A, (nb, c.in_dim))
    b = wl.normal_f32(c.config_id, wl.T_B, (nb, c.in_dim))
    x = oracle.silu_mul_f16(np.concatenate([a, b], axis=1))
    y_ref, bound = oracle.gemv(down.packed, down.qm.scale, down.qm.bias, x)
    y = host(q4a.gemv(down.w, down.s, down.b, dev(x)))
    check(y, y_ref, bound, f"down nb={nb}")
    # the GPU activation step on the same a, b gives the same x within one binary16 ulp
    h, _ = q4a.silu_mul_xsum(dev(np.concatenate([a, b], axis=1)))
    hv = host(h).view(np.float16).astype(np.float64)
    rv = x.view(np.float16).astype(np.float64)
    assert np.all(np.abs(hv - rv) <= np.spacing(np.abs(rv).astype(np.float16)).astype(np.float64))
    q4a.check_device_error()


def test_moe_bank_64_experts():
    """64 experts, hidden 2048, inter 640, 16 tokens routed top-8 by N(0,1) logits:
    gate|up over the union with the token map, the activation step, then down."""
    gu_q, dn_q = wl.moe_banks()
    r = wl.route_by_logits(wl.moe_logits(), wl.MOE_TOP_K)
    assert int(r.token_offsets[-1]) == wl.MOE_TOKENS * wl.MOE_TOP_K
    gu = Dense(gu_q)
    dn = Dense(dn_q)
    x = wl.normal_f16(wl.MOE_BANK, wl.T_X, (wl.MOE_TOKENS, wl.MOE_HIDDEN))
    y_ref, bound = oracle.gemv_experts(gu.packed, gu_q.scale, gu_q.bias, x, r.x_rows, r.expert_ids,
                                       r.token_offsets, wl.MOE_EXPERTS, 2 * wl.MOE_INTER)
    y = host(q4a.gemv_experts(gu.w, gu.s, gu.b, dev(x), dev(r.x_rows), r.expert_ids, r.token_offsets,
                              wl.MOE_EXPERTS, 2 * wl.MOE_INTER))
    check(y, y_ref, bound, "moe gate|up")
    # activation on the oracle's gate|up output (shared input), then the down projection
    h_ref = oracle.silu_mul_f16(y_ref.astype(np.float32))
    h, hs = q4a.silu_mul_xsum(dev(y_ref.astype(np.float32)))
    hv, rv = host(h).view(np.float16).astype(np.float64), h_ref.view(np.float16).astype(np.float64)
    assert np.all(np.abs(hv - rv) <= np.spacing(np.abs(rv).astype(np.float16)).astype(np.float64))
    yd_ref, bd = oracle.gemv_experts(dn.packed, dn_q.scale, dn_q.bias, h_ref, None, r.expert_ids,
                                     r.token_offsets, wl.MOE_EXPERTS, wl.MOE_HIDDEN)
    yd = host(q4a.gemv_experts(dn.w, dn.s, dn.b, dev(h_ref), None, r.expert_ids, r.token_offsets,
                               wl.MOE_EXPERTS, wl.MOE_HIDDEN))
    check(yd, yd_ref, bd, "moe down")
    q4a.check_device_error()


@pytest.fixture(scope="module")
def lm_head():
    c = wl.LM_HEAD_CASE
    return Dense(wl.quant_matrix(c.config_id, c.out_dim, c.in_dim))


@pytest.mark.parametrize("nb", wl.LM_HEAD_CASE.nbs)
def test_lm_head_4096x151936_sampled(lm_head, nb):
    """Whole output checked for finiteness; 768 sampled entries (the first and last rows,
    every activation row, random rows) against one oracle dot product each."""
    c = wl.LM_HEAD_CASE
    x = wl.dense_x(c, nb)
    y = host(q4a.gemv(lm_head.w, lm_head.s, lm_head.b, dev(x)))
    assert y.shape == (nb, c.out_dim) and np.isfinite(y).all()
    rng = np.random.default_rng(nb)
    o = np.concatenate([[0, 1, 15, 16, c.out_dim - 1, c.out_dim - 17],
                        rng.integers(0, c.out_dim, 762)]).astype(np.int64)
    rr = np.concatenate([np.arange(min(nb, 6)), rng.integers(0, nb, 768 - min(nb, 6))]).astype(np.int64)
    rr = rr[:o.shape[0]]
    y_ref, bound = oracle.gemv_entries(lm_head.packed, lm_head.qm.scale, lm_head.qm.bias, x, rr, o)
    check(y[rr, o], y_ref, bound, f"lm_head nb={nb}")
    q4a.check_device_error()
