"""GPU parity of the routed experts' fused gate|up with the SiLU*up epilogue
(q4a_gemv_experts_gate_up_silu: "BATCH_MSL" experts.metal fn_moe_gate_up_b followed by
fn_moe_act_b) against the CPU oracle, through the C ABI.

Expert e of the bank holds its gate rows at e*2*inter.. and its up rows right after them
(reading 13), so the oracle's routed product over the bank read with 2*inter rows per expert
gives the gate and up values of every routed row. Bar on h, as for the dense fused gate|up:
with g, u the oracle's values and bg, bu their GEMV bounds (2e-3 * sum|w x| + 1e-5),
|h - silu(g) u| <= 1.1 (|u| + bu) bg + (|silu(g)| + 1.1 bg) bu + 2^-11 |silu(g) u| + 2^-24
(silu' <= 1.1, one rounding to binary16).
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


def bank(n_exp, inter, in_dim, seed):
    rng = np.random.default_rng(seed)
    rows = n_exp * 2 * inter
    codes = rng.integers(0, 16, size=(rows, in_dim), dtype=np.uint8)
    s = wl.f32_to_bf16_bits(np.abs(rng.normal(0, 0.02, (rows, in_dim // 64))).astype(np.float32))
    b = wl.f32_to_bf16_bits((-8 * rng.normal(0, 0.01, (rows, in_dim // 64))).astype(np.float32))
    return oracle.pack(codes), s, b


def run(packed, s, b, x, x_rows, ids, offs, n_exp, inter):
    n_rows = int(offs[-1])
    h = torch.full((n_rows, inter), float("nan"), dtype=torch.float16, device=DEV)
    xr = None if x_rows is None else dev(np.asarray(x_rows, np.int32))
    q4a.gemv_experts_gate_up_silu(dev(packed), dev(s), dev(b), dev(x), xr, ids, offs, n_exp, inter, out=h)
    torch.cuda.synchronize()
    q4a.check_device_error()
    return h.cpu().numpy()


def check_h(h, packed, s, b, x, x_rows, ids, offs, n_exp, inter, what, rows=None):
    y, bound = oracle.gemv_experts(packed, s, b, x, x_rows, ids, offs, n_exp, 2 * inter)
    if rows is not None:
        h, y, bound = h[rows], y[rows], bound[rows]
    g, u, bg, bu = y[:, :inter], y[:, inter:], bound[:, :inter], bound[:, inter:]
    sg = g / (1.0 + np.exp(-g))
    ref = sg * u
    tol = 1.1 * (np.abs(u) + bu) * bg + (np.abs(sg) + 1.1 * bg) * bu + 2.0 ** -11 * np.abs(ref) + 2.0 ** -24
    assert np.isfinite(h).all(), f"{what}: non-finite h"
    worst = float((np.abs(h.astype(np.float64) - ref) / tol).max())
    assert worst <= 1.0, f"{what}: h worst err/bound {worst:.3g}"


@pytest.mark.parametrize("n_exp,inter,in_dim", [(6, 32, 512), (4, 48, 1024), (3, 640, 2048)])
def test_duplicates_empty_segment_and_row_map(n_exp, inter, in_dim):
    packed, s, b = bank(n_exp, inter, in_dim, n_exp + inter + in_dim)
    x = wl.normal_f16(94, n_exp, (5, in_dim))
    ids = np.array([n_exp - 1, 0, n_exp - 1, 1, 2], np.int32)   # a duplicate expert, an empty segment
    offs = np.array([0, 2, 3, 3, 7, 9], np.int32)
    x_rows = np.array([4, 0, 1, 2, 3, 4, 0, 1, 1], np.int32)
    h = run(packed, s, b, x, x_rows, ids, offs, n_exp, inter)
    check_h(h, packed, s, b, x, x_rows, ids, offs, n_exp, inter, f"experts gate|up {n_exp}x{inter}x{in_dim}")


def test_many_rows_per_expert():
    """40 and 30 rows for one expert each: the segments span several 8-row activation blocks."""
    n_exp, inter, in_dim = 2, 64, 512
    packed, s, b = bank(n_exp, inter, in_dim, 31)
    x = wl.normal_f16(95, 0, (70, in_dim))
    ids = np.array([1, 0], np.int32)
    offs = np.array([0, 40, 70], np.int32)
    h = run(packed, s, b, x, None, ids, offs, n_exp, inter)
    check_h(h, packed, s, b, x, None, ids, offs, n_exp, inter, "many rows per expert")


def test_invalid_expert_gives_nan_rows():
    n_exp, inter, in_dim = 3, 32, 512
    packed, s, b = bank(n_exp, inter, in_dim, 32)
    x = wl.normal_f16(96, 0, (4, in_dim))
    ids = np.array([1, 7, 0], np.int32)
    offs = np.array([0, 1, 3, 4], np.int32)
    h = run(packed, s, b, x, None, ids, offs, n_exp, inter)
    assert np.isnan(h[1:3].astype(np.float32)).all()
    check_h(h, packed, s, b, x, None, ids, offs, n_exp, inter, "valid rows", rows=[0, 3])


def test_moe_bank_64_experts_fused():
    """The routed MoE workload: 64 experts, hidden 2048, inter 640, 16 tokens top-8 by N(0,1)
    logits; h from the fused call against the oracle's gate|up products."""
    gu_q, _ = wl.moe_banks()
    r = wl.route_by_logits(wl.moe_logits(), wl.MOE_TOP_K)
    packed = oracle.pack(gu_q.codes)
    x = wl.normal_f16(wl.MOE_BANK, wl.T_X, (wl.MOE_TOKENS, wl.MOE_HIDDEN))
    h = run(packed, gu_q.scale, gu_q.bias, x, r.x_rows, r.expert_ids, r.token_offsets, wl.MOE_EXPERTS,
            wl.MOE_INTER)
    check_h(h, packed, gu_q.scale, gu_q.bias, x, r.x_rows, r.expert_ids, r.token_offsets, wl.MOE_EXPERTS,
            wl.MOE_INTER, "moe gate|up fused")
