"""GPU parity of the routed low-bit experts (q4a_gemv_experts_lowbit) against the CPU oracle:
2- and 3-bit codes derived from 4-bit ones ("BATCH_MSL" quantized_rows.metal fn_q2_rows_h /
fn_q3_rows_h, routed; expert_gemm.metal fn_expert_qmm, the prefill contraction over 8/16/32
token rows of fp32 activations).

Bar: the GEMV bound 2e-3 * sum|w x| + 1e-5 per element, with the oracle's exact product of
the activations as given. The kernel rounds fp32 activations to binary16 when it stages them
(as the pages' contraction does): at most 2^-11 of each |w x| term, inside the bound. Rows of
an out-of-range expert are NaN; every other output must be written (NaN sentinel)."""

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


def bank(seed, n_exp, out_dim, in_dim):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(n_exp * out_dim, in_dim), dtype=np.uint8)
    s = wl.f32_to_bf16_bits(np.abs(rng.normal(0, 0.02, (n_exp * out_dim, in_dim // 64))).astype(np.float32))
    b = wl.f32_to_bf16_bits((-8 * rng.normal(0, 0.01, (n_exp * out_dim, in_dim // 64))).astype(np.float32))
    return codes, s, b


def run(bits, codes, s, b, x, x_rows, ids, offs, n_exp, out_dim):
    w2, lo = oracle.lowbit_pack2(codes), oracle.lowbit_pack3lo(codes)
    n_rows = int(offs[-1])
    y = torch.full((n_rows, out_dim), float("nan"), device=DEV)
    xd = torch.from_numpy(np.ascontiguousarray(x)).to(DEV) if x.dtype == np.float32 else dev(x)
    q4a.gemv_experts_lowbit(bits, dev(w2), dev(lo) if bits == 3 else None, dev(s), dev(b), xd,
                            None if x_rows is None else torch.from_numpy(x_rows).to(DEV), ids, offs, n_exp, out_dim,
                            out=y)
    torch.cuda.synchronize()
    q4a.check_device_error()
    ref, bound = oracle.experts_lowbit(w2, lo if bits == 3 else None, s, b, x, x_rows, ids, offs, n_exp, out_dim)
    return y.cpu().numpy().astype(np.float64), ref, bound


def check(yh, ref, bound, what):
    ok = np.isfinite(ref)
    assert np.isnan(yh[~ok]).all(), f"{what}: rows of an invalid expert must be NaN"
    assert np.isfinite(yh[ok]).all(), f"{what}: unwritten or non-finite output"
    worst = float((np.abs(yh[ok] - ref[ok]) / bound[ok]).max())
    assert worst <= 1.0, f"{what}: worst err/bound {worst:.3g}"


@pytest.mark.parametrize("bits", [2, 3])
@pytest.mark.parametrize("f32", [True, False])
def test_moe_bank_shapes(bits, f32):
    """The 64-expert bank of the MoE workload (gate|up 2048 -> 1280, down 640 -> 2048), routed
    top-8 for 16 tokens: the gate|up product through the token map, the down product over the
    128 slot rows, prefill (fp32) and decode (binary16) activations."""
    r = wl.route_by_logits(wl.moe_logits(), wl.MOE_TOP_K)
    E, H, I = wl.MOE_EXPERTS, wl.MOE_HIDDEN, wl.MOE_INTER
    rng = np.random.default_rng(11 + bits)
    for out_dim, in_dim, seed, rows in ((2 * I, H, 31, wl.MOE_TOKENS), (H, I, 32, int(r.token_offsets[-1]))):
        codes, s, b = bank(seed + bits, E, out_dim, in_dim)
        x = rng.normal(0, 1, (rows, in_dim)).astype(np.float32)
        x = x if f32 else wl.f16_bits(x.astype(np.float64))
        x_rows = r.x_rows if rows == wl.MOE_TOKENS else None
        yh, ref, bound = run(bits, codes, s, b, x, x_rows, r.expert_ids, r.token_offsets, E, out_dim)
        check(yh, ref, bound, f"moe bank {in_dim}->{out_dim} bits={bits} f32={f32}")


@pytest.mark.parametrize("bits", [2, 3])
def test_prefill_token_tiles_and_edges(bits):
    """Segments of 8, 16, 32 and 40 token rows (the pages' tiles, and a segment longer than one
    tile), an empty segment, a repeated expert and an invalid expert id."""
    n_exp, out_dim, in_dim = 5, 136, 1024
    codes, s, b = bank(40 + bits, n_exp, out_dim, in_dim)
    ids = np.array([0, 3, 1, 9, 3, 4], np.int32)
    lens = [8, 16, 0, 5, 32, 40]
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    x = (np.random.default_rng(50 + bits).normal(0, 1, (int(offs[-1]), in_dim)) * 3).astype(np.float32)
    yh, ref, bound = run(bits, codes, s, b, x, None, ids, offs, n_exp, out_dim)
    check(yh, ref, bound, f"tiles bits={bits}")
