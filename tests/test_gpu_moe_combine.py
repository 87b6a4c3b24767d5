"""GPU parity of q4a_moe_combine (the routed-expert combine plus the gated shared expert)
against the CPU oracle, through the C ABI.

Bar, derived from the fp32 arithmetic of the kernel: each output is a chain of top_k + 1
fused multiply-adds (relative error <= (top_k + 1) 2^-24 of the sum of the absolute terms),
and the shared gate sigmoid(d) takes the gate dot d from a fixed-tree fp32 reduction over
hidden terms (|dd| <= 2^-20 sum|gate x| for hidden <= 2^12 per CTA thread count) through
sigmoid' <= 1/4 and expf (a few ulp):
    |out - out_ref| <= 2^-20 * sum|terms| + |y_shared| * (2^-20 * sum|gate x| + 2^-21).
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


def run(y, slot, w, ysh=None, gate=None, x=None):
    out = torch.full((slot.shape[0], y.shape[1]), float("nan"), dtype=torch.float32, device=DEV)
    q4a.moe_combine(dev(y), dev(slot), dev(w), None if ysh is None else dev(ysh),
                    None if gate is None else dev(gate), None if x is None else dev(x), out=out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def check(got, y, slot, w, ysh=None, gate=None, x=None, what=""):
    ref, asum, gabs = oracle.moe_combine(y, slot, w, ysh, gate, x)
    bound = 2.0 ** -20 * asum + 1e-30
    if ysh is not None:
        bound = bound + np.abs(ysh.astype(np.float64)) * (2.0 ** -20 * gabs[:, None] + 2.0 ** -21)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    worst = float((np.abs(got.astype(np.float64) - ref) / bound).max())
    assert worst <= 1.0, f"{what}: worst err/bound {worst:.3g}"


def moe_routing():
    """The 64-expert workload's routing: slots sorted by (expert, token); for every token
    the slot of each of its top-8 experts, and the renormalised softmax weights."""
    logits = wl.moe_logits()
    r = wl.route_by_logits(logits, wl.MOE_TOP_K)
    idx, wts = oracle.route_topk(logits, wl.MOE_TOP_K)
    where = {}
    for a, e in enumerate(r.expert_ids):
        for s_ in range(int(r.token_offsets[a]), int(r.token_offsets[a + 1])):
            where[(int(e), int(r.x_rows[s_]))] = s_
    slot = np.array([[where[(int(e), t)] for e in idx[t]] for t in range(idx.shape[0])], np.int32)
    return slot, wts.astype(np.float32), int(r.token_offsets[-1])


def test_combine_moe_workload():
    slot, w, n_slots = moe_routing()
    rng = np.random.default_rng(31)
    y = rng.normal(0, 1, (n_slots, wl.MOE_HIDDEN)).astype(np.float32)
    check(run(y, slot, w), y, slot, w, what="routed only")
    ysh = rng.normal(0, 1, (wl.MOE_TOKENS, wl.MOE_HIDDEN)).astype(np.float32)
    gate = wl.f32_to_bf16_bits(rng.normal(0, 0.02, wl.MOE_HIDDEN).astype(np.float32))
    x = rng.normal(0, 1, (wl.MOE_TOKENS, wl.MOE_HIDDEN)).astype(np.float32)
    check(run(y, slot, w, ysh, gate, x), y, slot, w, ysh, gate, x, what="with shared expert")


@pytest.mark.parametrize("n_tok,top_k,n_slots,hidden", [(1, 1, 1, 4), (3, 2, 5, 2052), (40, 64, 100, 1024),
                                                        (7, 8, 56, 5120)])
def test_combine_shapes(n_tok, top_k, n_slots, hidden):
    rng = np.random.default_rng(n_tok + top_k + hidden)
    y = rng.normal(0, 1, (n_slots, hidden)).astype(np.float32)
    slot = rng.integers(0, n_slots, (n_tok, top_k)).astype(np.int32)
    w = rng.random((n_tok, top_k)).astype(np.float32)
    ysh = rng.normal(0, 3, (n_tok, hidden)).astype(np.float32)
    gate = wl.f32_to_bf16_bits(rng.normal(0, 0.05, hidden).astype(np.float32))
    x = rng.normal(0, 1, (n_tok, hidden)).astype(np.float32)
    check(run(y, slot, w, ysh, gate, x), y, slot, w, ysh, gate, x, what=f"{n_tok}x{top_k}x{hidden}")


def test_combine_invalid_slot_and_determinism():
    rng = np.random.default_rng(33)
    y = rng.normal(0, 1, (10, 256)).astype(np.float32)
    slot = np.array([[1, 2], [3, 10], [-1, 0], [9, 9]], np.int32)
    w = rng.random((4, 2)).astype(np.float32)
    got = run(y, slot, w)
    assert np.isnan(got[1]).all() and np.isnan(got[2]).all()
    ok = np.array([0, 3])
    check(got[ok], y, slot[ok], w[ok], what="valid rows beside invalid ones")
    again = run(y, slot, w)
    assert np.array_equal(got.view(np.uint32), again.view(np.uint32))
