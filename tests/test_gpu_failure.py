"""Failure detection on the GPU without faulting it: a launch that never receives one of its
weight stages (the q4a_debug_withhold_stage hook keeps the producer from loading it) gives up
its bounded wait, finishes, and q4a_check_device_error reports Q4A_ERR_TIMEOUT; the stream and
the context stay usable, and the next call is correct (checked against the CPU oracle)."""

import time

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
    return oracle.pack(codes), s, b, x


@pytest.mark.parametrize("out_dim,in_dim,nb", [(512, 4096, 2), (1024, 12288, 1)])
def test_withheld_stage_times_out_and_the_next_call_is_clean(out_dim, in_dim, nb):
    """One CTA per row range (4096 inputs) and a two-CTA cluster splitting K (12288 inputs):
    every CTA misses its second weight stage."""
    packed, s, b, x = case(out_dim, in_dim, nb, out_dim + in_dim)
    w_d, s_d, b_d, x_d = dev(packed), dev(s), dev(b), dev(x)
    q4a.check_device_error()                      # start from a clean error word
    q4a.debug_withhold_stage(1)
    t0 = time.perf_counter()
    q4a.gemv(w_d, s_d, b_d, x_d)
    with pytest.raises(q4a.Q4AError) as err:
        q4a.check_device_error()
    waited = time.perf_counter() - t0
    assert err.value.status_name == "ERR_TIMEOUT"
    assert waited < 30.0
    # the request was for one launch only: the same call now runs clean and matches the oracle
    y = torch.full((nb, out_dim), float("nan"), device=DEV)
    q4a.gemv(w_d, s_d, b_d, x_d, out=y)
    q4a.check_device_error()
    ref, bound = oracle.gemv(packed, s, b, x)
    worst = float((np.abs(y.cpu().numpy().astype(np.float64) - ref) / bound).max())
    assert worst <= 1.0, f"after the timeout: worst err/bound {worst:.3g}"


def test_withheld_stage_routed_short_rows():
    """The routed down projection's form: 640-wide rows whose scales and biases the consumers
    read from the raw staging buffers (three in flight). 16 experts of 2048 rows give every CTA
    three row blocks; every CTA misses its second weight stage (the 2-group second stage of its
    first row block). The launch gives up its wait, drains its copies, reports Q4A_ERR_TIMEOUT,
    and the next call on the stream matches the oracle."""
    n_exp, out_dim, in_dim, per = 16, 2048, 640, 2
    packed, s, b, x = case(n_exp * out_dim, in_dim, n_exp * per, 77)
    w_d, s_d, b_d, x_d = dev(packed), dev(s), dev(b), dev(x)
    ids = np.arange(n_exp, dtype=np.int32)[::-1].copy()
    offs = np.arange(n_exp + 1, dtype=np.int32) * per
    n_rows = int(offs[-1])
    q4a.check_device_error()
    q4a.debug_withhold_stage(1)
    t0 = time.perf_counter()
    q4a.gemv_experts(w_d, s_d, b_d, x_d, None, ids, offs, n_exp, out_dim)
    with pytest.raises(q4a.Q4AError) as err:
        q4a.check_device_error()
    waited = time.perf_counter() - t0
    assert err.value.status_name == "ERR_TIMEOUT"
    assert waited < 30.0
    y = torch.full((n_rows, out_dim), float("nan"), device=DEV)
    q4a.gemv_experts(w_d, s_d, b_d, x_d, None, ids, offs, n_exp, out_dim, out=y)
    q4a.check_device_error()
    ref, bound = oracle.gemv_experts(packed, s, b, x, None, ids, offs, n_exp, out_dim)
    worst = float((np.abs(y.cpu().numpy().astype(np.float64) - ref) / bound).max())
    assert worst <= 1.0, f"after the timeout: worst err/bound {worst:.3g}"
