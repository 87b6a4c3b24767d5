"""GPU parity: every entry point of libq4a.so against the CPU oracle on identical
seeded inputs, through the C ABI (via the thin binding).

Bars:
  * q4a_pack: bit-exact.
  * q4a_gemv / _experts / _rmsnorm: per element |y - y_ref| <= 2e-3 * sum_i |w_oi x_ri| + 1e-5
    (the oracle's bound), every element, plus a NaN-sentinel check that every
    output is written.
  * q4a_xsum: fp32 summation of 64 binary16 values: |d| <= 64 * 2^-24 * sum |x| + 1e-30.
  * q4a_silu_mul_xsum: h within one binary16 ulp of the oracle's correctly rounded
    value (fp32 vs fp64 evaluation of silu(g)*u may straddle a rounding boundary);
    the group sums within 64 ulp-sized steps of the oracle's.
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


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def ragged_case(out_dim, in_dim, nb, seed):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(out_dim, in_dim), dtype=np.uint8)
    s = wl.f32_to_bf16_bits(np.abs(rng.normal(0, 0.02, (out_dim, in_dim // 64))).astype(np.float32))
    b = wl.f32_to_bf16_bits((-8 * rng.normal(0, 0.01, (out_dim, in_dim // 64))).astype(np.float32))
    x = wl.f16_bits(rng.normal(0, 1, (nb, in_dim)))
    return codes, s, b, x


def assert_within_bound(y: np.ndarray, y_ref: np.ndarray, bound: np.ndarray, what: str) -> float:
    assert y.shape == y_ref.shape, what
    assert np.isfinite(y).all(), f"{what}: non-finite output (unwritten or overflow)"
    ratio = np.abs(y.astype(np.float64) - y_ref) / bound
    worst = float(ratio.max())
    assert worst <= 1.0, f"{what}: worst err/bound {worst:.3g} at {np.unravel_index(ratio.argmax(), ratio.shape)}"
    return worst


def run_gemv(packed, s, b, x, out_dim):
    y = torch.full((x.shape[0], out_dim), float("nan"), dtype=torch.float32, device=DEV)
    q4a.gemv(dev(packed), dev(s), dev(b), dev(x), out=y)
    torch.cuda.synchronize()
    q4a.check_device_error()
    return host(y)


# ---- A1 / A2 ---------------------------------------------------------------------------

@pytest.mark.parametrize("rows,in_dim", [(1, 64), (7, 192), (300, 4096), (33, 640)])
def test_pack_bit_exact(rows, in_dim):
    rng = np.random.default_rng(rows + in_dim)
    codes = rng.integers(0, 256, size=(rows, in_dim), dtype=np.uint8)   # high bits must be masked
    got = host(q4a.pack(dev(codes)))
    assert np.array_equal(got, oracle.pack(codes))


@pytest.mark.parametrize("nb,in_dim", [(1, 64), (3, 320), (16, 4096)])
def test_xsum(nb, in_dim):
    x = wl.f16_bits(np.random.default_rng(nb).normal(0, 1, (nb, in_dim)))
    got = host(q4a.xsum(dev(x))).astype(np.float64)
    ref = oracle.xsum(x)
    mag = np.abs(x.view(np.float16).astype(np.float64)).reshape(nb, -1, 64).sum(axis=2)
    assert np.all(np.abs(got - ref) <= 64 * 2.0 ** -24 * mag + 1e-30)


# ---- A4 --------------------------------------------------------------------------------

GEMV_CASES = [
    (256, 512, 1),      # the 256 x 512 single-row workload
    (1, 64, 1),         # smallest
    (7, 128, 3),        # odd rows, partial tile
    (33, 192, 5),       # odd group count (2-byte scale copies)
    (100, 640, 8),      # 10 groups (4-byte scale copies), 8 rows
    (300, 1024, 9),     # 16-wide activation tiles
    (129, 2048, 17),    # 32-wide activation tiles
    (65, 4096, 32),     # cluster K split, 32 rows
    (50, 512, 33),      # two activation chunks
    (40, 4096, 16),     # cluster of 2
    (24, 12288, 2),     # long rows, cluster of 4
    (17, 12288, 16),    # long rows, cluster of 8
    (2000, 256, 4),     # many tiles per cluster
    (40, 98304, 1),     # 1536 groups, the longest row at NB <= 8 on any matrix: an 8-CTA K split
    (16, 131072, 1),    # 2048 groups on one tile: an 8-CTA K split of 2-tile row blocks
    (20, 576, 63),      # the widest batch below the tensor-core path (two segments)
    (10, 576, 256),     # 9 groups keep NB 256 on the GEMV kernel: eight 32-row segments
]


def test_gemv_row_longer_than_the_budget_is_unsupported():
    """The GEMV kernel keeps a CTA's K-slice of activations and of the row block's scales and
    biases in shared memory: 16384 groups at NB 1 exceed it even split 8 ways (2048 groups of
    activation fragments per CTA), and the call reports Q4A_ERR_UNSUPPORTED before launching
    anything."""
    codes, s, b, x = ragged_case(16, 1048576, 1, 5)
    with pytest.raises(q4a.Q4AError) as e:
        run_gemv(oracle.pack(codes), s, b, x, 16)
    assert e.value.status == 4


@pytest.mark.parametrize("out_dim,in_dim,nb", GEMV_CASES)
def test_gemv_matches_oracle(out_dim, in_dim, nb):
    codes, s, b, x = ragged_case(out_dim, in_dim, nb, out_dim * 7 + in_dim + nb)
    packed = oracle.pack(codes)
    y = run_gemv(packed, s, b, x, out_dim)
    y_ref, bound = oracle.gemv(packed, s, b, x)
    assert_within_bound(y, y_ref, bound, f"gemv {out_dim}x{in_dim} nb={nb}")


def test_gemv_is_deterministic():
    codes, s, b, x = ragged_case(513, 4096, 16, 1)
    packed = oracle.pack(codes)
    y1 = run_gemv(packed, s, b, x, 513)
    y2 = run_gemv(packed, s, b, x, 513)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_gemv_closed_forms_on_gpu():
    """codes == 0 -> y = sum_g b*xsum; codes == 15 and b == 0 -> 15 * sum_g s*xsum."""
    _, s, b, x = ragged_case(48, 1024, 4, 3)
    zero = oracle.pack(np.zeros((48, 1024), np.uint8))
    y0 = run_gemv(zero, s, b, x, 48)
    r0, bd0 = oracle.gemv(zero, s, b, x)
    assert_within_bound(y0, r0, bd0, "codes=0")
    fif = oracle.pack(np.full((48, 1024), 15, np.uint8))
    zb = np.zeros_like(b)
    y15 = run_gemv(fif, s, zb, x, 48)
    r15, bd15 = oracle.gemv(fif, s, zb, x)
    assert_within_bound(y15, r15, bd15, "codes=15,b=0")


def test_gemv_adversarial_scales():
    codes, s, b, x = ragged_case(32, 256, 2, 4)
    s = s.copy()
    s[0, 0] = 0x7FC0   # NaN scale
    s[1, 1] = 0x7F80   # +inf scale
    s[2, 2] = 0x0001   # subnormal bf16
    s[3, 3] = 0x7B00   # 6.6e35: the result stays inside fp32, scale * 2^24 would not
    s[4, 0] = 0x7F7F   # largest finite bf16: the result leaves the fp32 range
    b = b.copy()
    b[5, 1] = 0x7B00   # huge bias
    packed = oracle.pack(codes)
    y = torch.zeros((2, 32), dtype=torch.float32, device=DEV)
    q4a.gemv(dev(packed), dev(s), dev(b), dev(x), out=y)
    y = host(y).astype(np.float64)
    y_ref, bound = oracle.gemv(packed, s, b, x)
    assert np.isnan(y[:, 0]).all()
    assert not np.isfinite(y[:, 1]).any()
    fits = np.isfinite(y_ref) & (np.abs(y_ref) < 3.0e38)
    fits[:, :2] = False
    assert np.all(np.abs(y[fits] - y_ref[fits]) <= bound[fits])
    assert fits[:, 3].all() and fits[:, 5].all()
    over = np.isfinite(y_ref) & (np.abs(y_ref) > 3.5e38)
    assert over[:, 4].all() and not np.isfinite(y[over]).any()


def test_gemv_extreme_activations():
    """Tiny (subnormal-range) and large activations: the 1/16 pre-scaling of
    high-nibble activations and the 2^24 code scale must stay inside the bound."""
    codes, s, b, _ = ragged_case(64, 512, 3, 5)
    rng = np.random.default_rng(6)
    x = np.stack([rng.normal(0, 1e-4, 512), rng.normal(0, 3e3, 512),
                  np.where(rng.random(512) < 0.5, 6e-8, -6e-8)])
    xb = wl.f16_bits(x)
    packed = oracle.pack(codes)
    y = run_gemv(packed, s, b, xb, 64)
    y_ref, bound = oracle.gemv(packed, s, b, xb)
    assert_within_bound(y, y_ref, bound, "extreme activations")


# ---- A3 --------------------------------------------------------------------------------

@pytest.mark.parametrize("out_dim,in_dim,nb,shift", [(300, 1024, 4, 0.0), (77, 4096, 16, 0.0),
                                                     (40, 512, 1, 1.0), (33, 12288, 3, 0.0)])
def test_gemv_rmsnorm_matches_oracle(out_dim, in_dim, nb, shift):
    codes, s, b, _ = ragged_case(out_dim, in_dim, nb, 11)
    a = wl.normal_f32(77, 0, (nb, in_dim)) * 3.0
    nw = wl.norm_weight(77, 1, in_dim)
    if shift:
        nw = wl.f32_to_bf16_bits(wl.bf16_bits_to_f32(nw) - np.float32(shift))
    packed = oracle.pack(codes)
    y = torch.full((nb, out_dim), float("nan"), dtype=torch.float32, device=DEV)
    q4a.gemv_rmsnorm(dev(packed), dev(s), dev(b), dev(a), dev(nw), eps=1e-6, shift=shift, out=y)
    torch.cuda.synchronize()
    q4a.check_device_error()
    xn, _ = oracle.rmsnorm_f16(a, nw, eps=1e-6, shift=shift)
    y_ref, bound = oracle.gemv(packed, s, b, xn)
    assert_within_bound(host(y), y_ref, bound, f"gemv_rmsnorm {out_dim}x{in_dim} nb={nb}")


@pytest.mark.parametrize("out_dim,in_dim,nb,groups", [(300, 1024, 4, 2), (77, 4096, 16, 4), (40, 512, 1, 8),
                                                      (33, 12288, 3, 3), (129, 2048, 9, 1)])
def test_gemv_rmsnorm_grouped_matches_oracle(out_dim, in_dim, nb, groups):
    """Each of `groups` segments of a row normalised on its own (one loud segment), on both
    the single-CTA and the cluster K-split layouts."""
    codes, s, b, _ = ragged_case(out_dim, in_dim, nb, 12)
    a = wl.normal_f32(78, 0, (nb, in_dim)) * 3.0
    n = in_dim // groups
    a[:, :n] *= 50.0
    nw = wl.norm_weight(78, 1, in_dim)
    packed = oracle.pack(codes)
    y = torch.full((nb, out_dim), float("nan"), dtype=torch.float32, device=DEV)
    q4a.gemv_rmsnorm_grouped(dev(packed), dev(s), dev(b), dev(a), dev(nw), groups, eps=1e-6, out=y)
    torch.cuda.synchronize()
    q4a.check_device_error()
    xn, _ = oracle.rmsnorm_groups_f16(a, nw, groups, eps=1e-6)
    y_ref, bound = oracle.gemv(packed, s, b, xn)
    assert_within_bound(host(y), y_ref, bound, f"gemv_rmsnorm_grouped {out_dim}x{in_dim} nb={nb} groups={groups}")


# ---- A7 --------------------------------------------------------------------------------

def ulp16(v: np.ndarray) -> np.ndarray:
    f = np.abs(v.astype(np.float16))
    return np.spacing(f).astype(np.float64)


@pytest.mark.parametrize("rows,inter", [(1, 64), (128, 640), (16, 6144)])
def test_silu_mul_xsum(rows, inter):
    gu = (np.random.default_rng(rows + inter).normal(0, 2, (rows, 2 * inter))).astype(np.float32)
    h, hs = q4a.silu_mul_xsum(dev(gu))
    h = host(h).view(np.uint16)
    hs = host(hs).astype(np.float64)
    ref = oracle.silu_mul_f16(gu)
    hv = h.view(np.float16).astype(np.float64)
    rv = ref.view(np.float16).astype(np.float64)
    assert np.all(np.abs(hv - rv) <= ulp16(rv)), "h differs by more than one binary16 ulp"
    assert (h == ref).mean() > 0.99
    ref_sum = oracle.xsum(ref)
    tol = 64 * ulp16(np.abs(rv).reshape(rows, -1, 64).max(axis=2)) + 64 * 2.0 ** -24 * np.abs(rv).reshape(rows, -1, 64).sum(axis=2)
    assert np.all(np.abs(hs - ref_sum) <= tol)


# ---- A6 --------------------------------------------------------------------------------

def bank_case(n_exp, out_dim, in_dim, seed):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(n_exp * out_dim, in_dim), dtype=np.uint8)
    s = wl.f32_to_bf16_bits(np.abs(rng.normal(0, 0.02, (n_exp * out_dim, in_dim // 64))).astype(np.float32))
    b = wl.f32_to_bf16_bits((-8 * rng.normal(0, 0.01, (n_exp * out_dim, in_dim // 64))).astype(np.float32))
    return oracle.pack(codes), s, b


def run_experts(packed, s, b, x, x_rows, ids, offs, n_exp, out_dim):
    n_rows = int(offs[-1])
    y = torch.full((n_rows, out_dim), -777.0, dtype=torch.float32, device=DEV)
    xr = None if x_rows is None else dev(np.asarray(x_rows, np.int32))
    q4a.gemv_experts(dev(packed), dev(s), dev(b), dev(x), xr, ids, offs, n_exp, out_dim, out=y)
    torch.cuda.synchronize()
    q4a.check_device_error()
    return host(y)


def test_experts_duplicates_empty_and_map():
    n_exp, out_dim, in_dim = 6, 40, 256
    packed, s, b = bank_case(n_exp, out_dim, in_dim, 21)
    x = wl.normal_f16(91, 0, (5, in_dim))
    ids = np.array([3, 5, 3, 0, 2], np.int32)          # duplicate expert, and an empty segment
    offs = np.array([0, 2, 3, 3, 7, 9], np.int32)
    x_rows = np.array([4, 0, 1, 2, 3, 4, 0, 1, 1], np.int32)
    y = run_experts(packed, s, b, x, x_rows, ids, offs, n_exp, out_dim)
    y_ref, bound = oracle.gemv_experts(packed, s, b, x, x_rows, ids, offs, n_exp, out_dim)
    assert_within_bound(y, y_ref, bound, "experts")


def test_experts_invalid_id_gives_nan_rows():
    n_exp, out_dim, in_dim = 3, 24, 128
    packed, s, b = bank_case(n_exp, out_dim, in_dim, 22)
    x = wl.normal_f16(92, 0, (4, in_dim))
    ids = np.array([1, 9, 0], np.int32)
    offs = np.array([0, 1, 3, 4], np.int32)
    y = run_experts(packed, s, b, x, None, ids, offs, n_exp, out_dim)
    assert np.isnan(y[1:3]).all()
    y_ref, bound = oracle.gemv_experts(packed, s, b, x, None, ids, offs, n_exp, out_dim)
    assert_within_bound(y[[0, 3]], y_ref[[0, 3]], bound[[0, 3]], "experts valid rows")


def test_experts_many_tokens_per_expert():
    n_exp, out_dim, in_dim = 2, 48, 640
    packed, s, b = bank_case(n_exp, out_dim, in_dim, 23)
    x = wl.normal_f16(93, 0, (70, in_dim))
    ids = np.array([1, 0], np.int32)
    offs = np.array([0, 40, 70], np.int32)               # 40 rows -> two chunks of the segment
    y = run_experts(packed, s, b, x, None, ids, offs, n_exp, out_dim)
    y_ref, bound = oracle.gemv_experts(packed, s, b, x, None, ids, offs, n_exp, out_dim)
    assert_within_bound(y, y_ref, bound, "experts 40 rows")


@pytest.mark.parametrize("in_dim,tokens", [(640, 1), (320, 12), (704, 20)])
def test_experts_short_rows_scales_read_in_place(in_dim, tokens):
    """Rows whose group count is not a multiple of 8 (10, 5 and 11 groups) take the raw scale
    mode: each row block's scales and biases arrive as one contiguous [rows][groups] copy and
    the consumers read them where they landed (odd group counts: 16-bit reads only). 48 experts
    of 600 rows (a ragged last tile each) and 1 / 12 / 20 tokens per expert (one, two and four
    8-row activation tiles) give every CTA several row blocks, so the three raw buffers cycle."""
    n_exp, out_dim = 48, 600
    packed, s, b = bank_case(n_exp, out_dim, in_dim, 24 + tokens)
    n_x = 7
    x = wl.normal_f16(94, 0, (n_x, in_dim))
    rng = np.random.default_rng(95 + tokens)
    ids = rng.permutation(n_exp).astype(np.int32)
    offs = np.arange(n_exp + 1, dtype=np.int32) * tokens
    x_rows = rng.integers(0, n_x, size=n_exp * tokens).astype(np.int32)
    y = run_experts(packed, s, b, x, x_rows, ids, offs, n_exp, out_dim)
    y_ref, bound = oracle.gemv_experts(packed, s, b, x, x_rows, ids, offs, n_exp, out_dim)
    assert_within_bound(y, y_ref, bound, f"experts, {in_dim // 64} groups per row")


def test_pack_then_gemv_back_to_back():
    """The GEMV streams weights without waiting for the previous kernel of the stream;
    q4a_pack must still be fully visible to a GEMV launched right after it. The same
    weight buffer is repacked with new codes and used immediately, several times."""
    out_dim, in_dim, nb = 2048, 4096, 4
    _, s, b, x = ragged_case(out_dim, in_dim, nb, 31)
    w = torch.empty((out_dim, in_dim // 2), dtype=torch.uint8, device=DEV)
    sd, bd, xd = dev(s), dev(b), dev(x)
    ys, refs = [], []
    for k in range(4):
        codes = np.random.default_rng(100 + k).integers(0, 16, size=(out_dim, in_dim), dtype=np.uint8)
        cd = dev(codes)
        torch.cuda.synchronize()
        q4a.pack(cd, out=w)
        ys.append(q4a.gemv(w, sd, bd, xd))
        refs.append(oracle.gemv(oracle.pack(codes), s, b, x))
    torch.cuda.synchronize()
    q4a.check_device_error()
    for k in range(4):
        assert_within_bound(host(ys[k]), refs[k][0], refs[k][1], f"pack->gemv round {k}")
