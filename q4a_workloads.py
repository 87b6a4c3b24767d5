"""Seeded synthetic inputs for the affine-4-bit dequantising GEMV workloads.

This module is shared by the CPU oracle's tests and by the GPU path's tests and
benchmark. It holds only random draws and storage-format conversions
(fp32 -> bfloat16 bit patterns with round-to-nearest-even, fp32 -> IEEE
binary16 through numpy). No step of the product y = W.x, of the activation or
of the normalisation is computed here.

Every tensor comes from ``numpy.random.default_rng(SeedSequence([seed,
config_id, tensor_id]))`` so that each (workload, tensor) pair is reproducible
on its own, whatever else a caller draws.

Distributions (the workloads' description of the inputs):
  codes q   uniform integers 0..15, one per byte (unpacked)
  scale s   bf16(|N(0, 0.02)|)          (second argument = standard deviation)
  bias  b   bf16(-8 * N(0, 0.01))
  x         fp16(N(0, 1))               (raw activations)
  norm w    bf16(1 + N(0, 0.05))
"""

from __future__ import annotations

import dataclasses

import numpy as np

# Workload identifiers (the config_id component of every seed).
GEMV_SMALL = 0        # 256 x 512, NB = 1
DENSE_GATE_UP = 1     # 4096 -> 12288 (fused gate|up), NB in {1, 2, 4, 8, 16}
DENSE_DOWN = 2        # 12288 -> 4096, NB in {1, 4, 16}
MOE_BANK = 3          # 64 experts, hidden 2048, inter 640, 16 tokens top-8
LM_HEAD = 4           # 4096 -> 151936, NB in {1, 8, 32, 64, 128}

# Tensor identifiers (the tensor_id component of every seed).
T_CODES, T_SCALE, T_BIAS, T_X, T_NORM_W, T_A, T_B, T_LOGITS = range(8)
T_CODES_DOWN, T_SCALE_DOWN, T_BIAS_DOWN = 8, 9, 10
T_COMBINE = 11


def rng(config_id: int, tensor_id: int, seed: int = 0) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed, config_id, tensor_id]))


def f32_to_bf16_bits(a) -> np.ndarray:
    """fp32 -> bfloat16 bit patterns, round to nearest, ties to even.

    NaNs stay NaN (quiet bit forced); infinities stay infinite.
    """
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    rounded = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        rounded = rounded.copy()
        rounded[nan] = ((u[nan] >> 16).astype(np.uint16) | np.uint16(0x0040))
    return rounded


def bf16_bits_to_f32(bits) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f16_bits(a) -> np.ndarray:
    """fp32/fp64 -> IEEE binary16 bit patterns (numpy's round to nearest even)."""
    return np.asarray(a).astype(np.float16).view(np.uint16)


def codes(config_id: int, tensor_id: int, rows: int, in_dim: int, seed: int = 0) -> np.ndarray:
    return rng(config_id, tensor_id, seed).integers(0, 16, size=(rows, in_dim), dtype=np.uint8)


def scales(config_id: int, tensor_id: int, rows: int, groups: int, seed: int = 0) -> np.ndarray:
    z = rng(config_id, tensor_id, seed).normal(0.0, 0.02, size=(rows, groups)).astype(np.float32)
    return f32_to_bf16_bits(np.abs(z))


def biases(config_id: int, tensor_id: int, rows: int, groups: int, seed: int = 0) -> np.ndarray:
    z = rng(config_id, tensor_id, seed).normal(0.0, 0.01, size=(rows, groups)).astype(np.float32)
    return f32_to_bf16_bits(np.float32(-8.0) * z)


def normal_f32(config_id: int, tensor_id: int, shape, std: float = 1.0, seed: int = 0) -> np.ndarray:
    return rng(config_id, tensor_id, seed).normal(0.0, std, size=shape).astype(np.float32)


def normal_f16(config_id: int, tensor_id: int, shape, seed: int = 0) -> np.ndarray:
    return f16_bits(normal_f32(config_id, tensor_id, shape, seed=seed))


def norm_weight(config_id: int, tensor_id: int, n: int, seed: int = 0) -> np.ndarray:
    z = rng(config_id, tensor_id, seed).normal(0.0, 0.05, size=(n,)).astype(np.float32)
    return f32_to_bf16_bits(np.float32(1.0) + z)


@dataclasses.dataclass
class QuantMatrix:
    """Unpacked codes plus per-64-group bf16 scale and bias bit patterns."""

    codes: np.ndarray   # uint8 [rows][in_dim], values 0..15
    scale: np.ndarray   # uint16 bf16 bits [rows][in_dim/64]
    bias: np.ndarray    # uint16 bf16 bits [rows][in_dim/64]

    @property
    def rows(self) -> int:
        return self.codes.shape[0]

    @property
    def in_dim(self) -> int:
        return self.codes.shape[1]


def quant_matrix(config_id: int, rows: int, in_dim: int, seed: int = 0,
                 tensor_ids=(T_CODES, T_SCALE, T_BIAS)) -> QuantMatrix:
    assert in_dim % 64 == 0
    g = in_dim // 64
    tc, ts, tb = tensor_ids
    return QuantMatrix(codes(config_id, tc, rows, in_dim, seed),
                       scales(config_id, ts, rows, g, seed),
                       biases(config_id, tb, rows, g, seed))


@dataclasses.dataclass
class Routing:
    """Routed-expert segments: slots sorted by (expert, token)."""

    expert_ids: np.ndarray      # int32 [n_active]  (unique experts, ascending)
    token_offsets: np.ndarray   # int32 [n_active + 1]
    x_rows: np.ndarray          # int32 [n_rows]    token of each slot
    chosen: np.ndarray          # int32 [n_tokens][top_k] experts picked per token


def route_by_logits(logits: np.ndarray, top_k: int) -> Routing:
    """Pick each token's top_k experts by logit (ties -> lowest index) and
    group the (token, expert) slots by expert.

    Softmax is monotonic, so ranking logits ranks the routing probabilities;
    no probability is computed here (the combine weights are not an input of
    the expert GEMV).
    """
    n_tok, n_exp = logits.shape
    order = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")
    chosen = order[:, :top_k].astype(np.int32)
    pairs = sorted((int(e), t) for t in range(n_tok) for e in chosen[t])
    experts = sorted({e for e, _ in pairs})
    offsets = [0]
    x_rows = []
    for e in experts:
        toks = [t for ee, t in pairs if ee == e]
        x_rows.extend(toks)
        offsets.append(offsets[-1] + len(toks))
    return Routing(np.asarray(experts, np.int32), np.asarray(offsets, np.int32),
                   np.asarray(x_rows, np.int32), chosen)


# ---- the five workloads -------------------------------------------------------

@dataclasses.dataclass
class DenseCase:
    name: str
    config_id: int
    out_dim: int
    in_dim: int
    nbs: tuple


GEMV_SMALL_CASE = DenseCase("gemv_256x512", GEMV_SMALL, 256, 512, (1,))
DENSE_GATE_UP_CASE = DenseCase("dense_gate_up_4096x12288", DENSE_GATE_UP, 12288, 4096, (1, 2, 4, 8, 16))
DENSE_DOWN_CASE = DenseCase("dense_down_12288x4096", DENSE_DOWN, 4096, 12288, (1, 4, 16))
LM_HEAD_CASE = DenseCase("lm_head_4096x151936", LM_HEAD, 151936, 4096, (1, 8, 32, 64, 128))

MOE_EXPERTS = 64
MOE_HIDDEN = 2048
MOE_INTER = 640
MOE_TOKENS = 16
MOE_TOP_K = 8


def dense_x(case: DenseCase, nb: int, seed: int = 0) -> np.ndarray:
    """fp16 N(0,1) activations [nb][in_dim] (raw draw; the gate|up workload
    normalises its raw fp32 draw first, the down workload applies SiLU*mul)."""
    return normal_f16(case.config_id, T_X, (nb, case.in_dim), seed=seed)


def moe_logits(seed: int = 0) -> np.ndarray:
    return normal_f32(MOE_BANK, T_LOGITS, (MOE_TOKENS, MOE_EXPERTS), seed=seed)


def moe_combine_inputs(routing: Routing, seed: int = 0):
    """For the combine step: slot[t][k] = the slot (row of the expert outputs) of token
    t's k-th chosen expert, and routing weights w[t][k] > 0 summing to 1 per token
    (uniform draws, normalised; the combine reads them as given)."""
    n_tok, k = routing.chosen.shape
    where = {}
    for a, e in enumerate(routing.expert_ids):
        for s_ in range(int(routing.token_offsets[a]), int(routing.token_offsets[a + 1])):
            where[(int(e), int(routing.x_rows[s_]))] = s_
    slot = np.array([[where[(int(e), t)] for e in routing.chosen[t]] for t in range(n_tok)], np.int32)
    u = rng(MOE_BANK, T_COMBINE, seed).random((n_tok, k)) + 0.05
    w = (u / u.sum(axis=1, keepdims=True)).astype(np.float32)
    return slot, w


def moe_banks(seed: int = 0, n_experts: int = MOE_EXPERTS):
    """gate|up bank [E*1280][2048] and down bank [E*2048][640], expert-major."""
    gu = quant_matrix(MOE_BANK, n_experts * 2 * MOE_INTER, MOE_HIDDEN, seed,
                      (T_CODES, T_SCALE, T_BIAS))
    dn = quant_matrix(MOE_BANK, n_experts * MOE_HIDDEN, MOE_INTER, seed,
                      (T_CODES_DOWN, T_SCALE_DOWN, T_BIAS_DOWN))
    return gu, dn
