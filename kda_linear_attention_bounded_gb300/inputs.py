"""Seeded synthetic inputs for the KDA bounded-gate prefill and verify calls.

This module draws random numbers and encodes them; it holds none of the
method's arithmetic.  Both the fp64 oracle and the CUDA path consume exactly
the arrays produced here:

* bf16 tensors are returned as ``uint16`` bit patterns, rounded from fp32
  draws with round-to-nearest-even;
* per-head / per-channel parameters are ``float32``;
* sequence boundaries (``cu_seqlens``) and slot ids are ``int32``.

Random numbers come from NumPy's PCG64 ``Generator`` seeded per workload, so
a workload is a pure function of its name.

Workload recipes (H heads, head dim D = 128, lower_bound = -5,
scale = 1/sqrt(128) unless stated):

* ``q, k, v, g_raw`` ~ N(0, 1) per element, ``beta_logits`` ~ N(0, 1) per
  (token, head), all bf16;
* ``A_log = log(U[1, 16])`` per head, ``dt_bias`` ~ N(0, 0.1) per
  (head, channel), fp32;
* state pools ~ N(0, 0.02) (standard deviation 0.02), fp32
  ``[slots, H, D(k), D(v)]``; slot ids are distinct, drawn as a prefix of a
  random permutation of the pool.
"""
from __future__ import annotations

from dataclasses import dataclass, field
import math

import numpy as np

D = 128
LOWER_BOUND = -5.0
SCALE = 1.0 / math.sqrt(128.0)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return the bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((b + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class ConvInputs:
    """The short causal convolutions of q, k and v: weights ``[3 (q, k, v), H, D, W]`` fp32 (tap W-1 on the
    current input), SiLU after each, and a pool of windows ``[slots, 3, W-1, H, D]`` (bf16 bit patterns: the
    W-1 previous raw inputs, oldest first) beside the state pool, indexed by the same slot ids."""

    weight: np.ndarray
    silu: bool
    pool: np.ndarray


@dataclass
class PrefillInputs:
    """One chunked-prefill call: packed varlen tokens ``[T, H, D]``."""

    name: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    g: np.ndarray
    beta: np.ndarray
    A_log: np.ndarray
    dt_bias: np.ndarray
    lower_bound: float
    scale: float
    cu_seqlens: np.ndarray
    pool: np.ndarray | None = None
    slot_ids: np.ndarray | None = None
    load_initial: bool = False
    final_to_pool: bool = False
    meta: dict = field(default_factory=dict)
    conv: ConvInputs | None = None

    @property
    def num_seqs(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def H(self) -> int:
        return int(self.q.shape[1])

    def initial_states(self) -> np.ndarray | None:
        """Initial state per sequence, ``[N, H, D, D]`` fp32 (None = zero)."""
        if not self.load_initial:
            return None
        return self.pool[self.slot_ids]


@dataclass
class VerifyInputs:
    """One speculative-verify call: ``B`` requests with draft blocks of ``T`` tokens."""

    name: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    g: np.ndarray
    beta: np.ndarray
    A_log: np.ndarray
    dt_bias: np.ndarray
    lower_bound: float
    scale: float
    B: int
    T: int
    pool: np.ndarray
    slot_ids: np.ndarray
    meta: dict = field(default_factory=dict)
    conv: ConvInputs | None = None

    @property
    def H(self) -> int:
        return int(self.q.shape[1])


def conv_inputs(H: int, slots: int, *, seed: int, d: int = D, W: int = 4, silu: bool = True,
                weight_std: float = 0.5) -> ConvInputs:
    """weights ~ N(0, weight_std) per tap, windows ~ N(0, 1) (bf16)."""
    rng = np.random.default_rng(seed)
    weight = (rng.standard_normal((3, H, d, W)) * weight_std).astype(np.float32)
    pool = f32_to_bf16_bits(rng.standard_normal((slots, 3, W - 1, H, d), dtype=np.float32))
    return ConvInputs(weight=weight, silu=bool(silu), pool=pool)


def _token_tensors(rng, total, H, d, g_mean):
    shape = (total, H, d)
    q = f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
    k = f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
    v = f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
    g = f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) + np.float32(g_mean))
    beta = f32_to_bf16_bits(rng.standard_normal((total, H), dtype=np.float32))
    return q, k, v, g, beta


def _head_params(rng, H, d):
    A_log = np.log(rng.uniform(1.0, 16.0, size=H)).astype(np.float32)
    dt_bias = (rng.standard_normal((H, d)) * 0.1).astype(np.float32)
    return A_log, dt_bias


def prefill_inputs(name: str, seq_lens, H: int, *, seed: int, d: int = D,
                   pool_slots: int | None = None, load_initial: bool = False,
                   final_to_pool: bool = False, lower_bound: float = LOWER_BOUND,
                   scale: float | None = None, g_mean: float = 0.0,
                   state_std: float = 0.02) -> PrefillInputs:
    """Draw one prefill workload.  Draw order: tokens, head params, pool, slot ids."""
    seq_lens = [int(x) for x in seq_lens]
    rng = np.random.default_rng(seed)
    cu = np.zeros(len(seq_lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(seq_lens)
    total = int(cu[-1])
    q, k, v, g, beta = _token_tensors(rng, total, H, d, g_mean)
    A_log, dt_bias = _head_params(rng, H, d)
    pool = slot_ids = None
    if pool_slots is not None:
        pool = (rng.standard_normal((pool_slots, H, d, d), dtype=np.float32) * np.float32(state_std))
        slot_ids = rng.permutation(pool_slots)[: len(seq_lens)].astype(np.int32)
    return PrefillInputs(
        name=name, q=q, k=k, v=v, g=g, beta=beta, A_log=A_log, dt_bias=dt_bias,
        lower_bound=float(lower_bound), scale=float(1.0 / math.sqrt(d) if scale is None else scale),
        cu_seqlens=cu, pool=pool, slot_ids=slot_ids, load_initial=load_initial,
        final_to_pool=final_to_pool, meta={"seed": seed, "seq_lens": seq_lens})


def verify_inputs(name: str, B: int, T: int, H: int, *, seed: int, d: int = D,
                  pool_slots: int = 256, lower_bound: float = LOWER_BOUND,
                  g_mean: float = 0.0, state_std: float = 0.02) -> VerifyInputs:
    """Draw one verify workload.  Draw order: tokens, head params, pool, slot ids."""
    rng = np.random.default_rng(seed)
    q, k, v, g, beta = _token_tensors(rng, B * T, H, d, g_mean)
    A_log, dt_bias = _head_params(rng, H, d)
    pool = rng.standard_normal((pool_slots, H, d, d), dtype=np.float32) * np.float32(state_std)
    slot_ids = rng.permutation(pool_slots)[:B].astype(np.int32)
    return VerifyInputs(
        name=name, q=q, k=k, v=v, g=g, beta=beta, A_log=A_log, dt_bias=dt_bias,
        lower_bound=float(lower_bound), scale=float(1.0 / math.sqrt(d)), B=B, T=T,
        pool=pool, slot_ids=slot_ids, meta={"seed": seed})


@dataclass
class SpecStepInputs:
    """One speculative-decoding step of a layer: a prefill segment and a verify
    segment that share the layer's head parameters and state pool, and the
    output row of every token of either segment."""

    name: str
    prefill: PrefillInputs
    verify: VerifyInputs
    non_spec_token_indx: np.ndarray   # [prefill tokens] int32
    spec_token_indx: np.ndarray       # [B * T] int32
    num_out_tokens: int
    meta: dict = field(default_factory=dict)

    @property
    def H(self) -> int:
        return self.prefill.H


def spec_step_inputs(name: str, prefill_lens, B: int, T: int, H: int, *, seed: int, d: int = D,
                     pool_slots: int | None = None, load_initial: bool = True, final_to_pool: bool = True,
                     order: str = "spec_first", extra_rows: int = 0, lower_bound: float = LOWER_BOUND,
                     g_mean: float = 0.0, state_std: float = 0.02) -> SpecStepInputs:
    """Draw one spec step.  Draw order: prefill tokens, verify tokens, head params,
    pool, slot ids (one permutation: the prefill sequences' slots, then the
    requests'), output rows.

    ``order``: ``"spec_first"`` puts the verify tokens in rows 0 .. B*T-1 and
    the prefill tokens after them (decode requests ahead of prefills in the
    batch); ``"interleaved"`` gives every token a random row.  ``extra_rows``
    output rows belong to no token."""
    prefill_lens = [int(x) for x in prefill_lens]
    rng = np.random.default_rng(seed)
    cu = np.zeros(len(prefill_lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(prefill_lens)
    tp = int(cu[-1])
    pq, pk, pv, pg, pb = _token_tensors(rng, tp, H, d, g_mean)
    sq, sk, sv, sg, sb = _token_tensors(rng, B * T, H, d, g_mean)
    A_log, dt_bias = _head_params(rng, H, d)
    n_slots = pool_slots if pool_slots is not None else len(prefill_lens) + B + 2
    pool = rng.standard_normal((n_slots, H, d, d), dtype=np.float32) * np.float32(state_std)
    perm = rng.permutation(n_slots).astype(np.int32)
    pslots, sslots = perm[:len(prefill_lens)], perm[len(prefill_lens):len(prefill_lens) + B]
    n_out = tp + B * T + extra_rows
    if order == "spec_first":
        rows = np.arange(n_out, dtype=np.int32)
    elif order == "interleaved":
        rows = rng.permutation(n_out).astype(np.int32)
    else:
        raise ValueError(f"unknown order {order!r}")
    scale = float(1.0 / math.sqrt(d))
    pre = PrefillInputs(name=name + ":prefill", q=pq, k=pk, v=pv, g=pg, beta=pb, A_log=A_log, dt_bias=dt_bias,
                        lower_bound=float(lower_bound), scale=scale, cu_seqlens=cu, pool=pool, slot_ids=pslots,
                        load_initial=load_initial, final_to_pool=final_to_pool,
                        meta={"seed": seed, "seq_lens": prefill_lens})
    ver = VerifyInputs(name=name + ":verify", q=sq, k=sk, v=sv, g=sg, beta=sb, A_log=A_log, dt_bias=dt_bias,
                       lower_bound=float(lower_bound), scale=scale, B=B, T=T, pool=pool, slot_ids=sslots,
                       meta={"seed": seed})
    return SpecStepInputs(name=name, prefill=pre, verify=ver, non_spec_token_indx=rows[B * T:B * T + tp].copy(),
                          spec_token_indx=rows[:B * T].copy(), num_out_tokens=n_out,
                          meta={"seed": seed, "order": order})


@dataclass
class NormInputs:
    """Inputs of the sigmoid-gated RMSNorm of the output rows: the bf16 gate
    ``[rows, H, D]`` (bit patterns), the fp32 weight ``[D]`` and eps."""

    gate: np.ndarray
    weight: np.ndarray
    eps: float


def norm_inputs(rows: int, H: int, *, seed: int, d: int = D, eps: float = 1e-6) -> NormInputs:
    """gate ~ N(0, 1) per element (bf16), weight ~ U[0.5, 1.5] per channel."""
    rng = np.random.default_rng(seed)
    gate = f32_to_bf16_bits(rng.standard_normal((rows, H, d), dtype=np.float32))
    weight = rng.uniform(0.5, 1.5, d).astype(np.float32)
    return NormInputs(gate=gate, weight=weight, eps=float(eps))


# ---------------------------------------------------------------------------
# The five named workloads.
# ---------------------------------------------------------------------------

def tiny_prefill() -> PrefillInputs:
    """1 sequence of 256 tokens, H=2, zero initial state, dense final state."""
    return prefill_inputs("prefill_1x256_h2", [256], 2, seed=1000)


def prefill_2048x8() -> PrefillInputs:
    """8 sequences of 2048 tokens, H=16; initial states gathered from a
    64-slot pool by slot id, dense final states."""
    return prefill_inputs("prefill_2048x8_h16", [2048] * 8, 16, seed=1001,
                          pool_slots=64, load_initial=True)


def prefill_8192x4() -> PrefillInputs:
    """4 sequences of 8192 tokens, H=16; zero initial state, final states
    written back to a 64-slot pool."""
    return prefill_inputs("prefill_8192x4_h16", [8192] * 4, 16, seed=1002,
                          pool_slots=64, final_to_pool=True)


def varlen_16384_plus_16(seed: int = 1003) -> PrefillInputs:
    """One 16384-token sequence followed by 16 sequences with lengths drawn
    uniformly from [1, 4096]; H=16, zero initial state, dense final states."""
    rng = np.random.default_rng(seed + 500)
    lens = [16384] + [int(x) for x in rng.integers(1, 4097, size=16)]
    return prefill_inputs("prefill_16384+16varlen_h16", lens, 16, seed=seed)


def verify_64x8() -> VerifyInputs:
    """64 requests x draft block of 8 tokens, H=16, 256-slot pool."""
    return verify_inputs("verify_64x8_h16", 64, 8, 16, seed=1004, pool_slots=256)


def verify_64x4() -> VerifyInputs:
    """64 requests x draft block of 4 tokens (MTP-3: three drafts plus the
    bonus token), H=16, 256-slot pool."""
    return verify_inputs("verify_64x4_h16", 64, 4, 16, seed=1005, pool_slots=256)


def verify_64x1() -> VerifyInputs:
    """64 requests x 1 token (plain decode step), H=16, 256-slot pool."""
    return verify_inputs("verify_64x1_h16", 64, 1, 16, seed=1006, pool_slots=256)


def spec_step_2048x4_64x4() -> SpecStepInputs:
    """One spec step of a layer: a prefill segment of 4 x 2048 tokens (initial
    states from the pool, final states back to it) beside 64 verify requests x
    4 tokens (MTP-3), H=16, 256-slot pool, verify tokens in the first rows."""
    return spec_step_inputs("spec_step_2048x4+64x4_h16", [2048] * 4, 64, 4, 16, seed=1007, pool_slots=256)


NAMED = {
    "prefill_1x256_h2": tiny_prefill,
    "prefill_2048x8_h16": prefill_2048x8,
    "prefill_8192x4_h16": prefill_8192x4,
    "prefill_16384+16varlen_h16": varlen_16384_plus_16,
    "verify_64x8_h16": verify_64x8,
    "verify_64x4_h16": verify_64x4,
    "verify_64x1_h16": verify_64x1,
    "spec_step_2048x4+64x4_h16": spec_step_2048x4_64x4,
}
