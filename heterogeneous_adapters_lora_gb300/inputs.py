"""Seeded synthetic inputs for the multi-tenant LoRA delta workloads.

This module only *draws* inputs: adapter indices, activations, stacked adapter
weights, per-slot rank/scale tables and (for MoE) the router's top-k choice.
It holds none of the LoRA arithmetic (no shrink, expand, sort or grouping), so
that both the CUDA path and the CPU oracle can consume exactly the same bits.

Conventions
-----------
* Every floating value is drawn in fp32 from numpy's PCG64 and rounded to bf16
  with round-to-nearest-even; arrays of bf16 are carried as ``uint16`` bit
  patterns.  ``bf16_bits_to_f32`` is the exact inverse widening.
* The stacked pool layout follows the vLLM LoRA layer pages
  (``MergedColumnParallelLinearWithLoRA.create_lora_weights``): per output
  slice ``j``, ``A[j]`` is ``[L][R][H]`` and ``B[j]`` is ``[L][O_j][R]``, both
  zero beyond the slot's rank (``set_lora`` copies into ``[:r, :in]`` after
  ``reset_lora``).  MoE pools follow ``FusedMoEWithLoRA._create_lora_a/b_weights``
  with the shared-outer variant of the Inkling PR report (expert dim 1 for
  w13-A and w2-B).
* Named presets reproduce the five benchmark workloads; seed = 1000 + preset
  number.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

# --------------------------------------------------------------------------
# bf16 encoding
# --------------------------------------------------------------------------


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round fp32 values to bf16 (round-to-nearest-even); returns uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 exactly."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, std: float = 0.02) -> np.ndarray:
    v = rng.standard_normal(size=shape, dtype=np.float32)
    v *= np.float32(std)
    return f32_to_bf16_bits(v)


# --------------------------------------------------------------------------
# dense (linear-layer) cases
# --------------------------------------------------------------------------


@dataclass
class DenseCase:
    """One batch for a LoRA-wrapped linear layer with ``len(out_dims)`` packed slices."""

    name: str
    T: int
    H: int
    out_dims: tuple
    L: int
    R: int
    ranks: np.ndarray        # [L] int32, rank of each slot (0 = empty)
    scales: np.ndarray       # [L] float32
    enabled: np.ndarray      # [L] int32 (1 after set_lora, 0 after reset_lora)
    idx: np.ndarray          # [T] int32, -1 = no adapter
    x: np.ndarray            # [T][H] bf16 bits
    A: List[np.ndarray]      # per slice [L][R][H] bf16 bits, rows >= rank zero
    B: List[np.ndarray]      # per slice [L][O_j][R] bf16 bits, cols >= rank zero
    y0: np.ndarray           # [T][sum(out_dims)] bf16 bits (base output)
    W: Optional[np.ndarray] = None   # [sum(out_dims)][H] bf16 base weight (tiny case)
    meta: dict = field(default_factory=dict)

    @property
    def n_slices(self) -> int:
        return len(self.out_dims)

    @property
    def out_total(self) -> int:
        return int(sum(self.out_dims))

    def slot_A(self, j: int, a: int) -> np.ndarray:
        """Checkpoint-layout A of slot ``a``, slice ``j``: ``[rank][H]``."""
        return self.A[j][a, : self.ranks[a], :]

    def slot_B(self, j: int, a: int) -> np.ndarray:
        """Checkpoint-layout B of slot ``a``, slice ``j``: ``[O_j][rank]``."""
        return self.B[j][a, :, : self.ranks[a]]


def _fill_stacked(rng, L, R, rows_per_slot, ranks, std, b_layout: bool):
    """Draw a stacked ``[L][R][X]`` (A) or ``[L][X][R]`` (B) bf16 pool, zero beyond each rank."""
    if b_layout:
        out = np.zeros((L, rows_per_slot, R), dtype=np.uint16)
        for a in range(L):
            r = int(ranks[a])
            if r:
                out[a, :, :r] = _normal_bf16(rng, (rows_per_slot, r), std)
    else:
        out = np.zeros((L, R, rows_per_slot), dtype=np.uint16)
        for a in range(L):
            r = int(ranks[a])
            if r:
                out[a, :r, :] = _normal_bf16(rng, (r, rows_per_slot), std)
    return out


def dense_case(
    *,
    name: str = "custom",
    T: int,
    H: int,
    out_dims: Sequence[int],
    L: int,
    R: int,
    seed: int,
    ranks=None,
    scales=None,
    enabled=None,
    idx=None,
    p_none: float = 0.0,
    base_y: str = "zero",
    with_W: bool = False,
    std: float = 0.02,
) -> DenseCase:
    """Generic seeded dense case.  ``idx`` defaults to uniform over slots with
    probability ``p_none`` of -1; ``ranks`` defaults to ``R`` for every slot."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out_dims = tuple(int(o) for o in out_dims)
    ranks = np.full(L, R, np.int32) if ranks is None else np.asarray(ranks, np.int32)
    scales = np.full(L, 1.0, np.float32) if scales is None else np.asarray(scales, np.float32)
    enabled = (ranks > 0).astype(np.int32) if enabled is None else np.asarray(enabled, np.int32)
    if idx is None:
        idx = rng.integers(0, L, size=T, dtype=np.int64).astype(np.int32)
        if p_none > 0:
            none = rng.random(T) < p_none
            idx[none] = -1
    idx = np.asarray(idx, np.int32)
    x = _normal_bf16(rng, (T, H), std)
    A = [_fill_stacked(rng, L, R, H, ranks, std, b_layout=False) for _ in out_dims]
    B = [_fill_stacked(rng, L, R, o, ranks, std, b_layout=True) for o in out_dims]
    O = sum(out_dims)
    if base_y == "zero":
        y0 = np.zeros((T, O), np.uint16)
    elif base_y == "random":
        y0 = _normal_bf16(rng, (T, O), std)
    else:
        raise ValueError(base_y)
    W = _normal_bf16(rng, (O, H), std) if with_W else None
    return DenseCase(name, T, H, out_dims, L, R, ranks, scales, enabled, idx, x, A, B, y0, W)


# --------------------------------------------------------------------------
# MoE cases
# --------------------------------------------------------------------------


@dataclass
class MoECase:
    """One batch for the fused-MoE LoRA (w13 before the activation, w2 before the top-k sum)."""

    name: str
    T: int
    K: int                   # top_k
    E: int                   # experts
    D: int                   # d_model (hidden)
    F: int                   # d_mlp per expert (w2 input width)
    F13: int                 # width of one w13 slice (F, or 2F for the 3D single-slice layout)
    L: int
    R: int
    shared_outer: bool
    ranks: np.ndarray        # [L] int32
    scales: np.ndarray       # [L] float32
    enabled: np.ndarray      # [L] int32 (adapter_enabled)
    idx: np.ndarray          # [T] int32 token -> slot
    topk_ids: np.ndarray     # [T][K] int32
    topk_w: np.ndarray       # [T][K] float32 routed weights
    x: np.ndarray            # [T][D] bf16 bits (hidden states)
    ic2: np.ndarray          # [T*K][F] bf16 bits (post-activation, w2 input)
    A13: List[np.ndarray]    # per w13 slice [L][E or 1][R][D]
    B13: List[np.ndarray]    # per w13 slice [L][E][F13][R]
    A2: np.ndarray           # [L][E][R][F]
    B2: np.ndarray           # [L][E or 1][D][R]
    ic1_0: np.ndarray        # [T*K][n13*F13] bf16 bits (base pre-activation)
    ic3_0: np.ndarray        # [T*K][D] bf16 bits (base w2 output)
    meta: dict = field(default_factory=dict)

    @property
    def n13(self) -> int:
        return len(self.A13)


def _moe_stack(rng, L, Ex, R, X, ranks, std, b_layout: bool):
    if b_layout:
        out = np.zeros((L, Ex, X, R), np.uint16)
        for a in range(L):
            r = int(ranks[a])
            if r:
                out[a, :, :, :r] = _normal_bf16(rng, (Ex, X, r), std)
    else:
        out = np.zeros((L, Ex, R, X), np.uint16)
        for a in range(L):
            r = int(ranks[a])
            if r:
                out[a, :, :r, :] = _normal_bf16(rng, (Ex, r, X), std)
    return out


def router_topk(rng: np.random.Generator, T: int, E: int, K: int):
    """Top-k routing from softmax of N(0,1) router logits (the base model's
    router, an input of the LoRA path).  Ties go to the lower expert id; the
    selected probabilities are not renormalised."""
    logits = rng.standard_normal((T, E))
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, :K]
    w = np.take_along_axis(p, order, axis=1)
    return order.astype(np.int32), w.astype(np.float32)


def moe_case(
    *,
    name: str = "custom",
    T: int,
    K: int,
    E: int,
    D: int,
    F: int,
    L: int,
    R: int,
    seed: int,
    shared_outer: bool = False,
    n13: int = 2,
    f13: Optional[int] = None,
    ranks=None,
    scales=None,
    enabled=None,
    idx=None,
    p_none: float = 0.0,
    base: str = "zero",
    std: float = 0.02,
) -> MoECase:
    rng = np.random.Generator(np.random.PCG64(seed))
    F13 = F if f13 is None else int(f13)
    ranks = np.full(L, R, np.int32) if ranks is None else np.asarray(ranks, np.int32)
    scales = np.full(L, 1.0, np.float32) if scales is None else np.asarray(scales, np.float32)
    enabled = (ranks > 0).astype(np.int32) if enabled is None else np.asarray(enabled, np.int32)
    topk_ids, topk_w = router_topk(rng, T, E, K)
    if idx is None:
        idx = rng.integers(0, L, size=T, dtype=np.int64).astype(np.int32)
        if p_none > 0:
            idx[rng.random(T) < p_none] = -1
    idx = np.asarray(idx, np.int32)
    x = _normal_bf16(rng, (T, D), std)
    ic2 = _normal_bf16(rng, (T * K, F), std)
    Ea = 1 if shared_outer else E
    A13 = [_moe_stack(rng, L, Ea, R, D, ranks, std, False) for _ in range(n13)]
    B13 = [_moe_stack(rng, L, E, R, F13, ranks, std, True) for _ in range(n13)]
    A2 = _moe_stack(rng, L, E, R, F, ranks, std, False)
    B2 = _moe_stack(rng, L, Ea, R, D, ranks, std, True)
    if base == "zero":
        ic1_0 = np.zeros((T * K, n13 * F13), np.uint16)
        ic3_0 = np.zeros((T * K, D), np.uint16)
    elif base == "random":
        ic1_0 = _normal_bf16(rng, (T * K, n13 * F13), std)
        ic3_0 = _normal_bf16(rng, (T * K, D), std)
    else:
        raise ValueError(base)
    return MoECase(name, T, K, E, D, F, F13, L, R, bool(shared_outer), ranks, scales, enabled,
                   idx, topk_ids, topk_w, x, ic2, A13, B13, A2, B2, ic1_0, ic3_0)


# --------------------------------------------------------------------------
# the five benchmark workloads
# --------------------------------------------------------------------------

PRESETS = {
    1: "tiny",
    2: "decode_qkv",
    3: "prefill_gate_up",
    4: "many_adapter_down",
    5: "moe",
}


def tiny(base_y: str = "zero") -> DenseCase:
    """Single 512 -> 512 projection, T=64, 4 slots of rank 8, scale 2.0,
    idx uniform over {-1, 0, 1, 2, 3}, with a base weight for the merged check."""
    rng = np.random.Generator(np.random.PCG64(1001))
    idx = (rng.integers(0, 5, size=64) - 1).astype(np.int32)
    c = dense_case(name="tiny", T=64, H=512, out_dims=(512,), L=4, R=8, seed=1001 + 7,
                   scales=np.full(4, 2.0, np.float32), idx=idx, base_y=base_y, with_W=True)
    return c


def decode_qkv(base_y: str = "zero", T: int = 256) -> DenseCase:
    """Llama-3-8B packed QKV (4096 -> 4096/1024/1024), one token per request,
    32 slots of rank 16, scale 2.0, idx uniform over 32 slots plus 10% -1."""
    return dense_case(name="decode_qkv", T=T, H=4096, out_dims=(4096, 1024, 1024), L=32, R=16,
                      seed=1002, scales=np.full(32, 2.0, np.float32), p_none=0.1, base_y=base_y)


def prefill_lengths(seed: int = 1003, n_req: int = 8, lo: int = 128, hi: int = 2048) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(lo, hi + 1, size=n_req).astype(np.int32)


def prefill_gate_up(base_y: str = "zero", permuted: bool = False, rank: int = 64) -> DenseCase:
    """gate_up (4096 -> 2 x 14336), 8 requests with lengths uniform in
    [128, 2048] laid out contiguously, request i uses slot i, rank 64 (or
    ``rank``), scale 1.0.  ``permuted`` assigns the slots to requests in a
    shuffled order instead."""
    lens = prefill_lengths()
    slots = np.arange(8, dtype=np.int32)
    if permuted:
        slots = np.random.Generator(np.random.PCG64(2003)).permutation(8).astype(np.int32)
    idx = np.concatenate([np.full(int(n), s, np.int32) for n, s in zip(lens, slots)])
    c = dense_case(name="prefill_gate_up" if rank == 64 else f"prefill_gate_up_r{rank}", T=int(lens.sum()), H=4096,
                   out_dims=(14336, 14336), L=8, R=rank, seed=1003 + 11, idx=idx, base_y=base_y)
    c.meta["lengths"] = lens
    return c


def linear_prefill() -> DenseCase:
    """The prefill gate_up batch as a full LoRA linear layer: base weight
    [28672][4096] ~ N(0, 0.02)."""
    lens = prefill_lengths()
    idx = np.concatenate([np.full(int(n), s, np.int32) for n, s in zip(lens, range(8))])
    c = dense_case(name="linear_prefill", T=int(lens.sum()), H=4096, out_dims=(14336, 14336), L=8, R=64,
                   seed=1104, idx=idx, with_W=True)
    c.meta["lengths"] = lens
    return c


def zipf_pmf(n: int, s: float) -> np.ndarray:
    k = np.arange(1, n + 1, dtype=np.float64)
    p = k ** (-s)
    return p / p.sum()


def many_adapter_down(base_y: str = "zero", T: int = 2048) -> DenseCase:
    """down_proj (14336 -> 4096), 1024 slots with ranks uniform over
    {8, 16, 32, 64} zero-padded to 64, Zipf(1.2) popularity (rank k -> slot
    k-1), T=2048 decode tokens, scale 1.0."""
    rng = np.random.Generator(np.random.PCG64(1004))
    ranks = rng.choice(np.array([8, 16, 32, 64], np.int32), size=1024).astype(np.int32)
    idx = rng.choice(1024, size=T, p=zipf_pmf(1024, 1.2)).astype(np.int32)
    return dense_case(name="many_adapter_down", T=T, H=14336, out_dims=(4096,), L=1024, R=64,
                      seed=1004 + 13, ranks=ranks, idx=idx, base_y=base_y)


def moe(shared_outer: bool = False, base: str = "zero", T: int = 1024) -> MoECase:
    """64 experts, top-8, d_model 2048, d_mlp 1408, rank 16 per (adapter,
    expert), 8 adapters uniform per token, 2 w13 slices (gate, up) + w2."""
    return moe_case(name="moe_shared_outer" if shared_outer else "moe", T=T, K=8, E=64, D=2048,
                    F=1408, L=8, R=16, seed=1005 + (17 if shared_outer else 0),
                    shared_outer=shared_outer, base=base)


def linear_qkv(T: int = 256) -> DenseCase:
    """The decode QKV layer as a full LoRA linear layer: the decode_qkv batch
    with a base weight [6144][4096] ~ N(0, 0.02)."""
    return dense_case(name="linear_qkv", T=T, H=4096, out_dims=(4096, 1024, 1024), L=32, R=16, seed=1102,
                      scales=np.full(32, 2.0, np.float32), p_none=0.1, with_W=True)


class SinkCase:
    """Inkling sink experts around their two LoRA layers: w13 (gate_up, two
    slices of n*d_mlp) and w2 (n*d_mlp -> d_model) share one batch (idx)."""

    def __init__(self, name, w13: DenseCase, w2: DenseCase, n_experts: int, d_mlp: int, gammas: np.ndarray):
        self.name = name
        self.w13 = w13            # y0 = base gate_up (bf16 bits), x = the layer input
        self.w2 = w2              # y0 = base w2 output; x unused (the input is h)
        self.n_experts = n_experts
        self.d_mlp = d_mlp
        self.gammas = gammas      # [T][n_experts] fp32
        self.T = w13.T


def sink_case(*, name="sink", T: int, D: int, n_experts: int, d_mlp: int, L: int, R: int, seed: int,
              p_none: float = 0.1, std: float = 0.1) -> SinkCase:
    """Seeded sink-expert case: x, A, B ~ N(0, std); base gate_up ~ N(0, 1);
    base w2 output ~ N(0, 0.02); gammas uniform in [0.5, 1.5]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    W = n_experts * d_mlp
    idx = rng.integers(0, L, size=T).astype(np.int32)
    idx[rng.random(T) < p_none] = -1
    scales = np.full(L, 2.0, np.float32)
    w13 = dense_case(name=name + "_w13", T=T, H=D, out_dims=(W, W), L=L, R=R, seed=seed + 1, scales=scales,
                     idx=idx, std=std)
    w13.y0 = _normal_bf16(rng, (T, 2 * W), 1.0)
    w2 = dense_case(name=name + "_w2", T=T, H=W, out_dims=(D,), L=L, R=R, seed=seed + 2, scales=scales,
                    idx=idx, std=std)
    w2.y0 = _normal_bf16(rng, (T, D), 0.02)
    gammas = rng.uniform(0.5, 1.5, size=(T, n_experts)).astype(np.float32)
    return SinkCase(name, w13, w2, n_experts, d_mlp, gammas)


def inkling_sink(T: int = 256) -> SinkCase:
    """Sink experts at decode: 256 tokens, d_model 2048, 2 sink experts of
    d_mlp 1408 (gate_up 2048 -> 2 x 2816, w2 2816 -> 2048), 8 slots of rank 16,
    scale 2.0, 10% of tokens without an adapter."""
    return sink_case(name="inkling_sink", T=T, D=2048, n_experts=2, d_mlp=1408, L=8, R=16, seed=1006)


def preset(n: int, **kw):
    return {1: tiny, 2: decode_qkv, 3: prefill_gate_up, 4: many_adapter_down, 5: moe}[n](**kw)
