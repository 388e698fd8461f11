"""Seeded synthetic inputs for the recurrent-state hot path.

This module holds only the input recipe: random draws, the L2 normalisation of
q and k that the model applies upstream of the recurrence, bf16 rounding of
the model's activations, and the decay/strength gates that produce alpha and
beta.  It holds none of the recurrence, quantisation or checkpoint arithmetic,
so the CUDA path and the CPU oracle can both consume its arrays byte for byte.

Everything is numpy (PCG64), so the same seed gives the same bytes on every
host.  Activations meant to be bf16 are returned as uint16 bit patterns plus
their exact float32 widening.

Workload shapes follow the pages' models (the pages themselves are cited in
the library header): GDN with 16 qk heads shared by 32 value heads
(Qwen3-Next-like), KDA with 32 heads (Kimi-Linear-like), dk = dv = 128.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


# --------------------------------------------------------------------------
# primitives
# --------------------------------------------------------------------------
def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    bias = ((u >> 16) & 1) + 0x7FFF
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def l2_normalise(x: np.ndarray) -> np.ndarray:
    """Per-head L2 normalisation over the last axis (done upstream by the model)."""
    x = x.astype(np.float32)
    n = np.sqrt(np.sum(x.astype(np.float64) ** 2, axis=-1, keepdims=True))
    return (x / np.maximum(n, 1e-30)).astype(np.float32)


def sigmoid(x):
    return (1.0 / (1.0 + np.exp(-x.astype(np.float64)))).astype(np.float32)


def softplus(x):
    x = x.astype(np.float64)
    return np.where(x > 20, x, np.log1p(np.exp(np.minimum(x, 20))))


def log_uniform(g: np.random.Generator, lo: float, hi: float, size) -> np.ndarray:
    return np.exp(g.uniform(np.log(lo), np.log(hi), size=size))


# --------------------------------------------------------------------------
# decode / replay workloads
# --------------------------------------------------------------------------
@dataclass
class DecodeInputs:
    """All steps of one decode workload, laid out step-major.

    q, k: [steps][B][Hk][dk]; v: [steps][B][Hv][dv]; alpha: [steps][B][Hv] (GDN)
    or [steps][B][Hv][dk] (KDA); beta: [steps][B][Hv].  ``*_bits`` hold the
    bf16 bit patterns when ``in_dtype == 'bf16'``; the float32 arrays are then
    their exact widening.  state0: [n_slots][Hv][dk][dv] float32.
    """
    B: int
    Hk: int
    Hv: int
    dk: int
    dv: int
    steps: int
    per_channel: bool
    in_dtype: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    alpha: np.ndarray
    beta: np.ndarray
    state0: np.ndarray
    slot_idx: np.ndarray
    q_bits: np.ndarray | None = None
    k_bits: np.ndarray | None = None
    v_bits: np.ndarray | None = None
    extra: dict = field(default_factory=dict)


def _qkv(g, steps, B, Hk, Hv, dk, dv, in_dtype):
    q = l2_normalise(g.standard_normal((steps, B, Hk, dk), dtype=np.float32))
    k = l2_normalise(g.standard_normal((steps, B, Hk, dk), dtype=np.float32))
    v = g.standard_normal((steps, B, Hv, dv), dtype=np.float32)
    if in_dtype == "bf16":
        qb, kb, vb = bf16_bits(q), bf16_bits(k), bf16_bits(v)
        return bf16_to_f32(qb), bf16_to_f32(kb), bf16_to_f32(vb), qb, kb, vb
    if in_dtype == "f16":  # IEEE half, nearest even; the widened values are what both sides see
        qh, kh, vh = (x.astype(np.float16) for x in (q, k, v))
        return (qh.astype(np.float32), kh.astype(np.float32), vh.astype(np.float32),
                qh.view(np.uint16), kh.view(np.uint16), vh.view(np.uint16))
    return q, k, v, None, None, None


def decode_workload(*, B, Hk, Hv, d, steps, per_channel, in_dtype="bf16", seed=0,
                    horizon=(4.0, 4096.0), tiny_gdn=False, n_slots=None,
                    state_std=0.1) -> DecodeInputs:
    """Synthetic decode workload.

    GDN (per_channel=False): alpha[b,t,h] = exp(-softplus(N(0,1)) / h_h) with
    h_h log-uniform over ``horizon`` per head; with ``tiny_gdn`` the decay is
    exp(-1/h_h), fixed over batch and steps.  KDA (per_channel=True):
    alpha[b,t,h,c] = exp(-softplus(N(0,1)) / h_{h,c}) with h_{h,c} log-uniform
    over ``horizon`` per key channel.  beta = sigmoid(N(0,1)).
    State: N(0, state_std) float32.  Slots: a seeded permutation of n_slots.
    """
    g = rng(seed)
    dk = dv = d
    n_slots = B if n_slots is None else n_slots
    state0 = (g.standard_normal((n_slots, Hv, dk, dv), dtype=np.float32)
              * np.float32(state_std)).astype(np.float32)
    slot_idx = g.permutation(n_slots)[:B].astype(np.int32)
    q, k, v, qb, kb, vb = _qkv(g, steps, B, Hk, Hv, dk, dv, in_dtype)
    if per_channel:
        hor = log_uniform(g, horizon[0], horizon[1], (Hv, dk))
        z = g.standard_normal((steps, B, Hv, dk))
        alpha = np.exp(-softplus(z) / hor[None, None]).astype(np.float32)
    elif tiny_gdn:
        hor = log_uniform(g, horizon[0], horizon[1], (Hv,))
        a_h = np.exp(-1.0 / hor).astype(np.float32)
        alpha = np.broadcast_to(a_h, (steps, B, Hv)).astype(np.float32).copy()
    else:
        hor = log_uniform(g, horizon[0], horizon[1], (Hv,))
        z = g.standard_normal((steps, B, Hv))
        alpha = np.exp(-softplus(z) / hor[None, None]).astype(np.float32)
    beta = sigmoid(g.standard_normal((steps, B, Hv)))
    return DecodeInputs(B=B, Hk=Hk, Hv=Hv, dk=dk, dv=dv, steps=steps,
                        per_channel=per_channel, in_dtype=in_dtype, q=q, k=k, v=v,
                        alpha=alpha, beta=beta, state0=state0, slot_idx=slot_idx,
                        q_bits=qb, k_bits=kb, v_bits=vb, extra={"horizon": hor})


def hi_rows(Hv: int, dk: int, k_hi: int, seed: int = 0) -> np.ndarray:
    """Seeded per-head list of ``k_hi`` high-precision key channels, ascending.
    Stands in for the offline selection; returns int16 [Hv][k_hi]."""
    g = rng(seed + 7919)
    return np.stack([np.sort(g.permutation(dk)[:k_hi]) for _ in range(Hv)]).astype(np.int16)


def n_accept(B: int, T_max: int, seed: int = 0, lo: int = 1) -> np.ndarray:
    """Accepted draft tokens per sequence, uniform over {lo..T_max}."""
    return rng(seed + 104729).integers(lo, T_max + 1, size=B).astype(np.int32)


def replay_view(w: DecodeInputs, T_max: int):
    """Reshape the first T_max steps into [B][T_max][...] replay inputs."""
    def bt(x):
        return np.ascontiguousarray(np.swapaxes(x[:T_max], 0, 1))
    return bt(w.q), bt(w.k), bt(w.v), bt(w.alpha), bt(w.beta)


# --------------------------------------------------------------------------
# checkpoint workloads
# --------------------------------------------------------------------------
def keep_mask(L: int, n_units: int, p: float, seed: int = 0) -> np.ndarray:
    """Independent Bernoulli(p) retention per unit: uint8 [L][n_units]."""
    return (rng(seed + 65537).random((L, n_units)) < p).astype(np.uint8)


def ckpt_slots(n_pool_slots: int, n: int, seed: int = 0):
    """A seeded permuted order of source pool slots and of checkpoint slots."""
    g = rng(seed + 31337)
    return (g.permutation(n_pool_slots)[:n].astype(np.int32),
            g.permutation(n)[:n].astype(np.int32))


def random_pool(shape, seed: int = 0, std: float = 0.1) -> np.ndarray:
    g = rng(seed + 17)
    return (g.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def value_scales(Hv: int, dv: int, seed: int = 0, group: int = 0, pow2: bool = False) -> np.ndarray:
    """Value-scaling factors c' > 0 per (head, value dimension), float32
    [Hv][dv] (DAMP Appendix A.1 "Value scaling and reordering", calibrated
    offline; synthetic here): log-uniform in [1/4, 4], or, with ``pow2``, one
    power of two 2^k (k in -3..3) per group of ``group`` consecutive values."""
    g = rng(seed + 4099)
    if pow2:
        k = g.integers(-3, 4, (Hv, dv // group))
        return np.repeat(np.ldexp(np.float32(1.0), k).astype(np.float32), group, axis=1)
    return np.exp(g.uniform(np.log(0.25), np.log(4.0), (Hv, dv))).astype(np.float32)
