"""Helpers shared by the GPU parity tests: move seeded numpy workloads to the
device in the dtype the library consumes, run decode steps through the C ABI,
and compare results with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import recurrent_state_gb300 as rs
from recurrent_state_gb300 import build as rsbuild
from recurrent_state_gb300 import inputs as gen

_built = False


def ensure_built():
    global _built
    if not _built:
        rsbuild.build()
        _built = True


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_f16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.float16)).cuda()


def dev_in(w: gen.DecodeInputs, bits: np.ndarray, values: np.ndarray) -> torch.Tensor:
    """A q, k or v tensor in the workload's input dtype."""
    if w.in_dtype == "bf16":
        return dev_bf16(bits)
    if w.in_dtype == "f16":
        return dev_f16(bits)
    return dev(values)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def step_inputs(w: gen.DecodeInputs, t: int):
    """Device tensors (q, k, v, alpha, beta) for decode step t."""
    if w.in_dtype in ("bf16", "f16"):
        q, k, v = (dev_in(w, b[t], None) for b in (w.q_bits, w.k_bits, w.v_bits))
    else:
        q, k, v = dev(w.q[t]), dev(w.k[t]), dev(w.v[t])
    return q, k, v, dev(w.alpha[t]), dev(w.beta[t])


def replay_inputs(w: gen.DecodeInputs, T_max: int):
    """Device tensors [B][T_max][...] from the first T_max steps."""
    def bt(x):
        return np.ascontiguousarray(np.swapaxes(x[:T_max], 0, 1))
    if w.in_dtype in ("bf16", "f16"):
        q, k, v = (dev_in(w, bt(b), None) for b in (w.q_bits, w.k_bits, w.v_bits))
    else:
        q, k, v = dev(bt(w.q)), dev(bt(w.k)), dev(bt(w.v))
    return q, k, v, dev(bt(w.alpha)), dev(bt(w.beta))


def same_bits(a: np.ndarray, b: np.ndarray) -> bool:
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    return a.shape == b.shape and np.array_equal(a.view(np.uint8), b.view(np.uint8))


def same_bits_nan(a: np.ndarray, b: np.ndarray) -> bool:
    """Bit equality of float32 arrays, except that a NaN only has to meet a
    NaN: the payload of a NaN produced by arithmetic (0 * inf) is the
    hardware's and not part of the result."""
    a = np.ascontiguousarray(a, np.float32)
    b = np.ascontiguousarray(b, np.float32)
    if a.shape != b.shape:
        return False
    na, nb = np.isnan(a), np.isnan(b)
    return np.array_equal(na, nb) and np.array_equal(a[~na].view(np.uint32), b[~nb].view(np.uint32))


def max_rel(x: np.ndarray, ref: np.ndarray) -> float:
    """max over tiles of ||x - ref||_inf / ||ref||_inf, tiles = last two axes
    (or the last axis for vectors)."""
    x = x.astype(np.float64)
    ref = ref.astype(np.float64)
    axes = tuple(range(x.ndim - 2, x.ndim)) if x.ndim >= 3 else (x.ndim - 1,)
    num = np.max(np.abs(x - ref), axis=axes)
    den = np.maximum(np.max(np.abs(ref), axis=axes), 1e-30)
    return float(np.max(num / den))


def sub_batch(w: gen.DecodeInputs, bsel: np.ndarray):
    """Restrict a workload to batch entries ``bsel`` (all heads of each), for
    oracle runs on sampled items of a full-size GPU run."""
    def take(x):
        return None if x is None else np.ascontiguousarray(x[:, bsel])
    out = gen.DecodeInputs(B=len(bsel), Hk=w.Hk, Hv=w.Hv, dk=w.dk, dv=w.dv, steps=w.steps,
                           per_channel=w.per_channel, in_dtype=w.in_dtype,
                           q=take(w.q), k=take(w.k), v=take(w.v), alpha=take(w.alpha),
                           beta=take(w.beta), state0=np.ascontiguousarray(w.state0[w.slot_idx[bsel]]),
                           slot_idx=np.arange(len(bsel), dtype=np.int32))
    return out
