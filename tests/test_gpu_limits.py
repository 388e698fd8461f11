"""GPU parity at the largest layouts the library takes.

The mixed layout's row map travels in the launch parameters (up to 8,192
bytes: 64 value heads at dk = 128) and the DAMP-exact layout's value-scaling
factors too (up to 4,096 floats: 32 heads at dv = 128).  At those limits the
shared-memory header of every kernel is largest and its stage ring shortest.
Decode (both requantisation modes), replay and prefill must still equal the
oracle bit for bit, with grouped-query heads (8 value heads per key head).
"""
import numpy as np
import pytest
import torch

import oracle as orc
import recurrent_state_gb300 as rs
from recurrent_state_gb300 import inputs as gen

from .gpu_util import dev, ensure_built, host, replay_inputs, same_bits, step_inputs

pytestmark = pytest.mark.gpu

D, KHI, G = 128, 16, 32


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def to_packed(lay, state0, Hv, Hk):
    f32 = rs.Layout("fp32", D, Hv, Hk)
    dst = lay.empty_pool(state0.shape[0])
    rs.state_convert(f32, dev(state0), lay, dst, torch.arange(state0.shape[0], dtype=torch.int32, device="cuda"))
    return dst


def layout(kind, Hv, Hk, seed, quant):
    hi = gen.hi_rows(Hv, D, KHI, seed=seed)
    cs = gen.value_scales(Hv, D, seed=seed) if kind == "damp" else None
    return rs.Layout(kind, D, Hv, Hk, k_hi=KHI, hi_rows=hi, value_scales=cs, quant=quant), orc.row_map(hi, D), cs


def oracle_pool(kind, state0, pi, cs, mode):
    if kind == "damp":
        return orc.convert_pool_f32_to_damp(state0, KHI, G, pi, cs, mode=mode)
    return orc.convert_pool_f32_to_mixed(state0, KHI, pi, mode=mode)


MAX_HEADS = {"mixed": (64, 8), "damp": (32, 4)}


@pytest.mark.parametrize("kind,quant", [("mixed", "ieee"), ("mixed", "fused"), ("damp", "fused")])
def test_decode_at_the_largest_layout(kind, quant):
    Hv, Hk = MAX_HEADS[kind]
    B, steps, seed = 5, 2, 64
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=steps, per_channel=True, in_dtype="bf16", seed=seed,
                            horizon=(2.0, 8192.0))
    lay, pi, cs = layout(kind, Hv, Hk, seed, quant)
    mode = 1 if quant == "fused" else 0
    pool = to_packed(lay, w.state0, Hv, Hk)
    ref = oracle_pool(kind, w.state0, pi, cs, mode)
    assert same_bits(host(pool), ref)
    for t in range(steps):
        q, k, v, a, b = step_inputs(w, t)
        o = torch.empty((B, Hv, D), device="cuda")
        rs.kda_decode_update(lay, pool, dev(w.slot_idx), q, k, v, a, b, o=o)
        if kind == "damp":
            o_r, _ = orc.decode_damp(ref, w.slot_idx, pi, cs, KHI, G, D, D, w.q[t], w.k[t], w.v[t],
                                     w.alpha[t], w.beta[t], mode=mode)
        else:
            o_r, _ = orc.decode_mixed(ref, w.slot_idx, pi, KHI, D, D, w.q[t], w.k[t], w.v[t],
                                      w.alpha[t], w.beta[t], mode=mode)
        torch.cuda.synchronize()
        assert same_bits(host(o), o_r), t
        assert same_bits(host(pool), ref), t


@pytest.mark.parametrize("kind,path", [("mixed", "replay"), ("mixed", "prefill"), ("damp", "replay")])
def test_multi_token_at_the_largest_layout(kind, path):
    Hv, Hk = MAX_HEADS[kind]
    B, T, seed = 4, 8, 65
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=T, per_channel=False, in_dtype="bf16", seed=seed,
                            horizon=(2.0, 8192.0))
    lay, pi, cs = layout(kind, Hv, Hk, seed, "fused")
    pool = to_packed(lay, w.state0, Hv, Hk)
    ref = oracle_pool(kind, w.state0, pi, cs, 1)
    n_tok = gen.rng(seed).integers(1, T + 1, B).astype(np.int32)
    qd, kd, vd, ad, bd = replay_inputs(w, T)
    q, k, v, a, b = gen.replay_view(w, T)
    o = torch.zeros((B, T, Hv, D), device="cuda")
    o_r = np.zeros((B, T, Hv, D), np.float32)
    if path == "replay":
        rs.spec_replay_update(lay, False, pool, dev(w.slot_idx), dev(n_tok), qd, kd, vd, ad, bd, o=o)
    else:
        rs.prefill_update(lay, False, pool, dev(w.slot_idx), qd, kd, vd, ad, bd, n_tokens=dev(n_tok), o=o)
    if kind == "damp":
        orc.replay_damp(ref, w.slot_idx, n_tok, pi, cs, KHI, G, D, D, q, k, v, a, b, o=o_r, mode=1)
    else:
        orc.replay_mixed(ref, w.slot_idx, n_tok, pi, KHI, D, D, q, k, v, a, b, o=o_r, mode=1)
    torch.cuda.synchronize()
    assert same_bits(host(o), o_r)
    assert same_bits(host(pool), ref)
