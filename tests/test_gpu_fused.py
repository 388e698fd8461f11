"""GPU parity of the fused requantisation arithmetic (RS_QUANT_FUSED) of the
mixed layouts: conversion, decode and speculative replay on the one-scale-
per-row layout, and conversion and decode on the DAMP-exact layout (INT8
groups of 32 along dv, value scaling).

Acceptance: the library and the oracle's mode 1 compute the same FP32
values and the same one-rounding codes, so every byte of the packed tiles
and every bit of o must match, step after step (NaN payloads excepted).  The
oracle pins mode 1 against the IEEE-quotient definition separately: its
codes differ only by one and only within the acceptance allowance of a
rounding boundary.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import recurrent_state_gb300 as rs
from recurrent_state_gb300 import inputs as gen

from .gpu_util import (dev, ensure_built, host, max_rel, replay_inputs, same_bits, step_inputs,
                       sub_batch)
from .test_gpu_mixed import adversarial_rows, nan_aware_same

pytestmark = pytest.mark.gpu

D, KHI, G = 128, 16, 32


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def layouts(Hv, Hk, seed=0, kind="mixed"):
    hi = gen.hi_rows(Hv, D, KHI, seed=seed)
    cs = gen.value_scales(Hv, D, seed=seed) if kind == "damp" else None
    lay = rs.Layout(kind, D, Hv, Hk, k_hi=KHI, hi_rows=hi, value_scales=cs, quant="fused")
    return rs.Layout("fp32", D, Hv, Hk), lay, orc.row_map(hi, D), cs


def to_packed_gpu(f32, lay, state0):
    dst = lay.empty_pool(state0.shape[0])
    rs.state_convert(f32, dev(state0), lay, dst,
                     torch.arange(state0.shape[0], dtype=torch.int32, device="cuda"))
    return dst


def test_fused_mode_is_reported_and_fp32_rejects_it():
    f32, lay, _, _ = layouts(4, 4)
    assert lay.quant == "fused"
    with pytest.raises(rs.RsError):
        rs.Layout("fp32", D, 4, 4, quant="fused")


def test_fused_convert_matches_oracle_near_half_integers():
    Hv = 4
    f32, lay, pi, _ = layouts(Hv, Hv, seed=12)
    state = adversarial_rows(3 * Hv, 12).reshape(3, Hv, D, D)
    g = host(to_packed_gpu(f32, lay, state))
    ref = orc.convert_pool_f32_to_mixed(state, KHI, pi, mode=1)
    hb = 2 * KHI * D
    assert same_bits(g[..., hb:], ref[..., hb:])
    hg = g[..., :hb].copy().view(np.float16)
    hr = ref[..., :hb].copy().view(np.float16)
    nan = np.isnan(hr)
    assert np.array_equal(np.isnan(hg), nan)
    assert np.array_equal(hg.view(np.uint16)[~nan], hr.view(np.uint16)[~nan])
    # the adversarial rows do exercise the difference between the two modes
    ieee = orc.convert_pool_f32_to_mixed(state, KHI, pi, mode=0)
    assert not np.array_equal(ieee[..., hb:], ref[..., hb:])


@pytest.mark.parametrize("per_channel,Hk", [(True, 4), (False, 4), (False, 2)])
def test_fused_decode_every_tile(per_channel, Hk):
    B, Hv = 97, 8
    f32, lay, pi, _ = layouts(Hv, Hk, seed=5)
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=6, per_channel=per_channel,
                            in_dtype="bf16", seed=5, horizon=(2.0, 8192.0))
    pool = to_packed_gpu(f32, lay, w.state0)
    ref = orc.convert_pool_f32_to_mixed(w.state0, KHI, pi, mode=1)
    assert same_bits(host(pool), ref)
    fn = rs.kda_decode_update if per_channel else rs.gdn_decode_update
    for t in range(w.steps):
        q, k, v, a, b = step_inputs(w, t)
        o = torch.empty((B, Hv, D), device="cuda")
        fn(lay, pool, dev(w.slot_idx), q, k, v, a, b, o=o)
        o_r, st = orc.decode_mixed(ref, w.slot_idx, pi, KHI, D, D, w.q[t], w.k[t], w.v[t],
                                   w.alpha[t], w.beta[t], mode=1)
        assert st == 0
        o_g = host(o)
        assert max_rel(o_g, o_r) <= 1e-3
        assert same_bits(o_g, o_r), f"o differs at step {t}"
        assert same_bits(host(pool), ref), f"packed state differs at step {t}"


def test_fused_decode_full_size_64_steps_sampled():
    """KDA, batch 256, 32 heads, 64 steps, fused arithmetic; oracle on 4
    sampled sequences (all heads)."""
    B, H = 256, 32
    f32, lay, pi, _ = layouts(H, H, seed=2)
    w = gen.decode_workload(B=B, Hk=H, Hv=H, d=D, steps=64, per_channel=True, in_dtype="bf16",
                            seed=2, horizon=(2.0, 8192.0))
    pool = to_packed_gpu(f32, lay, w.state0)
    slots = dev(w.slot_idx)
    outs = []
    for t in range(64):
        q, k, v, a, b = step_inputs(w, t)
        o = torch.empty((B, H, D), device="cuda")
        rs.kda_decode_update(lay, pool, slots, q, k, v, a, b, o=o)
        outs.append(o)
    torch.cuda.synchronize()
    bsel = np.array([0, 77, 128, 255])
    ws = sub_batch(w, bsel)
    ref = orc.convert_pool_f32_to_mixed(ws.state0, KHI, pi, mode=1)
    for t in range(64):
        o_r, _ = orc.decode_mixed(ref, ws.slot_idx, pi, KHI, D, D, ws.q[t], ws.k[t], ws.v[t],
                                  ws.alpha[t], ws.beta[t], mode=1)
        assert same_bits(host(outs[t])[bsel], o_r), t
    assert same_bits(host(pool)[w.slot_idx[bsel]], ref)


@pytest.mark.parametrize("per_channel", [True, False])
def test_fused_replay_matches_oracle(per_channel):
    B, Hk, Hv, T = 67, 4, 8, 8
    f32, lay, pi, _ = layouts(Hv, Hk, seed=9)
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=T, per_channel=per_channel,
                            in_dtype="bf16", seed=9, horizon=(2.0, 8192.0))
    n_acc = gen.n_accept(B, T, seed=9)
    n_acc[0], n_acc[1], n_acc[2] = 0, T, 1
    qd, kd, vd, ad, bd = replay_inputs(w, T)
    q, k, v, a, b = gen.replay_view(w, T)
    o = torch.full((B, T, Hv, D), 5.0, device="cuda")
    pool = to_packed_gpu(f32, lay, w.state0)
    rs.spec_replay_update(lay, per_channel, pool, dev(w.slot_idx), dev(n_acc), qd, kd, vd, ad, bd, o=o)
    ref = orc.convert_pool_f32_to_mixed(w.state0, KHI, pi, mode=1)
    o_r = np.full((B, T, Hv, D), 5.0, np.float32)
    _, st = orc.replay_mixed(ref, w.slot_idx, n_acc, pi, KHI, D, D, q, k, v, a, b, o=o_r, mode=1)
    torch.cuda.synchronize()
    assert st == 0
    assert same_bits(host(o), o_r)
    assert same_bits(host(pool), ref)


def test_fused_replay_of_one_token_equals_decode():
    B, Hk, Hv = 33, 4, 8
    f32, lay, pi, _ = layouts(Hv, Hk, seed=10)
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=1, per_channel=True, in_dtype="bf16",
                            seed=10, horizon=(2.0, 8192.0))
    p1 = to_packed_gpu(f32, lay, w.state0)
    p2 = p1.clone()
    q, k, v, a, b = step_inputs(w, 0)
    o1 = torch.empty((B, Hv, D), device="cuda")
    rs.kda_decode_update(lay, p1, dev(w.slot_idx), q, k, v, a, b, o=o1)
    qd, kd, vd, ad, bd = replay_inputs(w, 1)
    o2 = torch.empty((B, 1, Hv, D), device="cuda")
    rs.spec_replay_update(lay, True, p2, dev(w.slot_idx), dev(np.ones(B, np.int32)), qd, kd, vd, ad,
                          bd, o=o2)
    torch.cuda.synchronize()
    assert same_bits(host(p1), host(p2))
    assert same_bits(host(o1), host(o2)[:, 0])


def test_fused_decode_nonfinite_state():
    """An infinite INT8 scale and a NaN FP16 value: the rows whose absmax is
    not finite take the IEEE quotient, the others in the same block keep the
    fused product code."""
    B, Hv = 4, 4
    f32, lay, pi, _ = layouts(Hv, Hv, seed=9)
    for per_channel in (True, False):
        w = gen.decode_workload(B=B, Hk=Hv, Hv=Hv, d=D, steps=1, per_channel=per_channel,
                                in_dtype="bf16", seed=9)
        ref = orc.convert_pool_f32_to_mixed(w.state0, KHI, pi, mode=1)
        s0, s1 = w.slot_idx[0], w.slot_idx[1]
        r, c = 3, 10
        off = 2 * (((r // 2) * D + c) * 2 + r % 2)
        ref[s0, 1, off:off + 2] = np.array([0x7E00], np.uint16).view(np.uint8)
        sc = 2 * KHI * D + (D - KHI) * D + 4 * 5
        ref[s1, 0, sc:sc + 4] = np.array([np.inf], np.float32).view(np.uint8)
        pool = dev(ref)
        q, k, v, a, b = step_inputs(w, 0)
        o = torch.empty((B, Hv, D), device="cuda")
        fn = rs.kda_decode_update if per_channel else rs.gdn_decode_update
        fn(lay, pool, dev(w.slot_idx), q, k, v, a, b, o=o)
        o_r, st = orc.decode_mixed(ref, w.slot_idx, pi, KHI, D, D, w.q[0], w.k[0], w.v[0],
                                   w.alpha[0], w.beta[0], mode=1)
        assert st == 0
        assert nan_aware_same(host(o), o_r)
        g = host(pool)
        hb = 2 * KHI * D
        assert same_bits(g[..., hb:], ref[..., hb:])
        hg = g[..., :hb].copy().view(np.float16)
        hr = ref[..., :hb].copy().view(np.float16)
        nan = np.isnan(hr)
        assert np.array_equal(np.isnan(hg), nan)
        assert np.array_equal(hg.view(np.uint16)[~nan], hr.view(np.uint16)[~nan])


# ---- DAMP-exact layout ------------------------------------------------------
def test_damp_fused_convert_matches_oracle():
    Hv, Hk = 4, 2
    f32, lay, pi, cs = layouts(Hv, Hk, seed=3, kind="damp")
    state0 = gen.random_pool((5, Hv, D, D), seed=3)
    state0[1, 2, 5] = 0.0
    state0[2, 1, 7, 3] = np.float32(2e4)
    g = to_packed_gpu(f32, lay, state0)
    torch.cuda.synchronize()
    assert same_bits(host(g), orc.convert_pool_f32_to_damp(state0, KHI, G, pi, cs, mode=1))


@pytest.mark.parametrize("per_channel", [True, False])
def test_damp_fused_decode_every_tile(per_channel):
    B, Hk, Hv = 97, 4, 8
    f32, lay, pi, cs = layouts(Hv, Hk, seed=5, kind="damp")
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=5, per_channel=per_channel, in_dtype="bf16",
                            seed=5, horizon=(2.0, 8192.0))
    pool = to_packed_gpu(f32, lay, w.state0)
    ref = orc.convert_pool_f32_to_damp(w.state0, KHI, G, pi, cs, mode=1)
    fn = rs.kda_decode_update if per_channel else rs.gdn_decode_update
    for t in range(w.steps):
        q, k, v, a, b = step_inputs(w, t)
        o = torch.empty((B, Hv, D), device="cuda")
        fn(lay, pool, dev(w.slot_idx), q, k, v, a, b, o=o)
        o_r, st = orc.decode_damp(ref, w.slot_idx, pi, cs, KHI, G, D, D, w.q[t], w.k[t], w.v[t],
                                  w.alpha[t], w.beta[t], mode=1)
        assert st == 0
        o_g = host(o)
        assert max_rel(o_g, o_r) <= 1e-3
        assert same_bits(o_g, o_r), f"o differs at step {t}"
        assert same_bits(host(pool), ref), f"packed state differs at step {t}"
