"""GPU parity of prefill chunks (DAMP Appendix A.4 "Prefill path": FP32
arithmetic within each chunk, the final state written to the same packed
cache).

The oracle of a chunk is the multi-token replay: every token one decode step
in FP32, the state dequantised once and requantised once.  The library must
match it bit for bit (every byte of the pool, every bit of o), for chunks
longer than the replay window, ragged per-sequence token counts (0 and L
included), GDN and KDA, FP32 and mixed layouts in both requantisation modes.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import recurrent_state_gb300 as rs
from recurrent_state_gb300 import inputs as gen

from .gpu_util import dev, ensure_built, host, replay_inputs, same_bits, sub_batch

pytestmark = pytest.mark.gpu

D, KHI = 128, 16


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def mixed_layout(Hv, Hk, seed, quant):
    hi = gen.hi_rows(Hv, D, KHI, seed=seed)
    return rs.Layout("mixed", D, Hv, Hk, k_hi=KHI, hi_rows=hi, quant=quant), orc.row_map(hi, D)


def to_mixed(f32, lay, state0):
    dst = lay.empty_pool(state0.shape[0])
    rs.state_convert(f32, dev(state0), lay, dst,
                     torch.arange(state0.shape[0], dtype=torch.int32, device="cuda"))
    return dst


@pytest.mark.parametrize("kind", ["fp32", "ieee", "fused"])
@pytest.mark.parametrize("per_channel", [True, False])
def test_prefill_chunk_matches_oracle(kind, per_channel):
    B, Hk, Hv, L = 13, 4, 8, 37
    seed = 40 + (kind == "ieee") + 2 * (kind == "fused")
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=L, per_channel=per_channel,
                            in_dtype="bf16", seed=seed, horizon=(2.0, 8192.0))
    n_tok = gen.rng(seed).integers(1, L + 1, B).astype(np.int32)
    n_tok[0], n_tok[1], n_tok[2] = 0, L, 1
    qd, kd, vd, ad, bd = replay_inputs(w, L)
    q, k, v, a, b = gen.replay_view(w, L)
    o = torch.full((B, L, Hv, D), 3.0, device="cuda")
    o_r = np.full((B, L, Hv, D), 3.0, np.float32)
    f32 = rs.Layout("fp32", D, Hv, Hk)
    if kind == "fp32":
        pool = dev(w.state0)
        rs.prefill_update(f32, per_channel, pool, dev(w.slot_idx), qd, kd, vd, ad, bd, n_tokens=dev(n_tok), o=o)
        ref = w.state0.copy()
        _, st = orc.replay_f32(ref, w.slot_idx, n_tok, q, k, v, a, b, o=o_r)
    else:
        mode = 1 if kind == "fused" else 0
        lay, pi = mixed_layout(Hv, Hk, seed, kind)
        pool = to_mixed(f32, lay, w.state0)
        rs.prefill_update(lay, per_channel, pool, dev(w.slot_idx), qd, kd, vd, ad, bd, n_tokens=dev(n_tok), o=o)
        ref = orc.convert_pool_f32_to_mixed(w.state0, KHI, pi, mode=mode)
        _, st = orc.replay_mixed(ref, w.slot_idx, n_tok, pi, KHI, D, D, q, k, v, a, b, o=o_r, mode=mode)
    torch.cuda.synchronize()
    assert st == 0
    assert same_bits(host(o), o_r)
    assert same_bits(host(pool), ref)


def test_prefill_fp32_equals_decode_steps_f32_inputs():
    """FP32 inputs, every sequence the full chunk (n_tokens omitted): the
    chunk equals L decode calls bit for bit."""
    B, Hk, Hv, L = 9, 2, 4, 11
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=L, per_channel=True, in_dtype="f32", seed=50)
    f32 = rs.Layout("fp32", D, Hv, Hk)
    p1 = dev(w.state0)
    p2 = p1.clone()
    qd, kd, vd, ad, bd = replay_inputs(w, L)
    o1 = torch.empty((B, L, Hv, D), device="cuda")
    rs.prefill_update(f32, True, p1, dev(w.slot_idx), qd, kd, vd, ad, bd, o=o1)
    slots = dev(w.slot_idx)
    outs = []
    for t in range(L):
        o = torch.empty((B, Hv, D), device="cuda")
        rs.kda_decode_update(f32, p2, slots, dev(w.q[t]), dev(w.k[t]), dev(w.v[t]), dev(w.alpha[t]),
                             dev(w.beta[t]), o=o)
        outs.append(o)
    torch.cuda.synchronize()
    assert same_bits(host(p1), host(p2))
    assert same_bits(host(o1), np.stack([host(x) for x in outs], axis=1))


def test_prefill_full_size_sampled():
    """KDA, batch 256, 32 heads, mixed layout with the fused arithmetic, a
    chunk of 64 tokens; oracle on 3 sampled sequences."""
    B, H, L = 256, 32, 64
    w = gen.decode_workload(B=B, Hk=H, Hv=H, d=D, steps=L, per_channel=True, in_dtype="bf16",
                            seed=51, horizon=(2.0, 8192.0))
    f32 = rs.Layout("fp32", D, H, H)
    lay, pi = mixed_layout(H, H, 51, "fused")
    pool = to_mixed(f32, lay, w.state0)
    qd, kd, vd, ad, bd = replay_inputs(w, L)
    o = torch.empty((B, L, H, D), device="cuda")
    rs.prefill_update(lay, True, pool, dev(w.slot_idx), qd, kd, vd, ad, bd, o=o)
    torch.cuda.synchronize()
    bsel = np.array([5, 130, 255])
    ws = sub_batch(w, bsel)
    q, k, v, a, b = gen.replay_view(ws, L)
    ref = orc.convert_pool_f32_to_mixed(ws.state0, KHI, pi, mode=1)
    o_r = np.zeros((len(bsel), L, H, D), np.float32)
    _, st = orc.replay_mixed(ref, ws.slot_idx, np.full(len(bsel), L, np.int32), pi, KHI, D, D,
                             q, k, v, a, b, o=o_r, mode=1)
    assert st == 0
    assert same_bits(host(o)[bsel], o_r)
    assert same_bits(host(pool)[w.slot_idx[bsel]], ref)


def test_prefill_bad_slot_and_count_reported():
    B, Hk, Hv, L = 4, 2, 4, 5
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=L, per_channel=False, in_dtype="bf16", seed=52,
                            n_slots=6)
    w.slot_idx[1] = 6
    n_tok = np.array([L, 2, L + 1, -1], np.int32)
    f32 = rs.Layout("fp32", D, Hv, Hk)
    pool = dev(w.state0)
    before = host(pool)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qd, kd, vd, ad, bd = replay_inputs(w, L)
    rs.prefill_update(f32, False, pool, dev(w.slot_idx), qd, kd, vd, ad, bd, n_tokens=dev(n_tok),
                      status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1 | 2
    after = host(pool)
    for bb in (2, 3):
        assert same_bits(after[w.slot_idx[bb]], before[w.slot_idx[bb]])
    ref = w.state0.copy()
    q, k, v, a, b = gen.replay_view(w, L)
    orc.replay_f32(ref, w.slot_idx[:1], n_tok[:1], q[:1], k[:1], v[:1], a[:1], b[:1])
    assert same_bits(after[w.slot_idx[0]], ref[w.slot_idx[0]])


@pytest.mark.parametrize("quant", ["ieee", "fused"])
@pytest.mark.parametrize("per_channel", [True, False])
def test_prefill_and_replay_on_damp_layout(quant, per_channel):
    """DAMP-exact layout (INT8 groups of 32, value scaling): a prefill chunk
    and a speculative replay both match the oracle's DAMP replay bit for bit."""
    B, Hk, Hv, L, G = 11, 2, 4, 19, 32
    seed = 60 + (quant == "fused")
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=L, per_channel=per_channel,
                            in_dtype="bf16", seed=seed, horizon=(2.0, 8192.0))
    hi = gen.hi_rows(Hv, D, KHI, seed=seed)
    pi = orc.row_map(hi, D)
    cs = gen.value_scales(Hv, D, seed=seed)
    lay = rs.Layout("damp", D, Hv, Hk, k_hi=KHI, hi_rows=hi, value_scales=cs, quant=quant)
    f32 = rs.Layout("fp32", D, Hv, Hk)
    mode = 1 if quant == "fused" else 0
    n_tok = gen.rng(seed).integers(1, L + 1, B).astype(np.int32)
    n_tok[0], n_tok[1] = 0, L
    qd, kd, vd, ad, bd = replay_inputs(w, L)
    q, k, v, a, b = gen.replay_view(w, L)
    pool = to_mixed(f32, lay, w.state0)
    o = torch.full((B, L, Hv, D), 2.0, device="cuda")
    rs.prefill_update(lay, per_channel, pool, dev(w.slot_idx), qd, kd, vd, ad, bd, n_tokens=dev(n_tok), o=o)
    ref = orc.convert_pool_f32_to_damp(w.state0, KHI, G, pi, cs, mode=mode)
    o_r = np.full((B, L, Hv, D), 2.0, np.float32)
    _, st = orc.replay_damp(ref, w.slot_idx, n_tok, pi, cs, KHI, G, D, D, q, k, v, a, b, o=o_r, mode=mode)
    torch.cuda.synchronize()
    assert st == 0
    assert same_bits(host(o), o_r)
    assert same_bits(host(pool), ref)
    # replay of up to 8 logged tokens on the same layout
    T = 8
    n_acc = np.minimum(n_tok, T).astype(np.int32)
    qd, kd, vd, ad, bd = replay_inputs(w, T)
    q, k, v, a, b = gen.replay_view(w, T)
    o2 = torch.full((B, T, Hv, D), 2.0, device="cuda")
    rs.spec_replay_update(lay, per_channel, pool, dev(w.slot_idx), dev(n_acc), qd, kd, vd, ad, bd, o=o2)
    o2_r = np.full((B, T, Hv, D), 2.0, np.float32)
    _, st = orc.replay_damp(ref, w.slot_idx, n_acc, pi, cs, KHI, G, D, D, q, k, v, a, b, o=o2_r, mode=mode)
    torch.cuda.synchronize()
    assert st == 0
    assert same_bits(host(o2), o2_r)
    assert same_bits(host(pool), ref)
