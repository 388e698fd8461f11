"""GPU parity of the DAMP-exact storage (INT8 groups of 32 along dv, value
scaling; DAMP Appendix A.1, A.3 Eq. 17-18, A.4): conversion and decode,
bit-exact against the oracle (every byte of the packed tiles, every bit of
o), with seeded log-uniform value-scaling factors."""
import numpy as np
import pytest
import torch

import oracle as orc
import recurrent_state_gb300 as rs
from recurrent_state_gb300 import inputs as gen

from .gpu_util import dev, ensure_built, host, max_rel, same_bits, step_inputs, sub_batch

pytestmark = pytest.mark.gpu

D, KHI, G = 128, 16, 32


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def layouts(Hv, Hk, seed=0):
    hi = gen.hi_rows(Hv, D, KHI, seed=seed)
    cs = gen.value_scales(Hv, D, seed=seed)
    return (rs.Layout("fp32", D, Hv, Hk), rs.Layout("damp", D, Hv, Hk, k_hi=KHI, hi_rows=hi, value_scales=cs),
            orc.row_map(hi, D), cs)


def to_damp_gpu(f32, damp, state0):
    dst = damp.empty_pool(state0.shape[0])
    rs.state_convert(f32, dev(state0), damp, dst, torch.arange(state0.shape[0], dtype=torch.int32, device="cuda"))
    return dst


def test_convert_matches_oracle_both_ways():
    Hv, Hk = 4, 2
    f32, damp, pi, cs = layouts(Hv, Hk, seed=3)
    assert damp.head_bytes == 20224 and damp.bits_per_value() == 9.875
    state0 = gen.random_pool((5, Hv, D, D), seed=3)
    state0[1, 2, 5] = 0.0
    state0[2, 1, 7, 3] = np.float32(2e4)
    g = to_damp_gpu(f32, damp, state0)
    ref = orc.convert_pool_f32_to_damp(state0, KHI, G, pi, cs)
    torch.cuda.synchronize()
    assert same_bits(host(g), ref)
    back = f32.empty_pool(5)
    rs.state_convert(damp, g, f32, back, torch.arange(5, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert same_bits(host(back), orc.convert_pool_damp_to_f32(ref, D, D, KHI, G, pi, cs))


@pytest.mark.parametrize("per_channel", [True, False])
def test_damp_decode_every_tile(per_channel):
    B, Hk, Hv = 97, 4, 8
    f32, damp, pi, cs = layouts(Hv, Hk, seed=5)
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=6, per_channel=per_channel, in_dtype="bf16",
                            seed=5, horizon=(2.0, 8192.0))
    pool = to_damp_gpu(f32, damp, w.state0)
    ref = orc.convert_pool_f32_to_damp(w.state0, KHI, G, pi, cs)
    fn = rs.kda_decode_update if per_channel else rs.gdn_decode_update
    for t in range(w.steps):
        q, k, v, a, b = step_inputs(w, t)
        o = torch.empty((B, Hv, D), device="cuda")
        fn(damp, pool, dev(w.slot_idx), q, k, v, a, b, o=o)
        o_r, st = orc.decode_damp(ref, w.slot_idx, pi, cs, KHI, G, D, D, w.q[t], w.k[t], w.v[t],
                                  w.alpha[t], w.beta[t])
        assert st == 0
        o_g = host(o)
        assert max_rel(o_g, o_r) <= 1e-3
        assert same_bits(o_g, o_r), f"o differs at step {t}"
        assert same_bits(host(pool), ref), f"packed state differs at step {t}"


def test_damp_full_size_sampled():
    """KDA, batch 256, 32 heads, 32 steps; oracle on 4 sampled sequences."""
    B, H = 256, 32
    f32, damp, pi, cs = layouts(H, H, seed=2)
    w = gen.decode_workload(B=B, Hk=H, Hv=H, d=D, steps=32, per_channel=True, in_dtype="bf16", seed=2,
                            horizon=(2.0, 8192.0))
    pool = to_damp_gpu(f32, damp, w.state0)
    slots = dev(w.slot_idx)
    outs = []
    for t in range(32):
        q, k, v, a, b = step_inputs(w, t)
        o = torch.empty((B, H, D), device="cuda")
        rs.kda_decode_update(damp, pool, slots, q, k, v, a, b, o=o)
        outs.append(o)
    torch.cuda.synchronize()
    outs = [host(o) for o in outs]
    bsel = np.array([0, 77, 128, 255])
    ws = sub_batch(w, bsel)
    ref = orc.convert_pool_f32_to_damp(ws.state0, KHI, G, pi, cs)
    for t in range(32):
        o_r, _ = orc.decode_damp(ref, ws.slot_idx, pi, cs, KHI, G, D, D, ws.q[t], ws.k[t], ws.v[t],
                                 ws.alpha[t], ws.beta[t])
        assert same_bits(outs[t][bsel], o_r), t
    assert same_bits(host(pool)[w.slot_idx[bsel]], ref)


def test_damp_small_batch_bad_slots_and_nonfinite():
    B, Hk, Hv = 6, 2, 4
    f32, damp, pi, cs = layouts(Hv, Hk, seed=8)
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=1, per_channel=True, in_dtype="bf16", seed=8,
                            n_slots=9)
    w.slot_idx[2] = 9
    w.slot_idx[4] = -1
    ref = orc.convert_pool_f32_to_damp(w.state0, KHI, G, pi, cs)
    sc0 = 2 * KHI * D + (D - KHI) * D
    s1 = w.slot_idx[1]
    ref[s1, 0, sc0 + 4 * (5 * 4 + 2):sc0 + 4 * (5 * 4 + 2) + 4] = np.array([np.inf], np.float32).view(np.uint8)
    pool = dev(ref)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, k, v, a, b = step_inputs(w, 0)
    o = torch.full((B, Hv, D), 7.0, device="cuda")
    rs.kda_decode_update(damp, pool, dev(w.slot_idx), q, k, v, a, b, o=o, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    oh = host(o)
    assert np.all(oh[[2, 4]] == 7.0)
    ok = np.array([0, 1, 3, 5])
    o_r, st = orc.decode_damp(ref, w.slot_idx[ok], pi, cs, KHI, G, D, D, w.q[0][ok], w.k[0][ok],
                              w.v[0][ok], w.alpha[0][ok], w.beta[0][ok])
    assert st == 0
    g = host(pool)
    hb = 2 * KHI * D
    assert same_bits(g[..., hb:], ref[..., hb:])          # INT8 codes and group scales
    hg, hr = g[..., :hb].copy().view(np.float16), ref[..., :hb].copy().view(np.float16)
    nan = np.isnan(hr)
    assert np.array_equal(np.isnan(hg), nan) and np.array_equal(hg.view(np.uint16)[~nan], hr.view(np.uint16)[~nan])
    og, orr = oh[ok], o_r
    assert np.array_equal(np.isnan(og), np.isnan(orr))
    assert np.array_equal(og[~np.isnan(og)].view(np.uint32), orr[~np.isnan(orr)].view(np.uint32))

