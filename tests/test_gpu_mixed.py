"""GPU parity of the mixed FP16/INT8 state path and of speculative replay.

Acceptance: INT8 codes, FP16 rows and scales bit-exact against the oracle
(codes may differ by one where the FP32 value before quantisation lies within
1e-6 of a rounding boundary); readout o within 1e-3 of the oracle that runs
the same quantisation.  The library computes the same FP32 values as the
oracle, so the tests require every byte of the packed tiles and every bit of
o to match, step after step, which implies both bars.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import recurrent_state_gb300 as rs
from recurrent_state_gb300 import inputs as gen

from .gpu_util import (dev, ensure_built, host, max_rel, replay_inputs, same_bits, step_inputs,
                       sub_batch)

pytestmark = pytest.mark.gpu

D, KHI = 128, 16


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def layouts(Hv, Hk, seed=0):
    hi = gen.hi_rows(Hv, D, KHI, seed=seed)
    return (rs.Layout("fp32", D, Hv, Hk), rs.Layout("mixed", D, Hv, Hk, k_hi=KHI, hi_rows=hi),
            orc.row_map(hi, D))


def to_mixed_gpu(f32_lay, mix_lay, state0):
    src = dev(state0)
    dst = mix_lay.empty_pool(state0.shape[0])
    slots = torch.arange(state0.shape[0], dtype=torch.int32, device="cuda")
    rs.state_convert(f32_lay, src, mix_lay, dst, slots)
    return dst


def test_convert_matches_oracle_both_ways():
    Hv, Hk = 8, 4
    f32, mix, pi = layouts(Hv, Hk, seed=3)
    state0 = gen.random_pool((5, Hv, D, D), seed=3)
    state0[1, 2, 5] = 0.0                     # an all-zero row: the scale floor
    state0[2, 1, 7, 3] = np.float32(2e4)      # a row with one outlier
    g = to_mixed_gpu(f32, mix, state0)
    ref = orc.convert_pool_f32_to_mixed(state0, KHI, pi)
    assert same_bits(host(g), ref)
    back = f32.empty_pool(5)
    rs.state_convert(mix, g, f32, back, torch.arange(5, dtype=torch.int32, device="cuda"))
    assert same_bits(host(back), orc.convert_pool_mixed_to_f32(ref, D, D, KHI, pi))


def mixed_gpu_steps(w, mix, pool, steps):
    slots = dev(w.slot_idx)
    fn = rs.kda_decode_update if w.per_channel else rs.gdn_decode_update
    outs = []
    for t in range(steps):
        q, k, v, a, b = step_inputs(w, t)
        o = torch.empty((w.B, w.Hv, D), device="cuda")
        fn(mix, pool, slots, q, k, v, a, b, o=o)
        outs.append(o)
    torch.cuda.synchronize()
    return [host(o) for o in outs]


@pytest.mark.parametrize("per_channel", [True, False])
def test_mixed_decode_every_tile(per_channel):
    B, Hk, Hv = 97, 4, 8
    f32, mix, pi = layouts(Hv, Hk, seed=5)
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=6, per_channel=per_channel,
                            in_dtype="bf16", seed=5, horizon=(2.0, 8192.0))
    pool = to_mixed_gpu(f32, mix, w.state0)
    ref = orc.convert_pool_f32_to_mixed(w.state0, KHI, pi)
    for t in range(w.steps):
        q, k, v, a, b = step_inputs(w, t)
        o = torch.empty((B, Hv, D), device="cuda")
        fn = rs.kda_decode_update if per_channel else rs.gdn_decode_update
        fn(mix, pool, dev(w.slot_idx), q, k, v, a, b, o=o)
        o_r, st = orc.decode_mixed(ref, w.slot_idx, pi, KHI, D, D, w.q[t], w.k[t], w.v[t],
                                   w.alpha[t], w.beta[t])
        assert st == 0
        o_g = host(o)
        assert max_rel(o_g, o_r) <= 1e-3
        assert same_bits(o_g, o_r), f"o differs at step {t}"
        assert same_bits(host(pool), ref), f"packed state differs at step {t}"


def test_mixed_full_size_64_steps_sampled():
    """KDA, batch 256, 32 heads, 16 FP16 rows per head, 64 steps; oracle on
    5 sampled sequences (all heads)."""
    B, H = 256, 32
    f32, mix, pi = layouts(H, H, seed=2)
    w = gen.decode_workload(B=B, Hk=H, Hv=H, d=D, steps=64, per_channel=True, in_dtype="bf16",
                            seed=2, horizon=(2.0, 8192.0))
    pool = to_mixed_gpu(f32, mix, w.state0)
    outs = mixed_gpu_steps(w, mix, pool, 64)
    bsel = np.array([0, 31, 128, 129, 255])
    ws = sub_batch(w, bsel)
    ref = orc.convert_pool_f32_to_mixed(ws.state0, KHI, pi)
    for t in range(64):
        o_r, _ = orc.decode_mixed(ref, ws.slot_idx, pi, KHI, D, D, ws.q[t], ws.k[t], ws.v[t],
                                  ws.alpha[t], ws.beta[t])
        assert max_rel(outs[t][bsel], o_r) <= 1e-3
        assert same_bits(outs[t][bsel], o_r), t
    assert same_bits(host(pool)[w.slot_idx[bsel]], ref)


@pytest.mark.parametrize("layout_kind,per_channel", [("fp32", True), ("fp32", False),
                                                     ("mixed", True), ("mixed", False)])
def test_replay_matches_oracle(layout_kind, per_channel):
    """Replay of n_accept[b] in {0..8} logged tokens (uniform 1..8 plus the
    0 and 8 edges), state read once and written once."""
    B, Hk, Hv, T = 67, 4, 8, 8
    f32, mix, pi = layouts(Hv, Hk, seed=9)
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=T, per_channel=per_channel,
                            in_dtype="bf16", seed=9, horizon=(2.0, 8192.0))
    n_acc = gen.n_accept(B, T, seed=9)
    n_acc[0], n_acc[1], n_acc[2] = 0, T, 1
    qd, kd, vd, ad, bd = replay_inputs(w, T)
    q, k, v, a, b = gen.replay_view(w, T)
    o = torch.full((B, T, Hv, D), 5.0, device="cuda")
    if layout_kind == "fp32":
        pool = dev(w.state0)
        rs.spec_replay_update(f32, per_channel, pool, dev(w.slot_idx), dev(n_acc), qd, kd, vd, ad,
                              bd, o=o)
        ref = w.state0.copy()
        o_r = np.full((B, T, Hv, D), 5.0, np.float32)
        _, st = orc.replay_f32(ref, w.slot_idx, n_acc, q, k, v, a, b, o=o_r)
    else:
        pool = to_mixed_gpu(f32, mix, w.state0)
        rs.spec_replay_update(mix, per_channel, pool, dev(w.slot_idx), dev(n_acc), qd, kd, vd, ad,
                              bd, o=o)
        ref = orc.convert_pool_f32_to_mixed(w.state0, KHI, pi)
        o_r = np.full((B, T, Hv, D), 5.0, np.float32)
        _, st = orc.replay_mixed(ref, w.slot_idx, n_acc, pi, KHI, D, D, q, k, v, a, b, o=o_r)
    torch.cuda.synchronize()
    assert st == 0
    o_g = host(o)
    assert same_bits(o_g, o_r)
    assert same_bits(host(pool), ref)


def test_replay_full_size_sampled():
    """KDA mixed, batch 256 x 32 heads, n_accept uniform over 1..8."""
    B, H, T = 256, 32, 8
    f32, mix, pi = layouts(H, H, seed=4)
    w = gen.decode_workload(B=B, Hk=H, Hv=H, d=D, steps=T, per_channel=True, in_dtype="bf16",
                            seed=4, horizon=(2.0, 8192.0))
    n_acc = gen.n_accept(B, T, seed=4)
    pool = to_mixed_gpu(f32, mix, w.state0)
    qd, kd, vd, ad, bd = replay_inputs(w, T)
    o = torch.zeros((B, T, H, D), device="cuda")
    rs.spec_replay_update(mix, True, pool, dev(w.slot_idx), dev(n_acc), qd, kd, vd, ad, bd, o=o)
    torch.cuda.synchronize()
    bsel = np.array([3, 64, 250])
    ws = sub_batch(w, bsel)
    q, k, v, a, b = gen.replay_view(ws, T)
    ref = orc.convert_pool_f32_to_mixed(ws.state0, KHI, pi)
    o_r = np.zeros((len(bsel), T, H, D), np.float32)
    orc.replay_mixed(ref, ws.slot_idx, np.ascontiguousarray(n_acc[bsel]), pi, KHI, D, D, q, k, v,
                     a, b, o=o_r)
    assert same_bits(host(o)[bsel], o_r)
    assert same_bits(host(pool)[w.slot_idx[bsel]], ref)


def test_replay_fp32_full_size_sampled():
    """KDA FP32, batch 256 x 32 heads, n_accept uniform over 1..8: several tiles per CTA."""
    B, H, T = 256, 32, 8
    f32, mix, pi = layouts(H, H, seed=5)
    w = gen.decode_workload(B=B, Hk=H, Hv=H, d=D, steps=T, per_channel=True, in_dtype="bf16",
                            seed=5, horizon=(2.0, 8192.0))
    n_acc = gen.n_accept(B, T, seed=5)
    pool = dev(w.state0)
    qd, kd, vd, ad, bd = replay_inputs(w, T)
    o = torch.zeros((B, T, H, D), device="cuda")
    rs.spec_replay_update(f32, True, pool, dev(w.slot_idx), dev(n_acc), qd, kd, vd, ad, bd, o=o)
    torch.cuda.synchronize()
    bsel = np.array([0, 100, 255])
    ws = sub_batch(w, bsel)
    q, k, v, a, b = gen.replay_view(ws, T)
    ref = ws.state0.copy()
    o_r = np.zeros((len(bsel), T, H, D), np.float32)
    orc.replay_f32(ref, ws.slot_idx, np.ascontiguousarray(n_acc[bsel]), q, k, v, a, b, o=o_r)
    assert same_bits(host(o)[bsel], o_r)
    assert same_bits(host(pool)[w.slot_idx[bsel]], ref)


@pytest.mark.parametrize("fused", [False, True])
def test_replay_nonfinite_state(fused):
    """Replay on tiles holding a NaN in an FP16 row and an infinite INT8 row scale: the
    requantisation takes the literal-division path for those tiles.  INT8 codes and scales
    match every byte; FP16 rows and o match up to NaN payloads."""
    B, Hv, T = 4, 4, 4
    hi = gen.hi_rows(Hv, D, KHI, seed=10)
    pi = orc.row_map(hi, D)
    lay = rs.Layout("mixed", D, Hv, Hv, k_hi=KHI, hi_rows=hi, quant="fused" if fused else "ieee")
    w = gen.decode_workload(B=B, Hk=Hv, Hv=Hv, d=D, steps=T, per_channel=True, in_dtype="bf16", seed=10)
    n_acc = np.array([T, 2, 3, 1], np.int32)
    ref = orc.convert_pool_f32_to_mixed(w.state0, KHI, pi)
    s0, s1 = w.slot_idx[0], w.slot_idx[1]
    r, c = 3, 10
    off = 2 * (((r // 2) * D + c) * 2 + r % 2)
    ref[s0, 1, off:off + 2] = np.array([0x7E00], np.uint16).view(np.uint8)
    sc = 2 * KHI * D + (D - KHI) * D + 4 * 5
    ref[s1, 0, sc:sc + 4] = np.array([np.inf], np.float32).view(np.uint8)
    pool = dev(ref)
    qd, kd, vd, ad, bd = replay_inputs(w, T)
    q, k, v, a, b = gen.replay_view(w, T)
    o = torch.full((B, T, Hv, D), 5.0, device="cuda")
    rs.spec_replay_update(lay, True, pool, dev(w.slot_idx), dev(n_acc), qd, kd, vd, ad, bd, o=o)
    o_r = np.full((B, T, Hv, D), 5.0, np.float32)
    _, st = orc.replay_mixed(ref, w.slot_idx, n_acc, pi, KHI, D, D, q, k, v, a, b, o=o_r,
                             mode=1 if fused else 0)
    torch.cuda.synchronize()
    assert st == 0
    assert np.isnan(o_r).any()
    assert nan_aware_same(host(o), o_r)
    g = host(pool)
    hb = 2 * KHI * D
    assert same_bits(g[..., hb:], ref[..., hb:])
    hg = g[..., :hb].copy().view(np.float16)
    hr = ref[..., :hb].copy().view(np.float16)
    nan = np.isnan(hr)
    assert nan.sum() >= KHI
    assert np.array_equal(np.isnan(hg), nan)
    assert np.array_equal(hg.view(np.uint16)[~nan], hr.view(np.uint16)[~nan])


def test_replay_bad_accept_count_reported():
    Hv, Hk, T = 4, 2, 4
    f32, mix, pi = layouts(Hv, Hk, seed=1)
    w = gen.decode_workload(B=3, Hk=Hk, Hv=Hv, d=D, steps=T, per_channel=True, in_dtype="bf16",
                            seed=1)
    n_acc = np.array([2, 9, -1], np.int32)
    pool = dev(w.state0)
    before = host(pool)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qd, kd, vd, ad, bd = replay_inputs(w, T)
    rs.spec_replay_update(f32, True, pool, dev(w.slot_idx), dev(n_acc), qd, kd, vd, ad, bd,
                          status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 2
    after = host(pool)
    for b in (1, 2):
        assert same_bits(after[w.slot_idx[b]], before[w.slot_idx[b]])


def adversarial_rows(n_heads, seed):
    """FP32 heads whose INT8 rows put many x/s within a few ulps of, or
    exactly on, a half-integer (x = (n + 1/2) s nudged by 0..3 ulps; scales
    that are powers of two give exact ties), plus rows holding NaN / inf."""
    g = gen.rng(seed)
    S = np.zeros((n_heads, D, D), np.float32)
    for h in range(n_heads):
        for r in range(D):
            e = int(g.integers(-20, 4))
            a = np.float32(127.0 * 2.0 ** e) if r % 3 == 0 else np.float32(g.uniform(0.05, 3.0))
            s = np.float32(np.float32(max(a, np.float32(1e-8))) / np.float32(127.0))
            n = g.integers(-126, 126, D).astype(np.float32)
            x = ((n + np.float32(0.5)) * s).astype(np.float32)
            nudge = g.integers(-3, 4, D)
            x = np.array([np.nextafter(xi, np.float32(np.inf) if k > 0 else np.float32(-np.inf))
                          if k else xi for xi, k in zip(x, nudge)], np.float32)
            for _ in range(2):
                x = np.where(nudge > 1, np.nextafter(x, np.float32(np.inf)), x)
                x = np.where(nudge < -1, np.nextafter(x, np.float32(-np.inf)), x)
            x[0] = a                      # the row's absmax
            x = np.clip(x, -a, a).astype(np.float32)
            S[h, r] = x
    S[0, 20, 5] = np.nan
    S[0, 21, 7] = np.inf
    S[0, 22, 9] = -np.inf
    S[0, 22, 10] = np.nan
    S[1, 40, :] = 0.0
    return S


def test_quantiser_rounding_near_half_integers():
    Hv = 4
    f32, mix, pi = layouts(Hv, Hv, seed=12)
    state = adversarial_rows(3 * Hv, 12).reshape(3, Hv, D, D)
    g = host(to_mixed_gpu(f32, mix, state))
    ref = orc.convert_pool_f32_to_mixed(state, KHI, pi)
    # INT8 codes and scales: every byte.  FP16 rows: every bit, except that a
    # NaN only has to stay a NaN (its payload bits are not part of the format).
    hb = 2 * KHI * D
    assert same_bits(g[..., hb:], ref[..., hb:])
    hg = g[..., :hb].copy().view(np.float16)
    hr = ref[..., :hb].copy().view(np.float16)
    nan = np.isnan(hr)
    assert np.array_equal(np.isnan(hg), nan)
    assert np.array_equal(hg.view(np.uint16)[~nan], hr.view(np.uint16)[~nan])
    assert nan.sum() >= 1  # the NaN planted in an FP16 row survives


@pytest.mark.parametrize("per_channel", [True, False])
def test_mixed_decode_small_batch_bad_slots(per_channel):
    """Fewer tiles than streaming multiprocessors, two of them with slots out
    of range: those are skipped and reported (status bit 1), the rest match
    the oracle bit for bit."""
    B, Hk, Hv = 6, 2, 4
    f32, mix, pi = layouts(Hv, Hk, seed=8)
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=1, per_channel=per_channel,
                            in_dtype="bf16", seed=8, n_slots=9)
    w.slot_idx[2] = 9
    w.slot_idx[4] = -1
    ref = orc.convert_pool_f32_to_mixed(w.state0, KHI, pi)
    pool = dev(ref)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, k, v, a, b = step_inputs(w, 0)
    o = torch.full((B, Hv, D), 7.0, device="cuda")
    fn = rs.kda_decode_update if per_channel else rs.gdn_decode_update
    fn(mix, pool, dev(w.slot_idx), q, k, v, a, b, o=o, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    oh = host(o)
    assert np.all(oh[[2, 4]] == 7.0)
    ok = np.array([0, 1, 3, 5])
    o_r, st = orc.decode_mixed(ref, w.slot_idx[ok], pi, KHI, D, D, w.q[0][ok], w.k[0][ok],
                               w.v[0][ok], w.alpha[0][ok], w.beta[0][ok])
    assert st == 0
    assert same_bits(oh[ok], o_r)
    assert same_bits(host(pool), ref)


def nan_aware_same(g, r):
    gn, rn = np.isnan(g), np.isnan(r)
    return np.array_equal(gn, rn) and np.array_equal(g[~gn].view(np.uint32), r[~rn].view(np.uint32))


def test_mixed_decode_nonfinite_state():
    """A NaN in an FP16 row spreads through the prediction to its whole
    column, and an infinite INT8 scale makes its row infinite: every INT8
    block of those tiles then takes the literal-division path.  INT8 codes
    and scales must match every byte; FP16 rows and o match up to NaN
    payloads."""
    B, Hv = 4, 4
    f32, mix, pi = layouts(Hv, Hv, seed=9)
    for per_channel in (True, False):
        w = gen.decode_workload(B=B, Hk=Hv, Hv=Hv, d=D, steps=1, per_channel=per_channel,
                                in_dtype="bf16", seed=9)
        ref = orc.convert_pool_f32_to_mixed(w.state0, KHI, pi)
        s0, s1 = w.slot_idx[0], w.slot_idx[1]
        r, c = 3, 10                               # FP16 row 3, column 10 of head 1
        off = 2 * (((r // 2) * D + c) * 2 + r % 2)
        ref[s0, 1, off:off + 2] = np.array([0x7E00], np.uint16).view(np.uint8)
        sc = 2 * KHI * D + (D - KHI) * D + 4 * 5  # INT8 row 5's scale in head 0
        ref[s1, 0, sc:sc + 4] = np.array([np.inf], np.float32).view(np.uint8)
        pool = dev(ref)
        q, k, v, a, b = step_inputs(w, 0)
        o = torch.empty((B, Hv, D), device="cuda")
        fn = rs.kda_decode_update if per_channel else rs.gdn_decode_update
        fn(mix, pool, dev(w.slot_idx), q, k, v, a, b, o=o)
        o_r, st = orc.decode_mixed(ref, w.slot_idx, pi, KHI, D, D, w.q[0], w.k[0], w.v[0],
                                   w.alpha[0], w.beta[0])
        assert st == 0
        assert np.isnan(o_r).any()
        assert nan_aware_same(host(o), o_r)
        g = host(pool)
        hb = 2 * KHI * D
        assert same_bits(g[..., hb:], ref[..., hb:])
        hg = g[..., :hb].copy().view(np.float16)
        hr = ref[..., :hb].copy().view(np.float16)
        nan = np.isnan(hr)
        assert nan.sum() >= KHI  # the NaN column of head 1, all its FP16 rows
        assert np.array_equal(np.isnan(hg), nan)
        assert np.array_equal(hg.view(np.uint16)[~nan], hr.view(np.uint16)[~nan])
