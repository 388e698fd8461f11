"""Pins for the oracle's DAMP-exact storage (CPU only): INT8 groups of 32
along dv with one FP32 scale per group and value scaling (DAMP Appendix A.1,
A.3 Eq. 17-18, A.4).

Pins: the printed storage accounting (9.9 bits per value, 69.1% less than
FP32, at 16 FP16 channels and groups of 32, d = 128); group = dv without
scaling is exactly the one-scale-per-row layout (tile bytes and decode);
closed forms for rows constant per group; the quantiser bound per group;
equivariance under power-of-two value scales constant per group (the
transformed recurrence of Eq. 18 then reproduces the unscaled readout and
codes bit for bit, and every scale by exactly 2^-k); replay of one token
equals a decode step; and the transformed step against the untransformed
map in fp64 (Eq. 17-18 in exact arithmetic).
"""
import json
import os

import numpy as np
import pytest

import oracle as orc
from recurrent_state_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
D, KHI, G = 128, 16, 32


def test_printed_accounting():
    g = json.load(open(os.path.join(GOLDEN, "accounting.json")))
    tb = orc.damp_tile_bytes(D, D, KHI, G)
    assert tb == 16 * 128 * 2 + 112 * 128 + 112 * 4 * 4 == 20224
    bits = tb * 8 / (D * D)
    assert bits == 9.875 and round(bits, 1) == g["printed_bits_per_value"]
    assert round(100 * (1 - bits / 32), 1) == g["printed_reduction_percent"]


def test_group_dv_unscaled_is_the_row_layout():
    g = gen.rng(1)
    T = g.standard_normal((32, 64)).astype(np.float32)
    assert np.array_equal(orc.damp_pack(T, 8, 64), orc.mixed_pack(T, 8))
    B, Hv, d = 3, 2, 32
    hi = gen.hi_rows(Hv, d, 4, seed=2)
    pi = orc.row_map(hi, d)
    w = gen.decode_workload(B=B, Hk=Hv, Hv=Hv, d=d, steps=1, per_channel=True, in_dtype="f32", seed=3)
    a = orc.convert_pool_f32_to_mixed(w.state0, 4, pi)
    b = a.copy()
    ones = np.ones((Hv, d), np.float32)
    oa, _ = orc.decode_mixed(a, w.slot_idx, pi, 4, d, d, w.q[0], w.k[0], w.v[0], w.alpha[0], w.beta[0])
    ob, _ = orc.decode_damp(b, w.slot_idx, pi, ones, 4, d, d, d, w.q[0], w.k[0], w.v[0], w.alpha[0], w.beta[0])
    assert np.array_equal(oa.view(np.uint32), ob.view(np.uint32)) and np.array_equal(a, b)


def test_constant_groups_closed_form():
    T = np.zeros((8, D), np.float32)
    c = np.array([3.0, -0.001, 1e4, 7.5], np.float32)
    for r in range(4, 8):
        T[r] = np.repeat(c * (r - 3), G)
    tile = orc.damp_pack(T, 4, G)
    lo = tile[2 * 4 * D: 2 * 4 * D + 4 * D].view(np.int8).reshape(1, D, 4)   # one word row of 4 INT8 rows
    sc = tile[2 * 4 * D + 4 * D:].view(np.float32).reshape(4, 4)
    for q in range(4):
        assert np.array_equal(sc[q], (np.abs(c * (q + 1)) / np.float32(127.0)).astype(np.float32))
        assert np.array_equal(lo[0, :, q], np.repeat(np.where(c > 0, 127, -127), G).astype(np.int8))


def test_group_error_bound():
    g = gen.rng(4)
    T = (g.standard_normal((24, D)) * 10.0 ** g.uniform(-3, 3, (24, 1))).astype(np.float32)
    T[10, 5] = 1e5   # an outlier confined to one group
    back = orc.damp_unpack(orc.damp_pack(T, 8, G), 24, D, 8, G)
    for r in range(8, 24):
        for gi in range(D // G):
            x = T[r, gi * G:(gi + 1) * G]
            s = np.float32(max(np.abs(x).max(), np.float32(1e-8))) / np.float32(127.0)
            err = np.abs(back[r, gi * G:(gi + 1) * G].astype(np.float64) - x)
            assert np.all(err <= s * 0.5 * (1 + 2.0 ** -20) + np.abs(x) * 2.0 ** -22)
    # the outlier's group is coarse, the other groups of its row are not
    assert np.abs(back[10, 32:] - T[10, 32:]).max() <= np.abs(T[10, 32:]).max() / 200


@pytest.mark.parametrize("per_channel", [True, False])
def test_pow2_value_scaling_equivariance(per_channel):
    """All rows INT8 here: FP16 rounding does not commute with a power-of-two
    scaling near the FP16 subnormal range, so FP16 rows would break exact
    equivariance for reasons unrelated to the transform."""
    B, Hv, d = 4, 2, D
    KHI = 0
    pi = np.tile(np.arange(d, dtype=np.int16), (Hv, 1))
    w = gen.decode_workload(B=B, Hk=1, Hv=Hv, d=d, steps=3, per_channel=per_channel, in_dtype="f32",
                            seed=6)
    cs = gen.value_scales(Hv, d, seed=7, group=G, pow2=True)
    ones = np.ones_like(cs)
    a = orc.convert_pool_f32_to_damp(w.state0, KHI, G, pi, ones)
    b = orc.convert_pool_f32_to_damp(w.state0, KHI, G, pi, cs)
    for t in range(3):
        oa, _ = orc.decode_damp(a, w.slot_idx, pi, ones, KHI, G, d, d, w.q[t], w.k[t], w.v[t],
                                w.alpha[t], w.beta[t])
        ob, _ = orc.decode_damp(b, w.slot_idx, pi, cs, KHI, G, d, d, w.q[t], w.k[t], w.v[t],
                                w.alpha[t], w.beta[t])
        assert np.array_equal(oa.view(np.uint32), ob.view(np.uint32)), t
    n_code = 2 * KHI * d + (d - KHI) * d
    assert np.array_equal(a[..., 2 * KHI * d:n_code], b[..., 2 * KHI * d:n_code])   # INT8 codes
    sa = a[..., n_code:].copy().view(np.float32).reshape(*a.shape[:2], d - KHI, d // G)
    sb = b[..., n_code:].copy().view(np.float32).reshape(*b.shape[:2], d - KHI, d // G)
    ratio = (cs[:, ::G])[None, :, None, :]          # the power of two of each group
    assert np.array_equal(sb * ratio, sa)


def test_replay_one_token_equals_decode():
    B, Hv, d = 3, 2, D
    hi = gen.hi_rows(Hv, d, KHI, seed=8)
    pi = orc.row_map(hi, d)
    w = gen.decode_workload(B=B, Hk=Hv, Hv=Hv, d=d, steps=2, per_channel=True, in_dtype="f32", seed=9)
    cs = gen.value_scales(Hv, d, seed=10)
    a = orc.convert_pool_f32_to_damp(w.state0, KHI, G, pi, cs)
    b = a.copy()
    oa, _ = orc.decode_damp(a, w.slot_idx, pi, cs, KHI, G, d, d, w.q[0], w.k[0], w.v[0], w.alpha[0], w.beta[0])
    rv = gen.replay_view(w, 2)
    ob, st = orc.replay_damp(b, w.slot_idx, np.ones(B, np.int32), pi, cs, KHI, G, d, d, *rv)
    assert st == 0
    assert np.array_equal(oa, ob[:, 0]) and np.array_equal(a, b)


def test_transformed_step_matches_original_map_fp64():
    """Eq. 17-18 in exact arithmetic: the transformed state and readout of
    the oracle (all rows FP16 so that only FP16 rounding intervenes) track
    the untransformed FP64 step to the FP16 tolerance."""
    g = gen.rng(11)
    d = 32
    S = (g.standard_normal((d, d)) * 0.1).astype(np.float32)
    q, k = g.standard_normal(d).astype(np.float32), g.standard_normal(d).astype(np.float32)
    k /= np.linalg.norm(k)
    q /= np.linalg.norm(q)
    v = g.standard_normal(d).astype(np.float32)
    alpha = g.uniform(0.5, 1.0, d).astype(np.float32)
    beta = np.float32(0.7)
    pi = g.permutation(d).astype(np.int16)
    cs = np.exp(g.uniform(-1, 1, d)).astype(np.float32)
    tile = np.zeros((1, 1, orc.damp_tile_bytes(d, d, d, d)), np.uint8)
    tile[0, 0] = orc.convert_pool_f32_to_damp(S[None, None], d, d, pi[None], cs[None])[0, 0]
    o, _ = orc.decode_damp(tile, np.zeros(1, np.int32), pi[None], cs[None], d, d, d, d, q[None, None],
                           k[None, None], v[None, None], alpha[None, None], np.array([[beta]], np.float32))
    S64 = S.astype(np.float64) * alpha[:, None]
    e = v - S64.T @ k
    S64 = S64 + beta * np.outer(k, e)
    o64 = S64.T @ q
    assert np.max(np.abs(o[0, 0] - o64)) <= 5e-3 * np.max(np.abs(o64))
    back = orc.convert_pool_damp_to_f32(tile, d, d, d, d, pi[None], cs[None])[0, 0]
    assert np.max(np.abs(back - S64)) <= 5e-3 * np.max(np.abs(S64))
