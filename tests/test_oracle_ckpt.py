"""Pins for the oracle's dasc checkpoint pack and restore (CPU only).

dasc §4.1 and Appendix B "Ragged (Scheme 2)": retained units of each layer
are flat-packed with offsets o_0 = 0, o_l = o_{l-1} + r_l; a GDN unit is one
head state, a KDA unit is one (head, key channel) row of dv values.  dasc
§4.2: dasc-nr restores the retained units exactly and leaves omitted units
at zero.  The pins: a hand-worked golden plan, an independent numpy
fancy-indexing statement of the same gather/scatter, the identity when
everything is kept, all zeros when nothing is, and the closed-form
compression ratios of §4.1 Eq. 6 / Appendix B.
"""
import json
import os

import numpy as np
import pytest

import oracle as orc
from recurrent_state_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def units_view(pool_l_slot, unit):
    """[Hv][dk][dv] float32 -> [n_units][unit_values] (head or channel rows)."""
    Hv, dk, dv = pool_l_slot.shape
    return pool_l_slot.reshape(Hv, dk * dv) if unit == 0 else pool_l_slot.reshape(Hv * dk, dv)


def numpy_pack(pool, keep, unit, src, dst, n_ckpt):
    L = pool.shape[0]
    rows = []
    per = []
    for i in range(len(src)):
        parts = [units_view(pool[l, src[i]], unit)[keep[l].astype(bool)] for l in range(L)]
        per.append(np.concatenate(parts).reshape(-1).view(np.uint8))
    out = np.zeros((n_ckpt, per[0].size if per else 0), np.uint8)
    for i, d in enumerate(dst):
        out[d] = per[i]
    return out


def test_golden_offsets_and_order():
    gdn = json.load(open(os.path.join(GOLDEN, "dasc_offsets.json")))
    keep = np.array(gdn["keep"], np.uint8)
    L, n = keep.shape
    # GDN plan: n units per layer = Hv heads
    off = orc.plan_offsets(keep, n, 1, 0)
    assert off.tolist() == gdn["offsets"]
    # pack order: build a pool whose every unit holds its own (layer, unit) id
    Hv, dk, dv = n, 2, 2
    pool = np.zeros((L, 1, Hv, dk, dv), np.float32)
    for l in range(L):
        for h in range(Hv):
            pool[l, 0, h] = 1000 * l + h
    ckpt = np.zeros((1, off[-1] * dk * dv * 4), np.uint8)
    assert orc.ckpt_pack(keep, 0, pool, np.array([0], np.int32), np.array([0], np.int32), ckpt) == 0
    ids = ckpt[0].view(np.float32).reshape(-1, dk * dv)[:, 0]
    assert [[int(x) // 1000, int(x) % 1000] for x in ids] == gdn["packed_order"]
    r = keep.sum(1)
    assert r.tolist() == gdn["r"]
    c_rag = keep.size / r.sum()
    c_pad = keep.size / (L * r.max())
    assert c_rag == pytest.approx(gdn["C_temp_rag"])
    assert c_pad == pytest.approx(gdn["C_temp_pad"])
    assert c_rag / c_pad == pytest.approx(gdn["R_max"] / gdn["r_bar"]) == pytest.approx(gdn["layout_gain"])


@pytest.mark.parametrize("unit,p", [(0, 0.5), (1, 0.45)])
def test_pack_matches_numpy_statement(unit, p):
    L, slots, Hv, d = 5, 6, 4, 8
    pool = gen.random_pool((L, slots, Hv, d, d), seed=unit)
    n_units = Hv if unit == 0 else Hv * d
    keep = gen.keep_mask(L, n_units, p, seed=unit)
    off = orc.plan_offsets(keep, Hv, d, unit)
    ub = (d * d * 4) if unit == 0 else d * 4
    src, dst = gen.ckpt_slots(slots, 4, seed=unit)
    ckpt = np.full((4, off[-1] * ub), 0xAB, np.uint8)
    assert orc.ckpt_pack(keep, unit, pool, src, dst, ckpt) == 0
    assert np.array_equal(ckpt, numpy_pack(pool, keep, unit, src, dst, 4))


@pytest.mark.parametrize("unit,p", [(0, 0.5), (1, 0.45)])
def test_restore_zero_fills_and_roundtrips(unit, p):
    L, slots, Hv, d = 4, 5, 3, 8
    pool = gen.random_pool((L, slots, Hv, d, d), seed=10 + unit)
    n_units = Hv if unit == 0 else Hv * d
    keep = gen.keep_mask(L, n_units, p, seed=20 + unit)
    off = orc.plan_offsets(keep, Hv, d, unit)
    ub = (d * d * 4) if unit == 0 else d * 4
    src = np.array([3, 1], np.int32)
    dst = np.array([0, 1], np.int32)
    ckpt = np.zeros((2, off[-1] * ub), np.uint8)
    assert orc.ckpt_pack(keep, unit, pool, src, dst, ckpt) == 0
    out = np.full_like(pool, np.nan)
    rest_dst = np.array([2, 4], np.int32)
    assert orc.ckpt_restore(keep, unit, ckpt, dst, out, rest_dst) == 0
    for i in range(2):
        for l in range(L):
            got = units_view(out[l, rest_dst[i]], unit)
            ref = units_view(pool[l, src[i]], unit)
            kb = keep[l].astype(bool)
            assert np.array_equal(got[kb].view(np.uint32), ref[kb].view(np.uint32))
            assert np.all(got[~kb].view(np.uint32) == 0)      # +0.0 bit pattern
    # untouched slots stay as they were
    assert np.all(np.isnan(out[:, [0, 1, 3]]))
    # pack(restore(pack)) == pack
    ckpt2 = np.zeros_like(ckpt)
    assert orc.ckpt_pack(keep, unit, out, rest_dst, dst, ckpt2) == 0
    assert np.array_equal(ckpt, ckpt2)


@pytest.mark.parametrize("unit", [0, 1])
def test_all_kept_is_identity_and_none_kept_is_zero(unit):
    L, slots, Hv, d = 3, 2, 2, 4
    pool = gen.random_pool((L, slots, Hv, d, d), seed=30 + unit)
    n_units = Hv if unit == 0 else Hv * d
    keep = np.ones((L, n_units), np.uint8)
    ckpt = np.zeros((1, L * Hv * d * d * 4), np.uint8)
    assert orc.ckpt_pack(keep, unit, pool, np.array([1], np.int32), np.array([0], np.int32), ckpt) == 0
    assert np.array_equal(ckpt[0], pool[:, 1].reshape(-1).view(np.uint8))
    out = np.full_like(pool, 3.0)
    assert orc.ckpt_restore(keep, unit, ckpt, np.array([0], np.int32), out,
                            np.array([0], np.int32)) == 0
    assert np.array_equal(out[:, 0], pool[:, 1])
    none = np.zeros((L, n_units), np.uint8)
    assert orc.plan_offsets(none, Hv, d, unit).tolist() == [0] * (L + 1)
    empty = np.zeros((1, 0), np.uint8)
    assert orc.ckpt_pack(none, unit, pool, np.array([1], np.int32), np.array([0], np.int32), empty) == 0
    assert orc.ckpt_restore(none, unit, empty, np.array([0], np.int32), out,
                            np.array([1], np.int32)) == 0
    assert np.all(out[:, 1].view(np.uint32) == 0)


def test_bad_slots_are_skipped():
    L, slots, Hv, d = 2, 2, 2, 4
    pool = gen.random_pool((L, slots, Hv, d, d), seed=40)
    keep = np.ones((L, Hv), np.uint8)
    ckpt = np.zeros((2, L * Hv * d * d * 4), np.uint8)
    st = orc.ckpt_pack(keep, 0, pool, np.array([5, 0], np.int32), np.array([0, 9], np.int32), ckpt)
    assert st == (1 | 4)
    assert np.all(ckpt == 0)
