"""Pins for the oracle's INT8 state checkpoint and whole-head checkpoints of
packed (mixed FP16/INT8) pools (CPU only).

dasc Appendix E.1 Eq. 8: the cached FP32 state is quantised once at insertion
(symmetric INT8, one FP32 scale per (layer, head, key channel) shared over
dv, s = max(a, 1e-8)/127, codes clip(round(S/s), -127, 127)) and dequantised
once on reuse (S^ = q s).  dasc §4.1 / Appendix B Scheme 2: retained units
packed in layer order; §4.2: omitted units restore as zero.  DAMP §5.2: a
mixed head (FP16 rows, INT8 rows, scales) is one packed unit.

Pins: closed forms for constant rows (codes +-127, scale = |c|/127), the
quantiser's error bound |S^ - S| <= s/2 on every retained element, exact
zeros for omitted units, the byte accounting (16,896 B per 128 x 128 head,
65,536 / 16,896 = 3.88 of FP32), agreement of head and channel granularity
when the same rows are kept, and agreement of the whole-head pack with the
pinned FP32 pack when the head is an FP32 tile.
"""
import numpy as np
import pytest

import oracle as orc
from recurrent_state_gb300 import inputs as gen


def test_int8_bytes_per_head_and_ratio():
    codes, slot = orc.ckpt_int8_layout(1, 0, 128, 128)
    assert codes == 128 * 128 and slot == 128 * 128 + 128 * 4 == 16896
    assert round(65536 / slot, 2) == 3.88       # dasc Appendix E.1: 3.88x rather than 4x
    codes, slot = orc.ckpt_int8_layout(1, 1, 128, 128)
    assert (codes, slot) == (128, 144)          # one channel: 128 codes + 1 scale, slot padded to 16


def constant_rows_pool(L, S, Hv, dk, dv, seed):
    """Every row of every head holds one value (sign and size per row), so
    codes are +-127 and the scale is |c|/127 in closed form."""
    g = gen.rng(seed)
    c = (g.choice([-1.0, 1.0], (L, S, Hv, dk)) * 10.0 ** g.uniform(-6, 3, (L, S, Hv, dk))).astype(np.float32)
    return np.repeat(c[..., None], dv, axis=-1).astype(np.float32), c


@pytest.mark.parametrize("unit", [0, 1])
def test_constant_rows_closed_form_and_order(unit):
    L, S, Hv, dk, dv = 3, 4, 2, 8, 16
    pool, c = constant_rows_pool(L, S, Hv, dk, dv, seed=1)
    keep = gen.keep_mask(L, Hv if unit == 0 else Hv * dk, 0.5, seed=2)
    nk = int(keep.sum())
    codes_b, slot_b = orc.ckpt_int8_layout(nk, unit, dk, dv)
    src, dst = np.array([2, 0], np.int32), np.array([1, 0], np.int32)
    ck = np.zeros((2, slot_b), np.uint8)
    assert orc.ckpt_pack_int8(keep, unit, pool, src, dst, ck) == 0
    R = 1 if unit else dk
    for i in range(2):
        codes = ck[dst[i], :codes_b].view(np.int8).reshape(nk * R, dv)
        scales = ck[dst[i], codes_b:codes_b + 4 * nk * R].view(np.float32)
        # rows of the retained units in packed order, stated directly
        want = []
        for l in range(L):
            for x in range(keep.shape[1]):
                if keep[l, x]:
                    want.extend(c[l, src[i], x] if unit == 0 else [c[l, src[i]].reshape(-1)[x]])
        want = np.array(want, np.float32)
        assert np.array_equal(scales, (np.abs(want) / np.float32(127.0)).astype(np.float32))
        assert np.array_equal(codes, np.repeat(np.where(want > 0, 127, -127)[:, None], dv, 1).astype(np.int8))


@pytest.mark.parametrize("unit", [0, 1])
def test_roundtrip_error_bound_and_zero_fill(unit):
    L, S, Hv, dk, dv = 2, 5, 3, 16, 32
    pool = gen.random_pool((L, S, Hv, dk, dv), seed=3)
    pool[1, 2, 1, 3] *= 1e4  # an outlier row
    keep = gen.keep_mask(L, Hv if unit == 0 else Hv * dk, 0.45, seed=4)
    nk = int(keep.sum())
    codes_b, slot_b = orc.ckpt_int8_layout(nk, unit, dk, dv)
    src, dst = np.array([4, 2, 0], np.int32), np.array([0, 2, 1], np.int32)
    ck = np.zeros((3, slot_b), np.uint8)
    assert orc.ckpt_pack_int8(keep, unit, pool, src, dst, ck) == 0
    out = np.full((L, 3, Hv, dk, dv), 9.0, np.float32)
    back_dst = np.array([1, 0, 2], np.int32)
    assert orc.ckpt_restore_int8(keep, unit, ck, dst, out, back_dst) == 0
    kr = keep.reshape(L, Hv, dk if unit else 1)
    for i in range(3):
        for l in range(L):
            for h in range(Hv):
                for u in range(dk):
                    got = out[l, back_dst[i], h, u]
                    if not kr[l, h, u if unit else 0]:
                        assert np.all(got == 0.0) and not np.signbit(got).any()
                        continue
                    row = pool[l, src[i], h, u]
                    s = np.float32(max(np.abs(row).max(), np.float32(1e-8))) / np.float32(127.0)
                    assert np.all(np.abs(got.astype(np.float64) - row) <= s * 0.5 * (1 + 2.0 ** -20)
                                  + np.abs(row) * 2.0 ** -22)


def test_head_and_channel_granularity_agree():
    """Keeping every channel of the kept heads stores the same rows in the
    same order: identical codes and scales."""
    L, S, Hv, dk, dv = 2, 2, 4, 8, 16
    pool = gen.random_pool((L, S, Hv, dk, dv), seed=5)
    kh = gen.keep_mask(L, Hv, 0.5, seed=6)
    kc = np.repeat(kh, dk, axis=1)
    nh, nc = int(kh.sum()), int(kc.sum())
    _, sh = orc.ckpt_int8_layout(nh, 0, dk, dv)
    _, sc = orc.ckpt_int8_layout(nc, 1, dk, dv)
    assert sh == sc
    a, b = np.zeros((1, sh), np.uint8), np.zeros((1, sc), np.uint8)
    one, zero = np.array([1], np.int32), np.array([0], np.int32)
    orc.ckpt_pack_int8(kh, 0, pool, one, zero, a)
    orc.ckpt_pack_int8(kc, 1, pool, one, zero, b)
    assert np.array_equal(a, b)


def test_int8_bad_slots_reported():
    pool = gen.random_pool((1, 2, 2, 4, 4), seed=7)
    keep = np.ones((1, 2), np.uint8)
    _, sb = orc.ckpt_int8_layout(2, 0, 4, 4)
    ck = np.zeros((1, sb), np.uint8)
    assert orc.ckpt_pack_int8(keep, 0, pool, np.array([5], np.int32), np.array([0], np.int32), ck) == 1
    assert orc.ckpt_pack_int8(keep, 0, pool, np.array([0], np.int32), np.array([3], np.int32), ck) == 4
    assert not ck.any()


def test_whole_head_pack_matches_fp32_pack():
    """An FP32 tile seen as head_bytes bytes packs exactly as the pinned FP32
    head-unit pack; restore zero-fills omitted heads."""
    L, S, Hv, d = 2, 3, 4, 8
    pool = gen.random_pool((L, S, Hv, d, d), seed=8)
    keep = gen.keep_mask(L, Hv, 0.5, seed=9)
    nk = int(keep.sum())
    src, dst = np.array([2, 1], np.int32), np.array([0, 1], np.int32)
    a = np.zeros((2, nk * d * d * 4), np.uint8)
    b = np.zeros_like(a)
    orc.ckpt_pack(keep, 0, pool, src, dst, a)
    orc.ckpt_pack_heads(keep, np.ascontiguousarray(pool.view(np.uint8).reshape(L, S, Hv, d * d * 4)),
                        src, dst, b)
    assert np.array_equal(a, b)
    back = np.full((L, S, Hv, d * d * 4), 0xAB, np.uint8)
    assert orc.ckpt_restore_heads(keep, b, dst, back, np.array([0, 2], np.int32)) == 0
    for i, s in enumerate((0, 2)):
        for l in range(L):
            for h in range(Hv):
                want = pool[l, src[i], h].view(np.uint8).reshape(-1) if keep[l, h] else 0
                assert np.all(back[l, s, h] == want)
    assert np.all(back[:, 1] == 0xAB)  # untouched slot


def test_mixed_heads_roundtrip_verbatim():
    """Mixed tiles (FP16 rows, INT8 rows, scales) round-trip byte for byte."""
    L, S, Hv, d, khi = 2, 2, 2, 32, 4
    g = gen.rng(10)
    tiles = np.stack([np.stack([np.stack([orc.mixed_pack(g.standard_normal((d, d)).astype(np.float32), khi)
                                          for _ in range(Hv)]) for _ in range(S)]) for _ in range(L)])
    keep = np.array([[1, 0], [1, 1]], np.uint8)
    hb = tiles.shape[-1]
    assert hb == orc.mixed_tile_bytes(d, d, khi)
    ck = np.zeros((1, 3 * hb), np.uint8)
    assert orc.ckpt_pack_heads(keep, tiles, np.array([1], np.int32), np.array([0], np.int32), ck) == 0
    back = np.zeros_like(tiles)
    assert orc.ckpt_restore_heads(keep, ck, np.array([0], np.int32), back, np.array([0], np.int32)) == 0
    assert np.array_equal(back[0, 0, 0], tiles[0, 1, 0]) and not back[0, 0, 1].any()
    assert np.array_equal(back[1, 0], tiles[1, 1])
