"""Pins for the oracle's state quantiser and mixed-precision tile (CPU only).

Sources: DAMP §3.2 Eq. 5-6 (symmetric INT8 per key-channel row), §5.2 and
Appendix A.4 (FP16 rows for the selected channels, INT8 for the rest, packed
contiguously), Appendix A.3 Eq. 17 (rows stored in the permuted order
T = P_K S); dasc Appendix E.1 Eq. 8 (scale floor 1e-8, clip to +-127, FP32).
Pins: hand-worked golden rows, closed-form special cases, the rounding error
bound |Q(x) - x| <= s/2, numpy's IEEE float16 conversion, and idempotence.
"""
import json
import os

import numpy as np
import pytest

import oracle as orc
from recurrent_state_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_golden_tie_rows():
    cases = json.load(open(os.path.join(GOLDEN, "quant_ties.json")))["cases"]
    for c in cases:
        row = np.array(c["row"], np.float32)
        codes, s = orc.quantise_row(row)
        if isinstance(c["scale"], str):
            assert s == np.float32(1e-8) / np.float32(127.0)
        else:
            assert s == np.float32(c["scale"])
        assert codes.tolist() == c["codes"], (row, codes)


def test_zero_row_uses_floor():
    codes, s = orc.quantise_row(np.zeros(128, np.float32))
    assert s == np.float32(np.float32(1e-8) / np.float32(127.0))
    assert np.all(codes == 0)


@pytest.mark.parametrize("val", [3.25, -0.001, 1e-6, -7e3])
def test_single_nonzero_maps_to_full_scale(val):
    row = np.zeros(64, np.float32)
    row[17] = val
    codes, s = orc.quantise_row(row)
    assert codes[17] == (127 if val > 0 else -127)
    assert np.count_nonzero(codes) == 1
    assert s == np.float32(max(np.float32(abs(np.float32(val))), np.float32(1e-8))) / np.float32(127.0)


def test_error_bound_and_range():
    g = gen.rng(11)
    for _ in range(200):
        n = int(g.integers(1, 200))
        x = (g.standard_normal(n) * 10.0 ** g.uniform(-6, 3)).astype(np.float32)
        codes, s = orc.quantise_row(x)
        assert np.all(np.abs(codes.astype(np.int32)) <= 127)
        assert np.abs(codes.astype(np.int32)).max() == 127  # the absmax element
        xr = orc.dequantise_row(codes, s)
        # |c s - x| <= s/2 up to the rounding of x/s and of c*s (a few ulp)
        bound = s * 0.5 * (1 + 2.0 ** -20) + np.abs(x) * 2.0 ** -22
        assert np.all(np.abs(xr.astype(np.float64) - x) <= bound)


def test_idempotent_on_dequantised_rows():
    g = gen.rng(12)
    for _ in range(100):
        x = g.standard_normal(128).astype(np.float32)
        c1, s1 = orc.quantise_row(x)
        c2, s2 = orc.quantise_row(orc.dequantise_row(c1, s1))
        assert np.array_equal(c1, c2)
        assert abs(float(s2) - float(s1)) <= 2 * np.spacing(np.float32(s1))


def test_nan_row_reading():
    """A NaN anywhere makes the absmax NaN; fmaxf then takes the 1e-8 floor,
    the NaN element clips to -127 and finite elements saturate."""
    row = np.array([0.5, np.nan, -2e-9, 0.0], np.float32)
    codes, s = orc.quantise_row(row)
    assert s == np.float32(1e-8) / np.float32(127.0)
    assert codes.tolist() == [127, -127, -25, 0]


def hi_region(tile, khi, dv):
    """FP16 rows [khi][dv] from the FP16 region (row pairs interleaved)."""
    h = tile[: 2 * khi * dv].view(np.uint16).reshape(khi // 2, dv, 2)
    return np.ascontiguousarray(h.transpose(0, 2, 1).reshape(khi, dv))


def lo_region(tile, dk, khi, dv):
    """INT8 rows [dk-khi][dv] from the INT8 region (row quads interleaved)."""
    n = (dk - khi) * dv
    b = tile[2 * khi * dv: 2 * khi * dv + n].view(np.int8).reshape((dk - khi) // 4, dv, 4)
    return np.ascontiguousarray(b.transpose(0, 2, 1).reshape(dk - khi, dv))


def test_fp16_rows_match_ieee_half():
    """FP16 rows round to nearest even like numpy's IEEE float16 conversion."""
    g = gen.rng(13)
    dk, dv, khi = 8, 32, 4
    T = (g.standard_normal((dk, dv)) * 10.0 ** g.uniform(-3, 4, (dk, 1))).astype(np.float32)
    T[0, :4] = [65504.0, 65520.0, -70000.0, 6e-8]  # max, overflow to inf, tiny
    tile = orc.mixed_pack(T, khi)
    hi = hi_region(tile, khi, dv)
    assert np.array_equal(hi, T[:khi].astype(np.float16).view(np.uint16))
    back = orc.mixed_unpack(tile, dk, dv, khi)
    assert np.array_equal(back[:khi], T[:khi].astype(np.float16).astype(np.float32))


def test_mixed_tile_layout_and_size():
    """16 FP16 rows + 112 INT8 rows + 112 FP32 row scales at d = 128; inside
    the regions, one 32-bit word holds one column of 2 FP16 rows or of 4
    INT8 rows."""
    dk = dv = 128
    khi = 16
    assert orc.mixed_tile_bytes(dk, dv, khi) == 16 * 128 * 2 + 112 * 128 + 112 * 4 == 18880
    g = gen.rng(14)
    T = g.standard_normal((dk, dv)).astype(np.float32)
    tile = orc.mixed_pack(T, khi)
    lo = lo_region(tile, dk, khi, dv)
    sc = tile[4096 + 112 * 128:].view(np.float32)
    for r in range(khi, dk):
        c, s = orc.quantise_row(T[r])
        assert np.array_equal(lo[r - khi], c)
        assert sc[r - khi] == s
    # the word holding column 5 of INT8 rows khi+4 .. khi+7
    w = tile[4096 + (1 * 128 + 5) * 4: 4096 + (1 * 128 + 5) * 4 + 4].view(np.int8)
    assert np.array_equal(w, lo[4:8, 5])
    # the word holding column 9 of FP16 rows 2, 3
    hw = tile[(1 * 128 + 9) * 4: (1 * 128 + 9) * 4 + 4].view(np.uint16)
    assert np.array_equal(hw, T[2:4, 9].astype(np.float16).view(np.uint16))


def test_convert_places_logical_rows():
    """Physical row r holds logical channel pi[r]: selected channels first,
    each region ascending (DAMP Appendix A.2, Algorithm 1 last step)."""
    dk = dv = 32
    khi = 4
    hi = gen.hi_rows(1, dk, khi, seed=3)
    pi = orc.row_map(hi, dk)[0]
    assert list(pi[:khi]) == sorted(hi[0].tolist())
    assert sorted(pi.tolist()) == list(range(dk))
    assert list(pi[khi:]) == sorted(pi[khi:].tolist())
    g = gen.rng(15)
    S = g.standard_normal((dk, dv)).astype(np.float32)
    tile = orc.convert_f32_to_mixed(S, khi, pi)
    T = orc.mixed_unpack(tile, dk, dv, khi)
    for r in range(dk):
        ref = S[pi[r]]
        if r < khi:
            assert np.array_equal(T[r], ref.astype(np.float16).astype(np.float32))
        else:
            s = orc.row_scale(ref)
            assert np.max(np.abs(T[r] - ref)) <= s * 0.5 * (1 + 2.0 ** -20)
    S_back = orc.convert_mixed_to_f32(tile, dk, dv, khi, pi)
    assert np.array_equal(S_back[pi], T)
