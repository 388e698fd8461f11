"""The C-ABI library on the host (CPU only, no CUDA call).

* The shared library loads and exports every function the header declares.
* Layout and plan objects: sizes, row maps, offsets, validation errors.
* Host-side argument validation returns its status before any launch.
* Storage accounting against the numbers the DAMP page prints.
"""
import ctypes
import json
import os
import re

import numpy as np
import pytest

import oracle as orc
from recurrent_state_gb300 import _abi
from recurrent_state_gb300 import build as rsbuild
from recurrent_state_gb300 import inputs as gen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "recurrent_state.h")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def L():
    rsbuild.build()
    return _abi.lib()


def header_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^(?:rs_status|const char \*)\s*(rs_\w+)\s*\(", text, re.M)))


def test_header_and_binding_agree():
    assert header_functions() == sorted(_abi.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in header_functions():
        assert hasattr(L, name), name
    assert L.rs_version().decode().count(".") == 2


def make_layout(L, kind, dk=128, Hv=32, Hk=16, k_hi=0, hi=None):
    p = _abi.LayoutParams(kind, dk, dk, Hv, Hk, k_hi)
    h = ctypes.c_void_p()
    st = L.rs_layout_create(ctypes.byref(h), ctypes.byref(p),
                            None if hi is None else np.ascontiguousarray(hi, np.int16).ctypes.data)
    return st, h


def head_bytes(L, h):
    nb = ctypes.c_size_t()
    assert L.rs_layout_head_bytes(h, ctypes.byref(nb)) == 0
    return nb.value


def test_layout_sizes_and_accounting(L):
    st, h = make_layout(L, _abi.RS_LAYOUT_FP32)
    assert st == 0 and head_bytes(L, h) == 65536
    L.rs_layout_destroy(h)
    hi = gen.hi_rows(32, 128, 16)
    st, h = make_layout(L, _abi.RS_LAYOUT_MIXED_FP16_INT8, k_hi=16, hi=hi)
    assert st == 0 and head_bytes(L, h) == 18880 == orc.mixed_tile_bytes(128, 128, 16)
    bits = ctypes.c_double()
    assert L.rs_layout_bits_per_value(h, ctypes.byref(bits)) == 0
    # FP16 rows + INT8 rows + one FP32 scale per INT8 row, per value
    assert bits.value == pytest.approx((16 * 16 + 112 * 8 + 112 * 32 / 128) / 128)
    L.rs_layout_destroy(h)


def test_damp_printed_storage_numbers():
    """DAMP prints 9.9 bits per value and a 69.1% reduction for 16 FP16 key
    channels plus INT8 groups of 32 with FP32 scales at d = 128; the closed
    form of that layout reproduces both printed numbers."""
    g = json.load(open(os.path.join(GOLDEN, "accounting.json")))
    d, khi, grp = g["head_dim"], g["k_hi"], g["group"]
    bits = (khi * 16 + (d - khi) * (8 + 32 / grp)) / d
    assert bits == 9.875
    assert round(bits, 1) == g["printed_bits_per_value"]
    assert round(100 * (1 - bits / 32), 1) == g["printed_reduction_percent"]
    assert 32 / 8 == g["int8_ideal_ratio"]


def test_row_map_puts_selected_channels_first(L):
    hi = gen.hi_rows(4, 64, 8, seed=3)
    hi_shuffled = np.ascontiguousarray(hi[:, ::-1])  # order within a head is irrelevant
    st, h = make_layout(L, _abi.RS_LAYOUT_MIXED_FP16_INT8, dk=64, Hv=4, Hk=2, k_hi=8, hi=hi_shuffled)
    assert st == 0
    pi = np.zeros((4, 64), np.int16)
    assert L.rs_layout_row_map(h, pi.ctypes.data) == 0
    assert np.array_equal(pi, orc.row_map(hi, 64))
    L.rs_layout_destroy(h)


@pytest.mark.parametrize("kw,expect", [
    (dict(kind=7), _abi.RS_ERR_INVALID_ARG),
    (dict(dk=96), _abi.RS_ERR_UNSUPPORTED),
    (dict(Hv=32, Hk=5), _abi.RS_ERR_INVALID_ARG),
    (dict(Hv=0), _abi.RS_ERR_INVALID_ARG),
    (dict(k_hi=4), _abi.RS_ERR_INVALID_ARG),                  # FP32 layout with FP16 rows
    (dict(kind=1, k_hi=16, hi="none"), _abi.RS_ERR_INVALID_ARG),
    (dict(kind=1, k_hi=16, hi="dup"), _abi.RS_ERR_INVALID_ARG),
    (dict(kind=1, k_hi=16, hi="range"), _abi.RS_ERR_INVALID_ARG),
])
def test_layout_validation(L, kw, expect):
    kind = kw.get("kind", 0)
    dk, Hv, Hk, k_hi = kw.get("dk", 128), kw.get("Hv", 32), kw.get("Hk", 16), kw.get("k_hi", 0)
    hi = None
    if kw.get("hi") == "dup":
        hi = gen.hi_rows(Hv, dk, k_hi)
        hi[3, 1] = hi[3, 0]
    elif kw.get("hi") == "range":
        hi = gen.hi_rows(Hv, dk, k_hi)
        hi[0, 0] = dk
    st, h = make_layout(L, kind, dk=dk, Hv=Hv, Hk=Hk, k_hi=k_hi, hi=hi)
    assert st == expect
    assert not h.value


def test_layout_size_limits():
    """The row map (8,192 bytes) and the value-scaling table (4,096 floats)
    travel in the launch parameters: one head more than fits is refused at
    layout creation; the largest that fits is accepted."""
    import recurrent_state_gb300 as rs
    for Hv, Hk, ok in ((64, 8, True), (72, 8, False)):
        if ok:
            rs.Layout("mixed", 128, Hv, Hk, k_hi=16, hi_rows=gen.hi_rows(Hv, 128, 16))
        else:
            with pytest.raises(_abi.RsError) as e:
                rs.Layout("mixed", 128, Hv, Hk, k_hi=16, hi_rows=gen.hi_rows(Hv, 128, 16))
            assert e.value.status == _abi.RS_ERR_UNSUPPORTED
    for Hv, Hk, ok in ((32, 4, True), (36, 4, False)):
        if ok:
            rs.Layout("damp", 128, Hv, Hk, k_hi=16, hi_rows=gen.hi_rows(Hv, 128, 16))
        else:
            with pytest.raises(_abi.RsError) as e:
                rs.Layout("damp", 128, Hv, Hk, k_hi=16, hi_rows=gen.hi_rows(Hv, 128, 16))
            assert e.value.status == _abi.RS_ERR_UNSUPPORTED


def test_host_validation_returns_before_launch(L):
    st, h = make_layout(L, _abi.RS_LAYOUT_FP32, dk=64, Hv=4, Hk=4)
    assert st == 0
    fake = ctypes.c_void_p(1 << 20)       # never dereferenced: validation fails first
    odd = ctypes.c_void_p((1 << 20) + 4)  # not 16-byte aligned
    f = L.rs_gdn_decode_update
    # B = 0 is a no-op, even with NULL pointers
    assert f(h, None, 0, None, 0, None, None, None, 0, None, None, None, 0, None, None) == 0
    # NULL input with B > 0
    assert f(h, fake, 4, fake, 4, None, fake, fake, 0, fake, fake, None, 0, None, None) == \
        _abi.RS_ERR_INVALID_ARG
    # misaligned q
    assert f(h, fake, 4, fake, 4, odd, fake, fake, 0, fake, fake, None, 0, None, None) == \
        _abi.RS_ERR_MISALIGNED
    # bad dtype
    assert f(h, fake, 4, fake, 4, fake, fake, fake, 9, fake, fake, None, 0, None, None) == \
        _abi.RS_ERR_INVALID_ARG
    # replay: T_max outside 1..8, per_channel flag not 0/1
    r = L.rs_spec_replay_update
    assert r(h, 0, fake, 4, fake, 4, 9, fake, fake, fake, fake, 0, fake, fake, None, 0, None,
             None) == _abi.RS_ERR_INVALID_ARG
    assert r(h, 2, fake, 4, fake, 4, 2, fake, fake, fake, fake, 0, fake, fake, None, 0, None,
             None) == _abi.RS_ERR_INVALID_ARG
    # prefill: L = 0 or B = 0 is a no-op; negative L, a bad flag, NULL or
    # misaligned inputs fail before any launch
    p = L.rs_prefill_update
    assert p(h, 0, None, 0, None, 4, 0, None, None, None, None, 0, None, None, None, 0, None, None) == 0
    assert p(h, 0, None, 0, None, 0, 7, None, None, None, None, 0, None, None, None, 0, None, None) == 0
    assert p(h, 0, fake, 4, fake, 4, -1, None, fake, fake, fake, 0, fake, fake, None, 0, None, None) == \
        _abi.RS_ERR_INVALID_ARG
    assert p(h, 3, fake, 4, fake, 4, 5, None, fake, fake, fake, 0, fake, fake, None, 0, None, None) == \
        _abi.RS_ERR_INVALID_ARG
    assert p(h, 1, fake, 4, fake, 4, 5, None, fake, None, fake, 0, fake, fake, None, 0, None, None) == \
        _abi.RS_ERR_INVALID_ARG
    assert p(h, 1, fake, 4, fake, 4, 5, None, fake, fake, fake, 0, odd, fake, None, 0, None, None) == \
        _abi.RS_ERR_MISALIGNED
    # fp16 inputs with a bf16 readout are not built: refused before any launch
    assert f(h, fake, 4, fake, 4, fake, fake, fake, _abi.RS_F16, fake, fake, None, _abi.RS_BF16, None, None) == \
        _abi.RS_ERR_UNSUPPORTED
    # quantisation mode: FP32 layouts take only the IEEE mode
    assert L.rs_layout_set_quant(h, _abi.RS_QUANT_FUSED) == _abi.RS_ERR_INVALID_ARG
    assert L.rs_layout_set_quant(h, 7) == _abi.RS_ERR_INVALID_ARG
    mode = ctypes.c_int32(-1)
    assert L.rs_layout_quant(h, ctypes.byref(mode)) == 0 and mode.value == _abi.RS_QUANT_IEEE
    L.rs_layout_destroy(h)


def test_noalloc_pack_refuses_a_plan_one_unit_beyond_its_table(L):
    """rs_ckpt_pack_noalloc holds at most 262,144 retained units; one more is
    refused on the host, before any CUDA call (the pointers are never read)."""
    st, lay = make_layout(L, _abi.RS_LAYOUT_FP32, dk=64, Hv=64, Hk=1)
    assert st == 0
    keep = np.zeros((65, 64 * 64), np.uint8)
    keep[:64] = 1
    keep[64, 17] = 1  # 262,145 retained units
    plan = ctypes.c_void_p()
    assert L.rs_plan_create(ctypes.byref(plan), lay, 65, _abi.RS_UNIT_CHANNEL,
                            keep.ctypes.data) == 0
    fake = ctypes.c_void_p(1 << 20)
    assert L.rs_ckpt_pack_noalloc(plan, fake, 1 << 24, 1, fake, fake, 1, fake, 1, None,
                                  None) == _abi.RS_ERR_UNSUPPORTED
    L.rs_plan_destroy(plan)
    L.rs_layout_destroy(lay)


def test_plan_offsets_match_golden_and_oracle(L):
    g = json.load(open(os.path.join(GOLDEN, "dasc_offsets.json")))
    keep = np.array(g["keep"], np.uint8)
    st, lay = make_layout(L, _abi.RS_LAYOUT_FP32, dk=64, Hv=keep.shape[1], Hk=1)
    assert st == 0
    ph = ctypes.c_void_p()
    assert L.rs_plan_create(ctypes.byref(ph), lay, keep.shape[0], _abi.RS_UNIT_HEAD,
                            keep.ctypes.data) == 0
    off = np.zeros(keep.shape[0] + 1, np.int64)
    ub = ctypes.c_int64()
    assert L.rs_plan_offsets(ph, off.ctypes.data, ctypes.byref(ub)) == 0
    assert off.tolist() == g["offsets"]
    assert ub.value == 64 * 64 * 4
    L.rs_plan_destroy(ph)
    # random KDA plans against the oracle's offsets
    Hv = keep.shape[1]
    for seed in range(3):
        keep = gen.keep_mask(36, Hv * 64, 0.45, seed=seed)
        assert L.rs_plan_create(ctypes.byref(ph), lay, 36, _abi.RS_UNIT_CHANNEL,
                                keep.ctypes.data) == 0
        off = np.zeros(37, np.int64)
        assert L.rs_plan_offsets(ph, off.ctypes.data, ctypes.byref(ub)) == 0
        assert np.array_equal(off, orc.plan_offsets(keep, Hv, 64, 1))
        assert ub.value == 64 * 4
        L.rs_plan_destroy(ph)
    bad = np.full((2, 8), 2, np.uint8)
    assert L.rs_plan_create(ctypes.byref(ph), lay, 2, _abi.RS_UNIT_HEAD, bad.ctypes.data) == \
        _abi.RS_ERR_INVALID_ARG
    L.rs_layout_destroy(lay)


def test_status_strings(L):
    for s in (0, -1, -2, -3, -4):
        assert L.rs_status_string(s).decode()


def test_mixed_head_plans_and_int8_checkpoint_sizes(L):
    """Mixed layouts take head units (a packed head is one unit); INT8
    checkpoint slots hold codes then one FP32 scale per row (dasc Appendix
    E.1), sizes agreeing with the oracle's."""
    Hv, d = 4, 128
    hi = np.stack([np.arange(16, dtype=np.int16) * 3 + h for h in range(Hv)])
    st, mix = make_layout(L, _abi.RS_LAYOUT_MIXED_FP16_INT8, dk=d, Hv=Hv, Hk=Hv, k_hi=16, hi=hi)
    assert st == 0
    keep = gen.keep_mask(3, Hv, 0.5, seed=1)
    ph = ctypes.c_void_p()
    assert L.rs_plan_create(ctypes.byref(ph), mix, 3, _abi.RS_UNIT_HEAD, keep.ctypes.data) == 0
    off = np.zeros(4, np.int64)
    ub = ctypes.c_int64()
    assert L.rs_plan_offsets(ph, off.ctypes.data, ctypes.byref(ub)) == 0
    assert ub.value == 18880 and off[-1] == keep.sum()
    cb, sb = ctypes.c_int64(), ctypes.c_int64()
    assert L.rs_ckpt_int8_bytes(ph, ctypes.byref(cb), ctypes.byref(sb)) == _abi.RS_ERR_UNSUPPORTED
    L.rs_plan_destroy(ph)
    keep_c = gen.keep_mask(3, Hv * d, 0.5, seed=2)
    assert L.rs_plan_create(ctypes.byref(ph), mix, 3, _abi.RS_UNIT_CHANNEL, keep_c.ctypes.data) == \
        _abi.RS_ERR_UNSUPPORTED
    L.rs_layout_destroy(mix)
    st, f32 = make_layout(L, _abi.RS_LAYOUT_FP32, dk=d, Hv=Hv, Hk=Hv)
    for unit, kp in ((_abi.RS_UNIT_HEAD, keep), (_abi.RS_UNIT_CHANNEL, keep_c)):
        assert L.rs_plan_create(ctypes.byref(ph), f32, 3, unit, kp.ctypes.data) == 0
        assert L.rs_ckpt_int8_bytes(ph, ctypes.byref(cb), ctypes.byref(sb)) == 0
        assert (cb.value, sb.value) == orc.ckpt_int8_layout(int(kp.sum()), unit, d, d)
        L.rs_plan_destroy(ph)
    L.rs_layout_destroy(f32)
