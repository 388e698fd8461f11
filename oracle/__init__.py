"""CPU oracle for the recurrent-state hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` import this package.  The product library never does, and
this package never imports the product library: the two share no code.

The arithmetic lives in ``rs_oracle.c`` (plain C loops, IEEE binary32,
``-ffp-contract=off``); this module only builds it with gcc and marshals numpy
arrays through ctypes.  Page citations are in the C source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rs_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
# Each result below depends on these flags: no contraction of a*b+c into an
# FMA, no fast-math reassociation, IEEE division and rounding.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
          "-fno-unsafe-math-optimizations", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``rs_oracle.c`` into ``_build/liboracle.so`` (gcc)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
        return _lib


def build_variant(source: str, out_path: str) -> str:
    """Compile an edited copy of the oracle source (used by the mutation test
    that checks the pins catch planted mistakes)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source)
    subprocess.check_call(["gcc", *CFLAGS, src, "-o", out_path, "-lm"])
    return out_path


class use_library:
    """Context manager: route every call of this module through another build
    of the oracle (a planted-mistake variant), then restore the real one."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self._saved = lib()
        variant = ctypes.CDLL(self.path)
        _declare(variant)
        with _lock:
            _lib = variant
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self._saved
        return False


def source() -> str:
    with open(_SRC) as f:
        return f.read()


_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_I64 = ctypes.c_int64


def _declare(L):
    L.orc_row_map.argtypes = [_I, _I, _P, _P]
    L.orc_row_map.restype = _I
    L.orc_step_tile_f32.argtypes = [_I, _I, _P, _P, _P, _P, _P, _I, _F, _P]
    L.orc_step_tile_f32.restype = None
    L.orc_row_scale.argtypes = [_I, _P]
    L.orc_row_scale.restype = _F
    L.orc_quant_code.argtypes = [_F, _F]
    L.orc_quant_code.restype = ctypes.c_int8
    L.orc_quantise_row.argtypes = [_I, _P, _P, _P]
    L.orc_quant_code_rcp.argtypes = [_F, _F]
    L.orc_quant_code_rcp.restype = ctypes.c_int8
    L.orc_quantise_row_m.argtypes = [_I, _P, _I, _P, _P]
    L.orc_mixed_pack_m.argtypes = [_I, _I, _I, _I, _P, _P]
    L.orc_convert_f32_to_mixed_m.argtypes = [_I, _I, _I, _I, _P, _P, _P]
    L.orc_convert_f32_to_mixed_m.restype = _I
    L.orc_decode_mixed_m.argtypes = [_I, _I, _I, _I, _I, _I, _I, _I, _P, _I, _P, _P, _P,
                                     _P, _P, _P, _P, _P, _I, _I]
    L.orc_decode_mixed_m.restype = _I
    L.orc_replay_mixed_m.argtypes = [_I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _I, _P, _P,
                                     _P, _P, _P, _P, _P, _P, _P, _I, _I]
    L.orc_replay_mixed_m.restype = _I
    L.orc_damp_pack_m.argtypes = [_I, _I, _I, _I, _I, _P, _P]
    L.orc_convert_f32_to_damp_m.argtypes = [_I, _I, _I, _I, _I, _P, _P, _P, _P]
    L.orc_convert_f32_to_damp_m.restype = _I
    L.orc_decode_damp_m.argtypes = [_I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _I, _P, _P, _P, _P,
                                    _P, _P, _P, _P, _P, _I, _I]
    L.orc_decode_damp_m.restype = _I
    L.orc_replay_damp_m.argtypes = [_I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _I, _P, _P, _P,
                                    _P, _P, _P, _P, _P, _P, _P, _I, _I]
    L.orc_replay_damp_m.restype = _I
    L.orc_dequantise_row.argtypes = [_I, _P, _F, _P]
    L.orc_mixed_tile_bytes.argtypes = [_I, _I, _I]
    L.orc_mixed_tile_bytes.restype = ctypes.c_size_t
    L.orc_mixed_unpack.argtypes = [_I, _I, _I, _P, _P]
    L.orc_mixed_pack.argtypes = [_I, _I, _I, _P, _P]
    L.orc_convert_f32_to_mixed.argtypes = [_I, _I, _I, _P, _P, _P]
    L.orc_convert_f32_to_mixed.restype = _I
    L.orc_convert_mixed_to_f32.argtypes = [_I, _I, _I, _P, _P, _P]
    L.orc_convert_mixed_to_f32.restype = _I
    L.orc_decode_f32.argtypes = [_I, _I, _I, _I, _I, _I, _P, _I, _P, _P, _P, _P,
                                 _P, _P, _P, _I, _I]
    L.orc_decode_f32.restype = _I
    L.orc_decode_mixed.argtypes = [_I, _I, _I, _I, _I, _I, _I, _P, _I, _P, _P, _P,
                                   _P, _P, _P, _P, _P, _I, _I]
    L.orc_decode_mixed.restype = _I
    L.orc_replay_f32.argtypes = [_I, _I, _I, _I, _I, _I, _I, _P, _I, _P, _P, _P,
                                 _P, _P, _P, _P, _P, _I, _I]
    L.orc_replay_f32.restype = _I
    L.orc_replay_mixed.argtypes = [_I, _I, _I, _I, _I, _I, _I, _I, _P, _I, _P, _P,
                                   _P, _P, _P, _P, _P, _P, _P, _I, _I]
    L.orc_replay_mixed.restype = _I
    L.orc_plan_offsets.argtypes = [_I, _I, _I, _I, _P, _P]
    L.orc_ckpt_pack.argtypes = [_I, _I, _I, _I, _I, _P, _P, _I64, _I, _P, _P, _I,
                                _P, _I]
    L.orc_ckpt_pack.restype = _I
    L.orc_ckpt_restore.argtypes = [_I, _I, _I, _I, _I, _P, _P, _I, _P, _P, _I64,
                                   _I, _P, _I]
    L.orc_ckpt_restore.restype = _I
    L.orc_damp_tile_bytes.argtypes = [_I, _I, _I, _I]
    L.orc_damp_tile_bytes.restype = ctypes.c_size_t
    L.orc_damp_unpack.argtypes = [_I, _I, _I, _I, _P, _P]
    L.orc_damp_pack.argtypes = [_I, _I, _I, _I, _P, _P]
    L.orc_convert_f32_to_damp.argtypes = [_I, _I, _I, _I, _P, _P, _P, _P]
    L.orc_convert_f32_to_damp.restype = _I
    L.orc_convert_damp_to_f32.argtypes = [_I, _I, _I, _I, _P, _P, _P, _P]
    L.orc_convert_damp_to_f32.restype = _I
    L.orc_decode_damp.argtypes = [_I, _I, _I, _I, _I, _I, _I, _I, _P, _I, _P, _P, _P, _P, _P, _P,
                                  _P, _P, _P, _I, _I]
    L.orc_decode_damp.restype = _I
    L.orc_replay_damp.argtypes = [_I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _I, _P, _P, _P, _P, _P,
                                  _P, _P, _P, _P, _P, _I, _I]
    L.orc_replay_damp.restype = _I
    L.orc_ckpt_pack_heads.argtypes = [_I, _I, _I64, _P, _P, _I64, _I, _P, _P, _I, _P, _I]
    L.orc_ckpt_pack_heads.restype = _I
    L.orc_ckpt_restore_heads.argtypes = [_I, _I, _I64, _P, _P, _I, _P, _P, _I64, _I, _P, _I]
    L.orc_ckpt_restore_heads.restype = _I
    L.orc_ckpt_int8_codes_bytes.argtypes = [_I64, _I, _I]
    L.orc_ckpt_int8_codes_bytes.restype = _I64
    L.orc_ckpt_int8_slot_bytes.argtypes = [_I64, _I, _I]
    L.orc_ckpt_int8_slot_bytes.restype = _I64
    L.orc_ckpt_pack_int8.argtypes = [_I, _I, _I, _I, _I, _P, _P, _I64, _I, _P, _P, _I, _P, _I]
    L.orc_ckpt_pack_int8.restype = _I
    L.orc_ckpt_restore_int8.argtypes = [_I, _I, _I, _I, _I, _P, _P, _I, _P, _P, _I64, _I, _P, _I]
    L.orc_ckpt_restore_int8.restype = _I


# --------------------------------------------------------------------------
# numpy marshalling helpers
# --------------------------------------------------------------------------
def _c(a: np.ndarray, dtype) -> np.ndarray:
    if a.dtype != dtype or not a.flags["C_CONTIGUOUS"]:
        raise TypeError(f"expected C-contiguous {np.dtype(dtype)}, got {a.dtype}")
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data


def row_map(hi, dk):
    """Row map of every head: ``hi`` int [Hv][k_hi] selected key channels
    (any order) -> int16 [Hv][dk], physical row r holding logical channel
    pi[r] (the selected channels first, each region ascending)."""
    hi = np.ascontiguousarray(np.asarray(hi).reshape(len(hi), -1), np.int16)
    out = np.empty((hi.shape[0], dk), np.int16)
    for h in range(hi.shape[0]):
        row = np.ascontiguousarray(hi[h])
        dst = out[h]
        if lib().orc_row_map(dk, row.size, _ptr(row), _ptr(dst)) != 0:
            raise ValueError(f"head {h}: selection must be distinct channels in [0, {dk})")
    return out


def step_tile(S, q, k, v, a, beta, want_o=True):
    """One decode step on one tile, in place on ``S`` [dk][dv] (float32).
    ``a`` is a float32 scalar array of shape () / (1,) for GDN or (dk,) for KDA."""
    dk, dv = S.shape
    _c(S, np.float32)
    q = np.ascontiguousarray(q, np.float32)
    k = np.ascontiguousarray(k, np.float32)
    v = np.ascontiguousarray(v, np.float32)
    a = np.ascontiguousarray(np.atleast_1d(a), np.float32)
    o = np.zeros(dv, np.float32) if want_o else None
    lib().orc_step_tile_f32(dk, dv, _ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(a),
                            0 if a.size == 1 else 1, float(np.float32(beta)), _ptr(o))
    return o


def row_scale(x):
    x = np.ascontiguousarray(x, np.float32)
    return np.float32(lib().orc_row_scale(x.size, _ptr(x)))


def quantise_row(x, mode=0):
    """Codes and scale of one INT8 row; ``mode`` 0 (IEEE quotient) or 1 (fused
    reciprocal arithmetic, see ``orc_quant_code_rcp`` in the C source)."""
    x = np.ascontiguousarray(x, np.float32)
    codes = np.zeros(x.size, np.int8)
    s = np.zeros(1, np.float32)
    lib().orc_quantise_row_m(x.size, _ptr(x), int(mode), _ptr(codes), _ptr(s))
    return codes, s[0]


def quant_code_rcp(x, y):
    """Mode-1 code of ``x`` given y = RN(1/s)."""
    return int(lib().orc_quant_code_rcp(float(np.float32(x)), float(np.float32(y))))


def dequantise_row(codes, s):
    codes = np.ascontiguousarray(codes, np.int8)
    x = np.zeros(codes.size, np.float32)
    lib().orc_dequantise_row(codes.size, _ptr(codes), float(np.float32(s)), _ptr(x))
    return x


def mixed_tile_bytes(dk, dv, khi):
    return int(lib().orc_mixed_tile_bytes(dk, dv, khi))


def mixed_unpack(tile, dk, dv, khi):
    tile = _c(np.ascontiguousarray(tile), np.uint8)
    T = np.zeros((dk, dv), np.float32)
    lib().orc_mixed_unpack(dk, dv, khi, _ptr(tile), _ptr(T))
    return T


def mixed_pack(T, khi, mode=0):
    T = _c(np.ascontiguousarray(T), np.float32)
    dk, dv = T.shape
    tile = np.zeros(mixed_tile_bytes(dk, dv, khi), np.uint8)
    lib().orc_mixed_pack_m(dk, dv, khi, int(mode), _ptr(T), _ptr(tile))
    return tile


def convert_f32_to_mixed(S, khi, pi, mode=0):
    """Logical FP32 head ``S`` [dk][dv] -> mixed tile bytes with row map ``pi``."""
    S = _c(np.ascontiguousarray(S), np.float32)
    dk, dv = S.shape
    pi = np.ascontiguousarray(pi, np.int16)
    tile = np.zeros(mixed_tile_bytes(dk, dv, khi), np.uint8)
    assert lib().orc_convert_f32_to_mixed_m(dk, dv, khi, int(mode), _ptr(pi), _ptr(S), _ptr(tile)) == 0
    return tile


def convert_mixed_to_f32(tile, dk, dv, khi, pi):
    tile = _c(np.ascontiguousarray(tile), np.uint8)
    pi = np.ascontiguousarray(pi, np.int16)
    S = np.zeros((dk, dv), np.float32)
    assert lib().orc_convert_mixed_to_f32(dk, dv, khi, _ptr(pi), _ptr(tile), _ptr(S)) == 0
    return S


def convert_pool_f32_to_mixed(pool, khi, pi, mode=0):
    """[..., Hv, dk, dv] float32 -> [..., Hv, tile_bytes] uint8; pi [Hv][dk]."""
    *lead, Hv, dk, dv = pool.shape
    flat = pool.reshape(-1, Hv, dk, dv)
    out = np.zeros((flat.shape[0], Hv, mixed_tile_bytes(dk, dv, khi)), np.uint8)
    for s in range(flat.shape[0]):
        for h in range(Hv):
            out[s, h] = convert_f32_to_mixed(np.ascontiguousarray(flat[s, h]), khi, pi[h], mode)
    return out.reshape(*lead, Hv, out.shape[-1])


def convert_pool_mixed_to_f32(pool, dk, dv, khi, pi):
    *lead, Hv, tb = pool.shape
    flat = pool.reshape(-1, Hv, tb)
    out = np.zeros((flat.shape[0], Hv, dk, dv), np.float32)
    for s in range(flat.shape[0]):
        for h in range(Hv):
            out[s, h] = convert_mixed_to_f32(np.ascontiguousarray(flat[s, h]), dk, dv, khi, pi[h])
    return out.reshape(*lead, Hv, dk, dv)


def decode_f32(pool, slot_idx, q, k, v, alpha, beta, o=None, per_channel=None,
               items=None):
    """Batched FP32 decode step in place on ``pool`` [n_slots][Hv][dk][dv].
    q, k: [B][Hk][dk]; v: [B][Hv][dv]; alpha: [B][Hv] or [B][Hv][dk];
    beta: [B][Hv].  Returns (o [B][Hv][dv], status bits)."""
    _c(pool, np.float32)
    n_slots, Hv, dk, dv = pool.shape
    B, Hk, _ = q.shape
    if per_channel is None:
        per_channel = alpha.ndim == 3
    if o is None:
        o = np.zeros((B, Hv, dv), np.float32)
    lo, hi = items if items is not None else (0, B * Hv)
    st = lib().orc_decode_f32(B, Hk, Hv, dk, dv, int(per_channel), _ptr(pool), n_slots,
                              _ptr(_c(slot_idx, np.int32)), _ptr(_c(q, np.float32)),
                              _ptr(_c(k, np.float32)), _ptr(_c(v, np.float32)),
                              _ptr(_c(alpha, np.float32)), _ptr(_c(beta, np.float32)),
                              _ptr(_c(o, np.float32)), lo, hi)
    return o, st


def decode_mixed(pool, slot_idx, pi, khi, dk, dv, q, k, v, alpha, beta, o=None,
                 per_channel=None, items=None, mode=0):
    """Batched mixed-layout decode in place on ``pool`` [n_slots][Hv][tile_bytes];
    ``mode`` selects the requantisation arithmetic (0 IEEE, 1 fused)."""
    _c(pool, np.uint8)
    n_slots, Hv, tb = pool.shape
    assert tb == mixed_tile_bytes(dk, dv, khi)
    B, Hk, _ = q.shape
    if per_channel is None:
        per_channel = alpha.ndim == 3
    if o is None:
        o = np.zeros((B, Hv, dv), np.float32)
    lo, hi = items if items is not None else (0, B * Hv)
    st = lib().orc_decode_mixed_m(B, Hk, Hv, dk, dv, khi, int(per_channel), int(mode), _ptr(pool),
                                n_slots, _ptr(_c(slot_idx, np.int32)),
                                _ptr(_c(pi, np.int16)), _ptr(_c(q, np.float32)),
                                _ptr(_c(k, np.float32)), _ptr(_c(v, np.float32)),
                                _ptr(_c(alpha, np.float32)), _ptr(_c(beta, np.float32)),
                                _ptr(_c(o, np.float32)), lo, hi)
    return o, st


def replay_f32(pool, slot_idx, n_accept, q, k, v, alpha, beta, o=None,
               per_channel=None, items=None):
    """Spec replay on the FP32 pool. Inputs are [B][T_max][...]."""
    _c(pool, np.float32)
    n_slots, Hv, dk, dv = pool.shape
    B, T_max, Hk, _ = q.shape
    if per_channel is None:
        per_channel = alpha.ndim == 4
    if o is None:
        o = np.zeros((B, T_max, Hv, dv), np.float32)
    lo, hi = items if items is not None else (0, B * Hv)
    st = lib().orc_replay_f32(B, T_max, Hk, Hv, dk, dv, int(per_channel), _ptr(pool),
                              n_slots, _ptr(_c(slot_idx, np.int32)),
                              _ptr(_c(n_accept, np.int32)), _ptr(_c(q, np.float32)),
                              _ptr(_c(k, np.float32)), _ptr(_c(v, np.float32)),
                              _ptr(_c(alpha, np.float32)), _ptr(_c(beta, np.float32)),
                              _ptr(_c(o, np.float32)), lo, hi)
    return o, st


def replay_mixed(pool, slot_idx, n_accept, pi, khi, dk, dv, q, k, v, alpha, beta,
                 o=None, per_channel=None, items=None, mode=0):
    _c(pool, np.uint8)
    n_slots, Hv, tb = pool.shape
    assert tb == mixed_tile_bytes(dk, dv, khi)
    B, T_max, Hk, _ = q.shape
    if per_channel is None:
        per_channel = alpha.ndim == 4
    if o is None:
        o = np.zeros((B, T_max, Hv, dv), np.float32)
    lo, hi = items if items is not None else (0, B * Hv)
    st = lib().orc_replay_mixed_m(B, T_max, Hk, Hv, dk, dv, khi, int(per_channel), int(mode),
                                _ptr(pool), n_slots, _ptr(_c(slot_idx, np.int32)),
                                _ptr(_c(n_accept, np.int32)), _ptr(_c(pi, np.int16)),
                                _ptr(_c(q, np.float32)), _ptr(_c(k, np.float32)),
                                _ptr(_c(v, np.float32)), _ptr(_c(alpha, np.float32)),
                                _ptr(_c(beta, np.float32)), _ptr(_c(o, np.float32)), lo, hi)
    return o, st


def plan_offsets(keep, Hv, dk, unit):
    """o_0..o_L for keep [L][n_units] (uint8)."""
    keep = _c(np.ascontiguousarray(keep, np.uint8), np.uint8)
    L = keep.shape[0]
    off = np.zeros(L + 1, np.int64)
    lib().orc_plan_offsets(L, Hv, dk, unit, _ptr(keep), _ptr(off))
    return off


def ckpt_pack(keep, unit, pool, src_slots, dst_slots, ckpt):
    """pool: [L][n_slots][Hv][dk][dv] float32; ckpt: [n_ckpt][total_units*unit_bytes] uint8."""
    keep = _c(np.ascontiguousarray(keep, np.uint8), np.uint8)
    L, n_slots, Hv, dk, dv = pool.shape
    st = lib().orc_ckpt_pack(L, Hv, dk, dv, unit, _ptr(keep), _ptr(_c(pool, np.float32)),
                             pool.strides[0], n_slots, _ptr(_c(src_slots, np.int32)),
                             _ptr(_c(dst_slots, np.int32)), len(src_slots),
                             _ptr(_c(ckpt, np.uint8)), ckpt.shape[0])
    return st


def ckpt_restore(keep, unit, ckpt, src_slots, pool, dst_slots):
    keep = _c(np.ascontiguousarray(keep, np.uint8), np.uint8)
    L, n_slots, Hv, dk, dv = pool.shape
    st = lib().orc_ckpt_restore(L, Hv, dk, dv, unit, _ptr(keep), _ptr(_c(ckpt, np.uint8)),
                                ckpt.shape[0], _ptr(_c(src_slots, np.int32)),
                                _ptr(_c(pool, np.float32)), pool.strides[0], n_slots,
                                _ptr(_c(dst_slots, np.int32)), len(src_slots))
    return st


def ckpt_pack_heads(keep, pool, src_slots, dst_slots, ckpt):
    """Whole-head checkpoint of a packed pool: pool [L][n_slots][Hv][head_bytes]
    uint8, keep [L][Hv]; ckpt [n_ckpt][o_L * head_bytes] uint8."""
    keep = _c(np.ascontiguousarray(keep, np.uint8), np.uint8)
    L, n_slots, Hv, hb = pool.shape
    return lib().orc_ckpt_pack_heads(L, Hv, hb, _ptr(keep), _ptr(_c(pool, np.uint8)), pool.strides[0],
                                     n_slots, _ptr(_c(src_slots, np.int32)),
                                     _ptr(_c(dst_slots, np.int32)), len(src_slots),
                                     _ptr(_c(ckpt, np.uint8)), ckpt.shape[0])


def ckpt_restore_heads(keep, ckpt, src_slots, pool, dst_slots):
    keep = _c(np.ascontiguousarray(keep, np.uint8), np.uint8)
    L, n_slots, Hv, hb = pool.shape
    return lib().orc_ckpt_restore_heads(L, Hv, hb, _ptr(keep), _ptr(_c(ckpt, np.uint8)), ckpt.shape[0],
                                        _ptr(_c(src_slots, np.int32)), _ptr(_c(pool, np.uint8)),
                                        pool.strides[0], n_slots, _ptr(_c(dst_slots, np.int32)),
                                        len(src_slots))


def ckpt_int8_layout(n_kept, unit, dk, dv):
    """(codes bytes, slot bytes) of one INT8 checkpoint slot."""
    rows = 1 if unit else dk
    return (lib().orc_ckpt_int8_codes_bytes(n_kept, rows, dv),
            lib().orc_ckpt_int8_slot_bytes(n_kept, rows, dv))


def ckpt_pack_int8(keep, unit, pool, src_slots, dst_slots, ckpt):
    """INT8 checkpoint of an FP32 pool [L][n_slots][Hv][dk][dv]; ckpt
    [n_ckpt][slot_bytes] uint8 (codes, then scales)."""
    keep = _c(np.ascontiguousarray(keep, np.uint8), np.uint8)
    L, n_slots, Hv, dk, dv = pool.shape
    return lib().orc_ckpt_pack_int8(L, Hv, dk, dv, unit, _ptr(keep), _ptr(_c(pool, np.float32)),
                                    pool.strides[0] // 4, n_slots, _ptr(_c(src_slots, np.int32)),
                                    _ptr(_c(dst_slots, np.int32)), len(src_slots),
                                    _ptr(_c(ckpt, np.uint8)), ckpt.shape[0])


def ckpt_restore_int8(keep, unit, ckpt, src_slots, pool, dst_slots):
    keep = _c(np.ascontiguousarray(keep, np.uint8), np.uint8)
    L, n_slots, Hv, dk, dv = pool.shape
    return lib().orc_ckpt_restore_int8(L, Hv, dk, dv, unit, _ptr(keep), _ptr(_c(ckpt, np.uint8)),
                                       ckpt.shape[0], _ptr(_c(src_slots, np.int32)),
                                       _ptr(_c(pool, np.float32)), pool.strides[0] // 4, n_slots,
                                       _ptr(_c(dst_slots, np.int32)), len(src_slots))


# --------------------------------------------------------------------------
# DAMP-exact storage: INT8 groups along dv, value scaling (DAMP Appendix A.1,
# A.3 Eq. 17-18, A.4)
# --------------------------------------------------------------------------
def damp_tile_bytes(dk, dv, khi, group):
    return int(lib().orc_damp_tile_bytes(dk, dv, khi, group))


def damp_unpack(tile, dk, dv, khi, group):
    tile = _c(np.ascontiguousarray(tile), np.uint8)
    T = np.zeros((dk, dv), np.float32)
    lib().orc_damp_unpack(dk, dv, khi, group, _ptr(tile), _ptr(T))
    return T


def damp_pack(T, khi, group, mode=0):
    T = _c(np.ascontiguousarray(T), np.float32)
    dk, dv = T.shape
    tile = np.zeros(damp_tile_bytes(dk, dv, khi, group), np.uint8)
    lib().orc_damp_pack_m(dk, dv, khi, group, int(mode), _ptr(T), _ptr(tile))
    return tile


def convert_pool_f32_to_damp(pool, khi, group, pi, cs, mode=0):
    """[..., Hv, dk, dv] float32 -> [..., Hv, tile_bytes] uint8; pi [Hv][dk],
    cs [Hv][dv] value-scaling factors."""
    *lead, Hv, dk, dv = pool.shape
    flat = pool.reshape(-1, Hv, dk, dv)
    pi = np.ascontiguousarray(pi, np.int16)
    cs = _c(np.ascontiguousarray(cs, np.float32), np.float32)
    out = np.zeros((flat.shape[0], Hv, damp_tile_bytes(dk, dv, khi, group)), np.uint8)
    for s in range(flat.shape[0]):
        for h in range(Hv):
            S = np.ascontiguousarray(flat[s, h])
            assert lib().orc_convert_f32_to_damp_m(dk, dv, khi, group, int(mode), _ptr(pi[h]),
                                                   _ptr(cs[h]), _ptr(S), _ptr(out[s, h])) == 0
    return out.reshape(*lead, Hv, out.shape[-1])


def convert_pool_damp_to_f32(pool, dk, dv, khi, group, pi, cs):
    *lead, Hv, tb = pool.shape
    flat = np.ascontiguousarray(pool.reshape(-1, Hv, tb))
    pi = np.ascontiguousarray(pi, np.int16)
    cs = _c(np.ascontiguousarray(cs, np.float32), np.float32)
    out = np.zeros((flat.shape[0], Hv, dk, dv), np.float32)
    for s in range(flat.shape[0]):
        for h in range(Hv):
            assert lib().orc_convert_damp_to_f32(dk, dv, khi, group, _ptr(pi[h]), _ptr(cs[h]),
                                                 _ptr(flat[s, h]), _ptr(out[s, h])) == 0
    return out.reshape(*lead, Hv, dk, dv)


def decode_damp(pool, slot_idx, pi, cs, khi, group, dk, dv, q, k, v, alpha, beta, o=None,
                per_channel=None, items=None, mode=0):
    """Batched DAMP-exact decode in place on ``pool`` [n_slots][Hv][tile_bytes]."""
    _c(pool, np.uint8)
    n_slots, Hv, tb = pool.shape
    assert tb == damp_tile_bytes(dk, dv, khi, group)
    B, Hk, _ = q.shape
    if per_channel is None:
        per_channel = alpha.ndim == 3
    if o is None:
        o = np.zeros((B, Hv, dv), np.float32)
    lo, hi = items if items is not None else (0, B * Hv)
    st = lib().orc_decode_damp_m(B, Hk, Hv, dk, dv, khi, group, int(per_channel), int(mode), _ptr(pool),
                                 n_slots,
                               _ptr(_c(slot_idx, np.int32)), _ptr(_c(pi, np.int16)),
                               _ptr(_c(cs, np.float32)), _ptr(_c(q, np.float32)),
                               _ptr(_c(k, np.float32)), _ptr(_c(v, np.float32)),
                               _ptr(_c(alpha, np.float32)), _ptr(_c(beta, np.float32)),
                               _ptr(_c(o, np.float32)), lo, hi)
    return o, st


def replay_damp(pool, slot_idx, n_accept, pi, cs, khi, group, dk, dv, q, k, v, alpha, beta, o=None,
                per_channel=None, items=None, mode=0):
    _c(pool, np.uint8)
    n_slots, Hv, tb = pool.shape
    assert tb == damp_tile_bytes(dk, dv, khi, group)
    B, T_max, Hk, _ = q.shape
    if per_channel is None:
        per_channel = alpha.ndim == 4
    if o is None:
        o = np.zeros((B, T_max, Hv, dv), np.float32)
    lo, hi = items if items is not None else (0, B * Hv)
    st = lib().orc_replay_damp_m(B, T_max, Hk, Hv, dk, dv, khi, group, int(per_channel), int(mode),
                                 _ptr(pool),
                               n_slots, _ptr(_c(slot_idx, np.int32)), _ptr(_c(n_accept, np.int32)),
                               _ptr(_c(pi, np.int16)), _ptr(_c(cs, np.float32)), _ptr(_c(q, np.float32)),
                               _ptr(_c(k, np.float32)), _ptr(_c(v, np.float32)),
                               _ptr(_c(alpha, np.float32)), _ptr(_c(beta, np.float32)),
                               _ptr(_c(o, np.float32)), lo, hi)
    return o, st
