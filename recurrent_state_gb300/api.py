"""torch-facing wrappers over the C ABI (argument marshalling only).

Each function takes torch CUDA tensors, checks that they are contiguous and
on the current device, and passes raw pointers, sizes and the current CUDA
stream to the library.  Semantics, layouts and citations are documented in
``include/recurrent_state.h``.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _abi
from ._abi import check

_DT = {torch.float32: _abi.RS_F32, torch.bfloat16: _abi.RS_BF16, torch.float16: _abi.RS_F16}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t, name, dtype=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


class Layout:
    """A state-pool layout (``rs_layout``)."""

    def __init__(self, kind: str, dk: int, num_v_heads: int, num_qk_heads: int,
                 k_hi: int = 0, hi_rows=None, dv: int | None = None, group: int = 32,
                 value_scales=None, quant: str = "ieee"):
        """kind: "fp32", "mixed" (one INT8 scale per row) or "damp" (DAMP-exact:
        INT8 groups of ``group`` values along dv and value-scaling factors
        ``value_scales`` [Hv][dv], default all ones).  quant: the requantisation
        arithmetic of a mixed layout, "ieee" (RS_QUANT_IEEE) or "fused"
        (RS_QUANT_FUSED)."""
        self.kind = {"fp32": _abi.RS_LAYOUT_FP32, "mixed": _abi.RS_LAYOUT_MIXED_FP16_INT8,
                     "damp": _abi.RS_LAYOUT_MIXED_FP16_INT8}[kind]
        self.kind_name = kind
        self.dk, self.dv = dk, dv or dk
        self.Hv, self.Hk, self.k_hi = num_v_heads, num_qk_heads, k_hi
        p = _abi.LayoutParams(self.kind, dk, self.dv, num_v_heads, num_qk_heads, k_hi)
        hr = None
        if hi_rows is not None:
            hr = np.ascontiguousarray(hi_rows, np.int16)
        h = ctypes.c_void_p()
        if kind == "damp":
            cs = None
            if value_scales is not None:
                cs = np.ascontiguousarray(value_scales, np.float32)
                if cs.shape != (num_v_heads, self.dv):
                    raise ValueError("value_scales must be [Hv][dv]")
            self.value_scales = cs
            check(_abi.lib().rs_layout_create_damp(ctypes.byref(h), ctypes.byref(p),
                                                   None if hr is None else hr.ctypes.data, group,
                                                   None if cs is None else cs.ctypes.data),
                  "rs_layout_create_damp")
        else:
            check(_abi.lib().rs_layout_create(ctypes.byref(h), ctypes.byref(p),
                                              None if hr is None else hr.ctypes.data), "rs_layout_create")
        self._h = h
        self.quant = quant
        check(_abi.lib().rs_layout_set_quant(h, {"ieee": _abi.RS_QUANT_IEEE,
                                                  "fused": _abi.RS_QUANT_FUSED}[quant]),
              "rs_layout_set_quant")
        nb = ctypes.c_size_t()
        check(_abi.lib().rs_layout_head_bytes(h, ctypes.byref(nb)))
        self.head_bytes = int(nb.value)

    @property
    def handle(self):
        return self._h

    def row_map(self) -> np.ndarray:
        pi = np.zeros((self.Hv, self.dk), np.int16)
        check(_abi.lib().rs_layout_row_map(self._h, pi.ctypes.data))
        return pi

    def bits_per_value(self) -> float:
        b = ctypes.c_double()
        check(_abi.lib().rs_layout_bits_per_value(self._h, ctypes.byref(b)))
        return b.value

    def empty_pool(self, n_slots: int, device="cuda") -> torch.Tensor:
        """Uninitialised pool [n_slots][Hv][dk][dv] float32 or [n_slots][Hv][head_bytes] uint8."""
        if self.kind == _abi.RS_LAYOUT_FP32:
            return torch.empty((n_slots, self.Hv, self.dk, self.dv), dtype=torch.float32, device=device)
        return torch.empty((n_slots, self.Hv, self.head_bytes), dtype=torch.uint8, device=device)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            try:
                _abi.lib().rs_layout_destroy(h)
            except Exception:
                pass
            self._h = None


def _pool_slots(layout, pool):
    _dev(pool, "pool")
    nbytes = pool.numel() * pool.element_size()
    per_slot = layout.Hv * layout.head_bytes
    if nbytes % per_slot:
        raise ValueError("pool size is not a whole number of slots")
    return nbytes // per_slot


def _step(fn, layout, pool, slot_idx, q, k, v, alpha, beta, o, status, stream):
    n_slots = _pool_slots(layout, pool)
    _dev(slot_idx, "slot_idx", torch.int32)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _dev(t, name)
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in _DT:
        raise ValueError("q, k, v must share one of float32/bfloat16/float16")
    _dev(alpha, "alpha", torch.float32)
    _dev(beta, "beta", torch.float32)
    _dev(o, "o")
    _dev(status, "status", torch.int32)
    B = slot_idx.numel()
    out_dt = _DT[o.dtype] if o is not None else _abi.RS_F32
    check(fn(layout.handle, _ptr(pool), n_slots, _ptr(slot_idx), B, _ptr(q), _ptr(k), _ptr(v),
             _DT[q.dtype], _ptr(alpha), _ptr(beta), _ptr(o), out_dt, _ptr(status),
             _stream(stream)), fn.__name__)


def gdn_decode_update(layout, pool, slot_idx, q, k, v, alpha, beta, o=None, status=None,
                      stream=None):
    """GDN decode step in place on ``pool``; writes ``o`` [B][Hv][dv] if given."""
    _step(_abi.lib().rs_gdn_decode_update, layout, pool, slot_idx, q, k, v, alpha, beta, o,
          status, stream)
    return o


def kda_decode_update(layout, pool, slot_idx, q, k, v, alpha, beta, o=None, status=None,
                      stream=None):
    """KDA decode step (alpha [B][Hv][dk]) in place on ``pool``."""
    _step(_abi.lib().rs_kda_decode_update, layout, pool, slot_idx, q, k, v, alpha, beta, o,
          status, stream)
    return o


def spec_replay_update(layout, per_channel_decay, pool, slot_idx, n_accept, q, k, v, alpha, beta,
                       o=None, status=None, stream=None):
    """Replay the first n_accept[b] of T_max logged tokens (inputs [B][T_max][...])."""
    n_slots = _pool_slots(layout, pool)
    _dev(slot_idx, "slot_idx", torch.int32)
    _dev(n_accept, "n_accept", torch.int32)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _dev(t, name)
    _dev(alpha, "alpha", torch.float32)
    _dev(beta, "beta", torch.float32)
    _dev(o, "o")
    _dev(status, "status", torch.int32)
    B, T_max = q.shape[0], q.shape[1]
    out_dt = _DT[o.dtype] if o is not None else _abi.RS_F32
    check(_abi.lib().rs_spec_replay_update(
        layout.handle, int(bool(per_channel_decay)), _ptr(pool), n_slots, _ptr(slot_idx), B, T_max,
        _ptr(n_accept), _ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], _ptr(alpha), _ptr(beta), _ptr(o),
        out_dt, _ptr(status), _stream(stream)), "rs_spec_replay_update")
    return o


def prefill_update(layout, per_channel_decay, pool, slot_idx, q, k, v, alpha, beta, n_tokens=None,
                   o=None, status=None, stream=None, chunked=False):
    """Apply a prefill chunk of L tokens (inputs [B][L][...]) to each sequence's
    state, read and written once; ``n_tokens`` [B] int32 limits each sequence
    to its first n_tokens[b] tokens (default: all L).  ``chunked``: the
    chunk-parallel form on the tensor cores (rs_prefill_chunked_update; FP32
    layout and the mixed ones with 16 FP16 rows; equal to the recurrence up
    to rounding)."""
    n_slots = _pool_slots(layout, pool)
    _dev(slot_idx, "slot_idx", torch.int32)
    _dev(n_tokens, "n_tokens", torch.int32)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _dev(t, name)
    _dev(alpha, "alpha", torch.float32)
    _dev(beta, "beta", torch.float32)
    _dev(o, "o")
    _dev(status, "status", torch.int32)
    B, L = q.shape[0], q.shape[1]
    out_dt = _DT[o.dtype] if o is not None else _abi.RS_F32
    fn = "rs_prefill_chunked_update" if chunked else "rs_prefill_update"
    check(getattr(_abi.lib(), fn)(
        layout.handle, int(bool(per_channel_decay)), _ptr(pool), n_slots, _ptr(slot_idx), B, L,
        _ptr(n_tokens), _ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], _ptr(alpha), _ptr(beta), _ptr(o),
        out_dt, _ptr(status), _stream(stream)), fn)
    return o


def state_convert(src_layout, src_pool, dst_layout, dst_pool, slots, status=None, stream=None):
    """Convert the listed slots between two layouts of the same shape."""
    n_slots = _pool_slots(src_layout, src_pool)
    if _pool_slots(dst_layout, dst_pool) != n_slots:
        raise ValueError("source and destination pools hold different slot counts")
    _dev(slots, "slots", torch.int32)
    _dev(status, "status", torch.int32)
    check(_abi.lib().rs_state_convert(src_layout.handle, _ptr(src_pool), dst_layout.handle,
                                      _ptr(dst_pool), n_slots, _ptr(slots), slots.numel(),
                                      _ptr(status), _stream(stream)), "rs_state_convert")


class Plan:
    """A dasc selection plan (``rs_plan``): head or key-channel units of an
    FP32 layout, or head units of a mixed layout."""

    def __init__(self, layout: Layout, keep: np.ndarray, unit: str):
        keep = np.ascontiguousarray(keep, np.uint8)
        self.unit = {"head": _abi.RS_UNIT_HEAD, "channel": _abi.RS_UNIT_CHANNEL}[unit]
        self.num_layers = keep.shape[0]
        self.layout = layout
        h = ctypes.c_void_p()
        check(_abi.lib().rs_plan_create(ctypes.byref(h), layout.handle, self.num_layers, self.unit,
                                        keep.ctypes.data), "rs_plan_create")
        self._h = h
        off = np.zeros(self.num_layers + 1, np.int64)
        ub = ctypes.c_int64()
        check(_abi.lib().rs_plan_offsets(h, off.ctypes.data, ctypes.byref(ub)))
        self.offsets = off
        self.unit_bytes = int(ub.value)
        self.ckpt_slot_bytes = int(off[-1]) * self.unit_bytes
        self._uploaded = False
        self.int8_codes_bytes = self.int8_slot_bytes = None
        if layout.kind == _abi.RS_LAYOUT_FP32:
            cb, sb = ctypes.c_int64(), ctypes.c_int64()
            check(_abi.lib().rs_ckpt_int8_bytes(h, ctypes.byref(cb), ctypes.byref(sb)), "rs_ckpt_int8_bytes")
            self.int8_codes_bytes, self.int8_slot_bytes = int(cb.value), int(sb.value)

    def upload(self):
        check(_abi.lib().rs_plan_upload(self._h), "rs_plan_upload")
        self._uploaded = True
        return self

    def empty_ckpt_pool(self, n_ckpt_slots: int, device="cuda") -> torch.Tensor:
        return torch.empty((n_ckpt_slots, self.ckpt_slot_bytes), dtype=torch.uint8, device=device)

    def empty_int8_ckpt_pool(self, n_ckpt_slots: int, device="cuda") -> torch.Tensor:
        """INT8 checkpoint slots: codes [o_L][rows][dv] int8, then scales f32."""
        return torch.empty((n_ckpt_slots, self.int8_slot_bytes), dtype=torch.uint8, device=device)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            try:
                _abi.lib().rs_plan_destroy(h)
            except Exception:
                pass
            self._h = None


def _layer_pool(pool, layout):
    """pool: [L][n_slots][Hv][...] (contiguous) -> (n_pool_slots, layer_stride_bytes)."""
    _dev(pool, "pool")
    L = pool.shape[0]
    layer_bytes = pool.numel() * pool.element_size() // L
    per_slot = layout.Hv * layout.head_bytes
    return layer_bytes // per_slot, layer_bytes


def ckpt_pack(plan: Plan, pool, src_slots, dst_ckpt_slots, ckpt_pool, status=None, stream=None):
    n_pool, stride = _layer_pool(pool, plan.layout)
    _dev(src_slots, "src_slots", torch.int32)
    _dev(dst_ckpt_slots, "dst_ckpt_slots", torch.int32)
    _dev(ckpt_pool, "ckpt_pool")
    _dev(status, "status", torch.int32)
    check(_abi.lib().rs_ckpt_pack(plan._h, _ptr(pool), stride, n_pool, _ptr(src_slots),
                                  _ptr(dst_ckpt_slots), src_slots.numel(), _ptr(ckpt_pool),
                                  ckpt_pool.shape[0], _ptr(status), _stream(stream)), "rs_ckpt_pack")


def ckpt_restore(plan: Plan, ckpt_pool, src_ckpt_slots, pool, dst_slots, status=None, stream=None):
    n_pool, stride = _layer_pool(pool, plan.layout)
    _dev(src_ckpt_slots, "src_ckpt_slots", torch.int32)
    _dev(dst_slots, "dst_slots", torch.int32)
    _dev(ckpt_pool, "ckpt_pool")
    _dev(status, "status", torch.int32)
    check(_abi.lib().rs_ckpt_restore(plan._h, _ptr(ckpt_pool), ckpt_pool.shape[0],
                                     _ptr(src_ckpt_slots), _ptr(pool), stride, n_pool,
                                     _ptr(dst_slots), dst_slots.numel(), _ptr(status),
                                     _stream(stream)), "rs_ckpt_restore")


def ckpt_pack_int8(plan: Plan, pool, src_slots, dst_ckpt_slots, ckpt_pool, status=None, stream=None):
    """dasc INT8 checkpoint: quantise the retained rows of FP32 pool slots."""
    n_pool, stride = _layer_pool(pool, plan.layout)
    _dev(src_slots, "src_slots", torch.int32)
    _dev(dst_ckpt_slots, "dst_ckpt_slots", torch.int32)
    _dev(ckpt_pool, "ckpt_pool")
    _dev(status, "status", torch.int32)
    check(_abi.lib().rs_ckpt_pack_int8(plan._h, _ptr(pool), stride, n_pool, _ptr(src_slots),
                                       _ptr(dst_ckpt_slots), src_slots.numel(), _ptr(ckpt_pool),
                                       ckpt_pool.shape[0], _ptr(status), _stream(stream)),
          "rs_ckpt_pack_int8")


def ckpt_restore_int8(plan: Plan, ckpt_pool, src_ckpt_slots, pool, dst_slots, status=None, stream=None):
    """dasc INT8 checkpoint reuse: dequantise into FP32 pool slots, omitted rows zero."""
    n_pool, stride = _layer_pool(pool, plan.layout)
    _dev(src_ckpt_slots, "src_ckpt_slots", torch.int32)
    _dev(dst_slots, "dst_slots", torch.int32)
    _dev(ckpt_pool, "ckpt_pool")
    _dev(status, "status", torch.int32)
    check(_abi.lib().rs_ckpt_restore_int8(plan._h, _ptr(ckpt_pool), ckpt_pool.shape[0],
                                          _ptr(src_ckpt_slots), _ptr(pool), stride, n_pool,
                                          _ptr(dst_slots), dst_slots.numel(), _ptr(status),
                                          _stream(stream)), "rs_ckpt_restore_int8")
