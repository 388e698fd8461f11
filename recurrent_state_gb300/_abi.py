"""ctypes declarations of the C ABI in ``include/recurrent_state.h``.

Loads the in-tree ``_build/librecurrent_state.so``.  There is no fallback:
if the library has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

RS_OK = 0
RS_ERR_INVALID_ARG = -1
RS_ERR_UNSUPPORTED = -2
RS_ERR_MISALIGNED = -3
RS_ERR_CUDA = -4

RS_DEV_BAD_SLOT = 1
RS_DEV_BAD_ACCEPT = 2
RS_DEV_BAD_CKPT_SLOT = 4
RS_DEV_PIPE_TIMEOUT = 8

RS_LAYOUT_FP32 = 0
RS_LAYOUT_MIXED_FP16_INT8 = 1
RS_F32, RS_BF16, RS_F16 = 0, 1, 2
RS_UNIT_HEAD, RS_UNIT_CHANNEL = 0, 1
RS_GATE_STD, RS_GATE_K3 = 0, 1
RS_QUANT_IEEE, RS_QUANT_FUSED = 0, 1

# Every function the header declares, for the symbol-table test.
EXPORTS = (
    "rs_status_string", "rs_last_cuda_error", "rs_version",
    "rs_layout_create", "rs_layout_create_damp", "rs_layout_destroy", "rs_layout_head_bytes", "rs_layout_row_map",
    "rs_layout_bits_per_value", "rs_layout_set_quant", "rs_layout_quant",
    "rs_gdn_decode_update", "rs_kda_decode_update", "rs_spec_replay_update", "rs_prefill_update", "rs_prefill_chunked_update",
    "rs_state_convert",
    "rs_plan_create", "rs_plan_destroy", "rs_plan_offsets", "rs_plan_upload",
    "rs_ckpt_pack", "rs_ckpt_restore", "rs_ckpt_pack_noalloc",
    "rs_ckpt_int8_bytes", "rs_ckpt_pack_int8", "rs_ckpt_restore_int8",
    "rs_dasc_horizons", "rs_dasc_keep", "rs_dasc_refresh_window", "rs_damp_risk_scores",
    "rs_damp_select_hi_rows",
)


class RsError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(what)


class LayoutParams(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("num_v_heads", ctypes.c_int32), ("num_qk_heads", ctypes.c_int32),
                ("k_hi", ctypes.c_int32)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"the CUDA library {path} is not built; run "
                    "`python -m recurrent_state_gb300.build` (needs nvcc)")
            L = ctypes.CDLL(path)
            _declare(L)
            _lib = L
        return _lib


def _declare(L):
    L.rs_status_string.argtypes = [_I32]
    L.rs_status_string.restype = ctypes.c_char_p
    L.rs_last_cuda_error.argtypes = []
    L.rs_last_cuda_error.restype = ctypes.c_char_p
    L.rs_version.argtypes = []
    L.rs_version.restype = ctypes.c_char_p
    L.rs_layout_create.argtypes = [ctypes.POINTER(_P), ctypes.POINTER(LayoutParams), _P]
    L.rs_layout_destroy.argtypes = [_P]
    L.rs_layout_head_bytes.argtypes = [_P, ctypes.POINTER(ctypes.c_size_t)]
    L.rs_layout_row_map.argtypes = [_P, _P]
    L.rs_layout_bits_per_value.argtypes = [_P, ctypes.POINTER(ctypes.c_double)]
    L.rs_layout_set_quant.argtypes = [_P, _I32]
    L.rs_layout_quant.argtypes = [_P, ctypes.POINTER(_I32)]
    step = [_P, _P, _I64, _P, _I32, _P, _P, _P, _I32, _P, _P, _P, _I32, _P, _P]
    L.rs_gdn_decode_update.argtypes = step
    L.rs_kda_decode_update.argtypes = step
    L.rs_spec_replay_update.argtypes = [_P, _I32, _P, _I64, _P, _I32, _I32, _P, _P, _P, _P, _I32,
                                        _P, _P, _P, _I32, _P, _P]
    L.rs_prefill_update.argtypes = [_P, _I32, _P, _I64, _P, _I32, _I32, _P, _P, _P, _P, _I32,
                                    _P, _P, _P, _I32, _P, _P]
    L.rs_prefill_chunked_update.argtypes = L.rs_prefill_update.argtypes
    L.rs_state_convert.argtypes = [_P, _P, _P, _P, _I64, _P, _I32, _P, _P]
    L.rs_plan_create.argtypes = [ctypes.POINTER(_P), _P, _I32, _I32, _P]
    L.rs_plan_destroy.argtypes = [_P]
    L.rs_plan_offsets.argtypes = [_P, _P, ctypes.POINTER(_I64)]
    L.rs_plan_upload.argtypes = [_P]
    L.rs_ckpt_pack.argtypes = [_P, _P, _I64, _I64, _P, _P, _I32, _P, _I64, _P, _P]
    L.rs_ckpt_restore.argtypes = [_P, _P, _I64, _P, _P, _I64, _I64, _P, _I32, _P, _P]
    L.rs_ckpt_pack_noalloc.argtypes = [_P, _P, _I64, _I64, _P, _P, _I32, _P, _I64, _P, _P]
    L.rs_ckpt_int8_bytes.argtypes = [_P, _P, _P]
    L.rs_layout_create_damp.argtypes = [ctypes.POINTER(_P), ctypes.POINTER(LayoutParams), _P, _I32, _P]
    L.rs_ckpt_pack_int8.argtypes = [_P, _P, _I64, _I64, _P, _P, _I32, _P, _I64, _P, _P]
    L.rs_ckpt_restore_int8.argtypes = [_P, _P, _I64, _P, _P, _I64, _I64, _P, _I32, _P, _P]
    L.rs_dasc_horizons.argtypes = [_I32, _P, _P, _I64, ctypes.c_double, ctypes.c_double, _P]
    L.rs_dasc_keep.argtypes = [_P, _I64, ctypes.c_double, _P]
    L.rs_dasc_refresh_window.argtypes = [_P, _P, _I64, _I64, _I64, _P]
    L.rs_damp_risk_scores.argtypes = [_P, _P, _I32, _I32, _I32, _I32, _P]
    L.rs_damp_select_hi_rows.argtypes = [_P, _I32, _I32, _I32, _P]
    for name in EXPORTS:
        if name not in ("rs_status_string", "rs_last_cuda_error", "rs_version"):
            getattr(L, name).restype = _I32


def check(status: int, what: str = ""):
    if status == RS_OK:
        return
    L = lib()
    msg = L.rs_status_string(status).decode()
    if status == RS_ERR_CUDA:
        msg += ": " + L.rs_last_cuda_error().decode()
    raise RsError(status, f"{what}: {msg}" if what else msg)
