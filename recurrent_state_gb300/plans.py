"""Host selection-plan builders of the C ABI (numpy in, numpy out).

dasc §3.3 Eq. 2-3 static retention horizons, §4.1 retention masks, §4.2
Eq. 7 suffix-refresh windows; DAMP §5.1 Eq. 14-15 accumulated-error risk and
the budgeted FP16 channel selection.  Argument marshalling only: the
arithmetic runs in the library (rs_dasc_*, rs_damp_*).
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _abi
from ._abi import check

GATES = {"std": _abi.RS_GATE_STD, "k3": _abi.RS_GATE_K3}


def _p(a):
    return a.ctypes.data if a.size else None


def dasc_horizons(gate: str, A_log, d_bias, a_s: float, epsilon: float = 1e-3) -> np.ndarray:
    """H_s per unit (float64) from the gate's A_log and decay bias (float32)."""
    A = np.ascontiguousarray(A_log, np.float32).reshape(-1)
    d = np.ascontiguousarray(d_bias, np.float32).reshape(-1)
    if A.size != d.size:
        raise ValueError("A_log and d_bias differ in size")
    H = np.empty(A.size, np.float64)
    check(_abi.lib().rs_dasc_horizons(GATES[gate], _p(A), _p(d), A.size, float(a_s), float(epsilon), _p(H)),
          "rs_dasc_horizons")
    return H


def dasc_keep(H, W_max: float) -> np.ndarray:
    """Retention mask (uint8): H_s > W_max."""
    H = np.ascontiguousarray(H, np.float64).reshape(-1)
    keep = np.empty(H.size, np.uint8)
    check(_abi.lib().rs_dasc_keep(_p(H), H.size, float(W_max), _p(keep)), "rs_dasc_keep")
    return keep


def dasc_refresh_window(H, keep, W_max: int, n_prefix: int) -> int:
    H = np.ascontiguousarray(H, np.float64).reshape(-1)
    keep = np.ascontiguousarray(keep, np.uint8).reshape(-1)
    if H.size != keep.size:
        raise ValueError("H and keep differ in size")
    out = ctypes.c_int64()
    check(_abi.lib().rs_dasc_refresh_window(_p(H), _p(keep), H.size, int(W_max), int(n_prefix),
                                            ctypes.byref(out)), "rs_dasc_refresh_window")
    return int(out.value)


def damp_risk_scores(states, decays) -> np.ndarray:
    """C_u per key channel of one head: states [N][dk][dv], decays [N][H][dk]."""
    S = np.ascontiguousarray(states, np.float32)
    A = np.ascontiguousarray(decays, np.float32)
    N, dk, dv = S.shape
    if A.shape[0] != N or A.shape[2] != dk:
        raise ValueError("decays must be [n_anchors][horizon][dk]")
    C = np.empty(dk, np.float64)
    check(_abi.lib().rs_damp_risk_scores(_p(S), _p(A), N, dk, dv, A.shape[1], _p(C)), "rs_damp_risk_scores")
    return C


def damp_select_hi_rows(C, k_hi: int) -> np.ndarray:
    """Top-k_hi channels per head (int16, ascending) from scores [n_heads][dk]."""
    C = np.ascontiguousarray(C, np.float64)
    if C.ndim == 1:
        C = C[None]
    out = np.empty((C.shape[0], k_hi), np.int16)
    check(_abi.lib().rs_damp_select_hi_rows(_p(C), C.shape[0], C.shape[1], int(k_hi), _p(out)),
          "rs_damp_select_hi_rows")
    return out
