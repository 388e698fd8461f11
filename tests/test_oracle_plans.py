"""Pins for the oracle's selection-plan builders (CPU only).

dasc §3.3 Eq. 2-3 (static horizons), §4.1 (mask H_s > W_max), §4.2 Eq. 7
(suffix-refresh window); DAMP §5.1 Eq. 14-15 (local error, accumulated-error
risk) and the budgeted top-K_hi selection.  Pins: closed forms at special
gate inputs, the identity exp(g H_s) = eps, the softplus of a library routine
(numpy logaddexp), hand-worked windows, exactly representable rows (zero
error) and half-way rows (known error), the geometric-series closed form of
the decay weight, and hand-worked top-K with ties.
"""
import math

import numpy as np
import pytest

from oracle import plans
from recurrent_state_gb300 import inputs as gen


def test_horizon_closed_forms():
    # standard gate at A_log = 0, a_s + d = 0: g = -ln 2, H = log2(1000)
    H = plans.static_horizons("std", [0.0], [0.3], -0.3)
    assert abs(H[0] - math.log2(1000.0)) < 1e-6
    # Kimi-K3 safe gate at the same point: g = -5 * 1/2, H = ln(1000) / 2.5
    H = plans.static_horizons("k3", [0.0], [-0.8], 0.8)
    assert abs(H[0] - math.log(1000.0) / 2.5) < 1e-6   # d is FP32: a_s + d = 0 up to 1e-8
    # the K3 gate is bounded by l = -5: H >= ln(1000)/5 for every input
    H = plans.static_horizons("k3", np.full(5, 3.0, np.float32), np.linspace(-2, 9, 5), 0.8)
    assert np.all(H >= math.log(1000.0) / 5 - 1e-12)


def test_horizon_identity_and_library_softplus():
    g = gen.rng(1)
    A = g.uniform(-3, 2, 64).astype(np.float32)
    d = g.uniform(-6, 6, 64).astype(np.float32)
    for gate, a_s in (("std", -0.3), ("k3", 0.8)):
        H = plans.static_horizons(gate, A, d, a_s)
        gs = np.array([plans.static_log_decay(gate, A[i], d[i], a_s) for i in range(64)])
        assert np.all(gs < 0) and np.all(H > 0)
        assert np.allclose(np.exp(gs * H), 1e-3, rtol=1e-12)   # alpha_s^H = eps
    ref = -np.exp(A.astype(np.float64)) * np.logaddexp(0.0, -0.3 + d.astype(np.float64))
    got = np.array([plans.static_log_decay("std", A[i], d[i], -0.3) for i in range(64)])
    assert np.allclose(got, ref, rtol=1e-13)


def test_mask_is_strict():
    H = np.array([16.0, 16.000001, 15.9, 1e6, 0.5])
    assert plans.retention_mask(H, 16).tolist() == [0, 1, 0, 1, 0]


def test_replay_window_hand_worked():
    H = [5.0, 3.0, 100.0, 0.0]
    keep = [0, 0, 1, 0]
    assert plans.replay_window(H, keep, 64, 1000) == 8      # next_pow2(5) = 8 is the widest
    assert plans.replay_window(H, keep, 64, 6) == 6         # capped by the prefix
    assert plans.replay_window(H, [1, 1, 1, 1], 64, 1000) == 0  # nothing omitted
    assert plans.replay_window([40.0], [0], 48, 1000) == 48  # next_pow2 64 clamped to W_max
    assert plans.replay_window([0.0, 1.0], [0, 0], 64, 1000) == 4  # zero and small map to 4
    assert [plans.next_pow2(x) for x in (0, 1, 2, 3, 9.97, 16, 16.5)] == [4, 1, 2, 4, 16, 16, 32]


def test_local_error_exact_rows_and_half_way_rows():
    S = np.zeros((3, 8), np.float32)
    S[0] = [127, -5, 0, 3, 64, -127, 1, 2]          # integers, absmax 127: s = 1, exact
    S[1] = [127, 0.5, 1.5, -2.5, 0, 0, 0, 0]        # s = 1: halves round to even
    S[2] = 0.0                                      # zero row: exact
    e = plans.local_errors(S)
    assert e[0] == 0.0 and e[2] == 0.0
    assert e[1] == 3 * 0.25


def test_risk_score_closed_form():
    """Constant decay a over H steps: weight 1 + sum_j a^(2j) = (1 - a^(2H+2)) / (1 - a^2)."""
    S = np.zeros((2, 4, 8), np.float32)
    S[:, 1] = [127, 0.5, 0, 0, 0, 0, 0, 0]         # e = 0.25 in channel 1
    S[1, 3] = [127, 0.5, 1.5, 0, 0, 0, 0, 0]       # e = 0.5 in channel 3 of the second anchor
    Hn, a = 7, 0.9
    dec = np.full((2, Hn, 4), a, np.float32)
    C = plans.risk_scores(S, dec)
    af = float(np.float32(a))
    w = (1 - af ** (2 * Hn + 2)) / (1 - af ** 2)
    assert abs(C[1] - 0.25 * w) < 1e-12 and abs(C[3] - 0.5 * w / 2) < 1e-12
    assert C[0] == 0.0 and C[2] == 0.0
    # no decay after the anchor (a = 0): the weight is 1
    assert np.allclose(plans.risk_scores(S, np.zeros((2, 3, 4), np.float32)), [0, 0.25, 0, 0.25])


def test_topk_selection():
    C = np.array([0.1, 5.0, 3.0, 5.0, 0.0, 2.0])
    assert plans.select_high_precision(C, 2).tolist() == [1, 3]
    assert plans.select_high_precision(C, 3).tolist() == [1, 2, 3]
    assert plans.select_high_precision(np.zeros(6), 2).tolist() == [0, 1]   # ties: lower index
