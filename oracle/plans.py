"""Selection-plan builders of the pages, written out plainly (fp64 numpy).

TEST INFRASTRUCTURE ONLY: only tests/, the smoke check and the benchmark's
CPU-baseline leg use this module; the library's host code computes the same
plans on its own.

dasc ("dasc: Decay-Aware State Compression for Hybrid Linear-Attention
Serving"):
  * §3.3 Eq. 2, static log-decay of unit u with the representative gate input
    a_s:  standard gate  g = -exp(A_log) * softplus(a_s + d);
          Kimi-K3 gate   g = l * sigmoid(exp(A_log) * (a_s + d)), l = -5;
  * §3.3 Eq. 3, static retention horizon H_s = ln(eps) / g, eps = 1e-3;
  * §4.1, retention mask: a unit is retained when H_s(u) > W_max;
  * §4.2 Eq. 7, suffix-refresh window: W_u = clamp(next_pow2(H_s(u)), 4, W_max)
    with next_pow2(x) = 2^ceil(log2 x) for x > 0 and 4 for x = 0;
    W_replay = min(n_p, max over omitted units of W_u), 0 if none is omitted.
DAMP ("DAMP: Decay-Aware Mixed-Precision Recurrent-State Quantization"):
  * §5.1 Eq. 14, local error of key channel u: e_u = ||[Q(S) - S]_u||^2 with Q
    the storage quantiser (one INT8 scale per row, the oracle's quantiser);
  * §5.1 Eq. 15, accumulated-error risk over calibration anchors:
    C_u = mean over anchors of e_u * (1 + sum_{j=1..H} prod_{r=1..j} a_{r,u}^2);
  * §5.1 budgeted selection: the K_hi channels with the largest C_u per head.

Readings fixed here (the pages leave them open): planning arithmetic in fp64
from FP32 inputs; softplus(x) = log(1 + exp(x)); e_u sums the squared
differences of the FP32 dequantised and original values in fp64; equal risk
scores rank the lower channel index first; the selected channels are returned
in ascending order.
"""
import math

import numpy as np

from . import quantise_row, dequantise_row

EPSILON = 1e-3
K3_FLOOR = -5.0


def softplus(x):
    return math.log1p(math.exp(x)) if x < 30 else x + math.log1p(math.exp(-x))


def sigmoid(x):
    return 1.0 / (1.0 + math.exp(-x))


def static_log_decay(gate, A_log, d, a_s):
    """dasc §3.3 Eq. 2 for one unit (gate 'std' or 'k3')."""
    if gate == "std":
        return -math.exp(float(A_log)) * softplus(a_s + float(d))
    return K3_FLOOR * sigmoid(math.exp(float(A_log)) * (a_s + float(d)))


def static_horizons(gate, A_log, d, a_s, eps=EPSILON):
    """dasc §3.3 Eq. 3, H_s = ln(eps) / g_s, for arrays of units."""
    A_log = np.asarray(A_log, np.float32).reshape(-1)
    d = np.asarray(d, np.float32).reshape(-1)
    out = np.empty(A_log.size, np.float64)
    for i in range(A_log.size):
        out[i] = math.log(eps) / static_log_decay(gate, A_log[i], d[i], a_s)
    return out


def retention_mask(H, W_max):
    """dasc §4.1: retained iff H_s > W_max."""
    return np.array([1 if h > W_max else 0 for h in np.asarray(H).reshape(-1)], np.uint8)


def next_pow2(x):
    if x == 0:
        return 4
    p = 1
    while p < x:
        p *= 2
    return p


def replay_window(H, keep, W_max, n_prefix):
    """dasc §4.2 Eq. 7."""
    widths = [min(max(next_pow2(h), 4), W_max) for h, k in zip(np.asarray(H).reshape(-1),
                                                                 np.asarray(keep).reshape(-1)) if not k]
    if not widths:
        return 0
    return min(n_prefix, max(widths))


def local_errors(S):
    """DAMP §5.1 Eq. 14 for one state [dk][dv] (FP32): e_u per key channel."""
    S = np.asarray(S, np.float32)
    e = np.zeros(S.shape[0], np.float64)
    for u in range(S.shape[0]):
        codes, s = quantise_row(S[u])
        back = dequantise_row(codes, s)
        e[u] = sum((float(b) - float(x)) ** 2 for b, x in zip(back, S[u]))
    return e


def risk_scores(states, decays):
    """DAMP §5.1 Eq. 15.  states [N][dk][dv] (anchors); decays [N][H][dk], the
    decay factors a_{t+r,u} of the H updates after each anchor."""
    states = np.asarray(states, np.float32)
    decays = np.asarray(decays, np.float32)
    N, dk, _ = states.shape
    C = np.zeros(dk, np.float64)
    for n in range(N):
        e = local_errors(states[n])
        for u in range(dk):
            w, prod = 1.0, 1.0
            for j in range(decays.shape[1]):
                prod *= float(decays[n, j, u]) ** 2
                w += prod
            C[u] += e[u] * w
    return C / N


def select_high_precision(C, k_hi):
    """DAMP §5.1: the k_hi channels with the largest scores (ties: lower
    index first), in ascending channel order."""
    C = np.asarray(C, np.float64)
    order = sorted(range(C.size), key=lambda u: (-C[u], u))
    return np.array(sorted(order[:k_hi]), np.int16)
