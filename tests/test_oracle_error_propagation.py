"""Pin of the oracle's mixed-precision decode against DAMP §3.3 (error
propagation under state quantization), CPU only.

DAMP Eq. 7 models the stored state as S^q_t = Q(A_t S^q_{t-1} + beta_t k_t
v_t^T) with A_t = (I - beta_t k_t k_t^T) Lambda_t (§3.1 Eq. 2); Eq. 8-9
define the accumulated error dS_t = S^q_t - S_t against the unquantised
recurrence and the local error R_t = S^q_t - (A_t S^q_{t-1} + beta k v^T);
Eq. 12 gives dS_t = A_t dS_{t-1} + R_t and Eq. 13 its unrolled form with
dS_0 = 0.  Here S^q_t is the oracle's mixed pool after t decode steps
(dequantised, logical rows), S_t the FP64 recurrence from the same start,
and the checks are: Eq. 12 and Eq. 13 hold to 1e-12; every local error is
the quantiser's (an INT8 row within half its scale step, an FP16 row within
half an FP16 ulp, plus the FP32 rounding of the update); and the
accumulated error is not just the last local one (the propagation term is
exercised), in both requantisation modes.
"""
import numpy as np
import pytest

import oracle as orc
from recurrent_state_gb300 import inputs as gen


def a_matrix(k, a, beta):
    return (np.eye(k.size) - beta * np.outer(k, k)) @ np.diag(a)


@pytest.mark.parametrize("mode", [0, 1])
def test_error_recursion_eq12_eq13(mode):
    B, Hk, Hv, d, khi, T = 2, 1, 2, 16, 4, 12
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=d, steps=T, per_channel=True, in_dtype="f32",
                            seed=90 + mode, horizon=(2.0, 64.0))
    hi = gen.hi_rows(Hv, d, khi, seed=90)
    pi = orc.row_map(hi, d)
    pool = orc.convert_pool_f32_to_mixed(w.state0, khi, pi, mode=mode)

    def logical():
        return orc.convert_pool_mixed_to_f32(pool, d, d, khi, pi).astype(np.float64)

    Sq_prev = logical()
    S = Sq_prev.copy()                      # the unquantised recurrence starts from S^q_0: dS_0 = 0
    dS_prev = np.zeros_like(S)
    R_hist, A_hist = [], []
    propagated = 0.0
    for t in range(T):
        _, st = orc.decode_mixed(pool, w.slot_idx, pi, khi, d, d, w.q[t], w.k[t], w.v[t], w.alpha[t],
                                 w.beta[t], mode=mode)
        assert st == 0
        Sq = logical()
        R_t = np.zeros_like(S)
        A_t = np.zeros(S.shape[:2] + (d, d))
        for b in range(B):
            s = w.slot_idx[b]
            for h in range(Hv):
                g = h // (Hv // Hk)
                k = w.k[t, b, g].astype(np.float64)
                bt = np.float64(w.beta[t, b, h])
                A = a_matrix(k, w.alpha[t, b, h].astype(np.float64), bt)
                A_t[s, h] = A
                write = bt * np.outer(k, w.v[t, b, h].astype(np.float64))
                S[s, h] = A @ S[s, h] + write
                R_t[s, h] = Sq[s, h] - (A @ Sq_prev[s, h] + write)
                # the local error is the quantiser's, row by row (physical row r = channel pi[r])
                for r in range(d):
                    c = pi[h, r]
                    x = A[c] @ Sq_prev[s, h] + write[c]
                    err = np.max(np.abs(R_t[s, h, c]))
                    slop = 4e-6 * max(1.0, np.max(np.abs(x)))
                    if r < khi:
                        bound = np.max(np.spacing(np.abs(x).astype(np.float16)).astype(np.float64)) / 2
                    else:
                        bound = np.max(np.abs(x)) / 127.0 * 0.5 * (1 + 1e-4)
                    assert err <= bound + slop, (t, b, h, r)
        dS = Sq - S
        # Eq. 12
        for s in w.slot_idx:
            for h in range(Hv):
                rhs = A_t[s, h] @ dS_prev[s, h] + R_t[s, h]
                scale = max(1e-30, np.max(np.abs(dS[s, h])))
                assert np.max(np.abs(dS[s, h] - rhs)) <= 1e-12 * max(1.0, np.max(np.abs(S[s, h]))), t
                propagated = max(propagated, np.max(np.abs(dS[s, h] - R_t[s, h])) / scale)
        R_hist.append(R_t)
        A_hist.append(A_t)
        dS_prev, Sq_prev = dS, Sq
    # Eq. 13: dS_T = R_T + sum_i (A_T ... A_{i+1}) R_i
    for s in w.slot_idx:
        for h in range(Hv):
            acc = R_hist[-1][s, h].copy()
            for i in range(T - 1):
                P = np.eye(d)
                for j in range(T - 1, i, -1):
                    P = P @ A_hist[j][s, h]
                acc += P @ R_hist[i][s, h]
            assert np.max(np.abs(dS_prev[s, h] - acc)) <= 1e-12 * max(1.0, np.max(np.abs(S[s, h])))
    # errors of earlier steps are carried, not only the last step's
    assert propagated > 1e-3
