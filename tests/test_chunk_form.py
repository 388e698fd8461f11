"""The chunk-parallel form of the gated delta rule, stated in numpy (fp64) and
checked against the oracle's token-by-token recurrence (CPU only).

For a chunk of C tokens starting from state S0 (rows = key channels u,
columns = value dimensions v; DAMP §3.1 Eq. 1-2, with the decay diag(alpha)
applied before each write), with cumulative decays
    Gamma_t[c] = prod_{s<=t} alpha_s[c]
the written rows w_t = beta_t (v_t - (diag(alpha_t) S_{t-1})^T k_t) satisfy
    (I + diag(beta) A) W = diag(beta) (V - Khat S0),
    A[t][i] = sum_c k_t[c] k_i[c] prod_{s=i+1..t} alpha_s[c]   (i < t),
    Khat[t][c] = k_t[c] Gamma_t[c],
and then
    O = Qhat S0 + Bm W,      Bm[t][i] = sum_c q_t[c] k_i[c] prod_{s=i+1..t} alpha_s[c]  (i <= t),
    S_C = diag(Gamma_C) S0 + Ktil^T W,   Ktil[i][c] = k_i[c] prod_{s=i+1..C} alpha_s[c].
This is the form the chunked prefill kernel evaluates (the three products
against S0 and the two against W on the tensor cores); the test pins the
algebra, independently of any kernel, to the page's recurrence.
"""
import numpy as np
import pytest

import oracle as orc
from recurrent_state_gb300 import inputs as gen


def chunk_step(S0, q, k, v, alpha, beta):
    """One chunk in fp64.  S0 [dk][dv]; q, k [C][dk]; v [C][dv]; alpha [C][dk];
    beta [C].  Returns (S_C, O [C][dv])."""
    C, dk = k.shape
    gam = np.cumprod(alpha, axis=0)                       # Gamma_t
    dec = np.ones((C, C, dk))                             # prod_{s=i+1..t} alpha_s, t >= i
    for i in range(C):
        for t in range(i + 1, C):
            dec[t, i] = dec[t - 1, i] * alpha[t]
    A = np.zeros((C, C))
    Bm = np.zeros((C, C))
    for t in range(C):
        for i in range(C):
            if i < t:
                A[t, i] = np.sum(k[t] * k[i] * dec[t, i])
            if i <= t:
                Bm[t, i] = np.sum(q[t] * k[i] * dec[t, i])
    Khat = k * gam
    Qhat = q * gam
    rhs = beta[:, None] * (v - Khat @ S0)
    W = np.linalg.solve(np.eye(C) + beta[:, None] * A, rhs)
    O = Qhat @ S0 + Bm @ W
    tail = np.ones((C, dk))                               # prod_{s=i+1..C-1} alpha_s
    for i in range(C - 2, -1, -1):
        tail[i] = tail[i + 1] * alpha[i + 1]
    Ktil = k * tail
    S = gam[-1][:, None] * S0 + Ktil.T @ W
    return S, O


@pytest.mark.parametrize("per_channel,C", [(True, 16), (False, 16), (True, 7)])
def test_chunk_form_equals_the_recurrence(per_channel, C):
    d = 64
    w = gen.decode_workload(B=2, Hk=2, Hv=2, d=d, steps=C, per_channel=per_channel, in_dtype="f32",
                            seed=11, horizon=(2.0, 8192.0) if per_channel else (4.0, 4096.0))
    pool = w.state0.copy()
    T = C
    q, k, v, a, b = gen.replay_view(w, T)
    o = np.zeros((w.B, T, w.Hv, d), np.float32)
    orc.replay_f32(pool, w.slot_idx, np.full(w.B, T, np.int32), q, k, v, a, b, o=o)
    for bb in range(w.B):
        s = w.slot_idx[bb]
        for h in range(w.Hv):
            g_ = h // (w.Hv // w.Hk)
            alpha = a[bb, :, h].astype(np.float64)
            if alpha.ndim == 1:
                alpha = np.repeat(alpha[:, None], d, axis=1)
            S, O = chunk_step(w.state0[s, h].astype(np.float64), q[bb, :, g_].astype(np.float64),
                              k[bb, :, g_].astype(np.float64), v[bb, :, h].astype(np.float64), alpha,
                              b[bb, :, h].astype(np.float64))
            ref_S = pool[s, h].astype(np.float64)
            ref_O = o[bb, :, h].astype(np.float64)
            assert np.max(np.abs(S - ref_S)) <= 2e-6 * np.max(np.abs(ref_S))
            assert np.max(np.abs(O - ref_O)) <= 2e-6 * np.max(np.abs(ref_O))
