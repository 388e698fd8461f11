"""Pins for the oracle's mixed-precision decode and replay (CPU only).

DAMP Appendix A.4: one fused pass loads the packed state, dequantises it,
applies the update and readout in FP32 and requantises.  DAMP Appendix A.3
Eq. 17-18: the stored state is T = P_K S and the update runs on it with
permuted inputs k' = P_K k, q' = P_K q, Lambda' = P_K Lambda P_K^T (value
scaling and value reordering are not applied here).  DAMP §3.3 Eq. 9: the
local quantisation error R_t = S^q_t - (A_t S^q_{t-1} + b k v^T) is what one
write adds; for a symmetric INT8 row it is at most half a scale step.

The pins evaluate the exact FP64 update in logical coordinates (DAMP §3.1
Eq. 2, unpermuted) from the dequantised input and bound the oracle's
requantised output against it, row by row.
"""
import numpy as np
import pytest

import oracle as orc
from recurrent_state_gb300 import inputs as gen


def damp_eq2_step(S, q, k, v, a, beta):
    dk = k.size
    A = (np.eye(dk) - beta * np.outer(k, k)) @ np.diag(a)
    S = A @ S + beta * np.outer(k, v)
    return S, S.T @ q


def make(seed, per_channel, B=3, Hk=2, Hv=4, d=32, khi=4, steps=6):
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=d, steps=steps, per_channel=per_channel,
                            in_dtype="bf16", seed=seed, horizon=(2.0, 8192.0))
    hi = gen.hi_rows(Hv, d, khi, seed=seed)
    pi = orc.row_map(hi, d)
    pool = orc.convert_pool_f32_to_mixed(w.state0, khi, pi)
    return w, pi, pool


def logical(pool, d, khi, pi):
    return orc.convert_pool_mixed_to_f32(pool, d, d, khi, pi).astype(np.float64)


@pytest.mark.parametrize("per_channel", [False, True])
def test_mixed_step_within_local_quantisation_error(per_channel):
    d, khi = 32, 4
    w, pi, pool = make(21, per_channel, d=d, khi=khi)
    for t in range(w.steps):
        S_in = logical(pool, d, khi, pi)           # dequantised, logical rows
        o, st = orc.decode_mixed(pool, w.slot_idx, pi, khi, d, d, w.q[t], w.k[t], w.v[t],
                                 w.alpha[t], w.beta[t])
        assert st == 0
        S_out = logical(pool, d, khi, pi)
        for b in range(w.B):
            s = w.slot_idx[b]
            for h in range(w.Hv):
                g_ = h // (w.Hv // w.Hk)
                a = (w.alpha[t, b, h] if per_channel else np.full(d, w.alpha[t, b, h]))
                S_ref, o_ref = damp_eq2_step(S_in[s, h], w.q[t, b, g_].astype(np.float64),
                                             w.k[t, b, g_].astype(np.float64),
                                             w.v[t, b, h].astype(np.float64),
                                             np.asarray(a, np.float64), np.float64(w.beta[t, b, h]))
                # readout is taken from the FP32 updated state (before requantisation)
                assert np.max(np.abs(o[b, h] - o_ref)) <= 2e-5 * max(1.0, np.max(np.abs(o_ref)))
                for r in range(d):
                    c = pi[h, r]
                    row_ref = S_ref[c]
                    err = np.max(np.abs(S_out[s, h, c] - row_ref))
                    slop = 4e-6 * max(1.0, np.max(np.abs(row_ref)))
                    if r < khi:   # FP16 row: half an FP16 ulp
                        half_ulp = np.max(np.spacing(np.abs(row_ref).astype(np.float16))
                                          .astype(np.float64)) / 2
                        assert err <= half_ulp + slop, (t, b, h, r)
                    else:         # INT8 row: half a scale step
                        sc = np.max(np.abs(row_ref)) / 127.0
                        assert err <= sc * 0.5 * (1 + 1e-4) + slop, (t, b, h, r, err, sc)


def test_mixed_replay_one_equals_decode():
    d, khi = 32, 4
    w, pi, pool = make(22, True, d=d, khi=khi)
    q, k, v, a, b = gen.replay_view(w, 1)
    p1 = pool.copy()
    o1, _ = orc.decode_mixed(p1, w.slot_idx, pi, khi, d, d, w.q[0], w.k[0], w.v[0],
                             w.alpha[0], w.beta[0])
    p2 = pool.copy()
    o2, st = orc.replay_mixed(p2, w.slot_idx, np.ones(w.B, np.int32), pi, khi, d, d,
                              q, k, v, a, b)
    assert st == 0
    assert np.array_equal(p1, p2)
    assert np.array_equal(o1.view(np.uint32), o2[:, 0].view(np.uint32))


@pytest.mark.parametrize("per_channel", [False, True])
def test_mixed_replay_requantises_once(per_channel):
    """Replay of n tokens = n FP32 steps from the dequantised state, then one
    requantisation: compare with the FP32 oracle replay on the dequantised
    state (same permuted coordinates is not needed: logical rows compared)."""
    d, khi, T_max = 32, 4, 6
    w, pi, pool = make(23, per_channel, d=d, khi=khi, steps=T_max)
    n_acc = np.array([0, 6, 3], np.int32)
    q, k, v, a, b = gen.replay_view(w, T_max)
    S_in = logical(pool, d, khi, pi)
    p = pool.copy()
    o_m, st = orc.replay_mixed(p, w.slot_idx, n_acc, pi, khi, d, d, q, k, v, a, b)
    assert st == 0
    S_out = logical(p, d, khi, pi)
    for bb in range(w.B):
        s = w.slot_idx[bb]
        for h in range(w.Hv):
            g_ = h // (w.Hv // w.Hk)
            S_ref = S_in[s, h].copy()
            for t in range(n_acc[bb]):
                aa = a[bb, t, h] if per_channel else np.full(d, a[bb, t, h])
                S_ref, o_ref = damp_eq2_step(S_ref, q[bb, t, g_].astype(np.float64),
                                             k[bb, t, g_].astype(np.float64),
                                             v[bb, t, h].astype(np.float64),
                                             np.asarray(aa, np.float64), np.float64(b[bb, t, h]))
                assert np.max(np.abs(o_m[bb, t, h] - o_ref)) <= 3e-5 * max(1, np.abs(o_ref).max())
            if n_acc[bb] == 0:
                assert np.array_equal(p[s, h], pool[s, h])
                continue
            for r in range(d):
                c = pi[h, r]
                err = np.max(np.abs(S_out[s, h, c] - S_ref[c]))
                slop = 1e-5 * max(1.0, np.max(np.abs(S_ref[c])))
                if r < khi:
                    half_ulp = np.max(np.spacing(np.abs(S_ref[c]).astype(np.float16))
                                      .astype(np.float64)) / 2
                    assert err <= half_ulp + slop
                else:
                    assert err <= np.max(np.abs(S_ref[c])) / 127.0 * 0.5 * (1 + 1e-4) + slop


def test_permutation_is_applied_to_inputs():
    """Pin that the mixed oracle gathers q, k and the per-channel decay by the
    row map: with an identity map the mixed step on the permuted pool must
    differ from the logical step unless the inputs are gathered."""
    d, khi = 16, 4
    w, pi, pool = make(24, True, d=d, khi=khi, B=1, Hk=1, Hv=1, steps=1)
    assert not np.array_equal(pi[0], np.arange(d))
    ident = np.arange(d, dtype=np.int16)[None]
    # permute the logical FP32 state by hand, then run the identity-map oracle
    # on inputs permuted by hand: both routes must agree bit for bit.
    S0 = w.state0.copy()
    S_perm = S0[:, :, pi[0]].copy()
    pool_a = orc.convert_pool_f32_to_mixed(S0, khi, pi)
    pool_b = orc.convert_pool_f32_to_mixed(S_perm, khi, ident)
    assert np.array_equal(pool_a, pool_b)
    oa, _ = orc.decode_mixed(pool_a, w.slot_idx, pi, khi, d, d, w.q[0], w.k[0], w.v[0],
                             w.alpha[0], w.beta[0])
    qp, kp = w.q[0][:, :, pi[0]].copy(), w.k[0][:, :, pi[0]].copy()
    ap = w.alpha[0][:, :, pi[0]].copy()
    ob, _ = orc.decode_mixed(pool_b, w.slot_idx, ident, khi, d, d, qp, kp, w.v[0], ap,
                             w.beta[0])
    assert np.array_equal(pool_a, pool_b)
    assert np.array_equal(oa.view(np.uint32), ob.view(np.uint32))
