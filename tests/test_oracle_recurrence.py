"""Pins for the oracle's decode recurrence (CPU only).

The oracle evaluates the expanded update of the DAMP page (§3.1) as explicit
FP32 loops.  These tests pin it to things other than itself:

* the pages' own matrix statements, evaluated in FP64 with numpy:
  DAMP §3.1 Eq. 2 ``S_t = (I - b k k^T) Lambda S_{t-1} + b k v^T`` with
  ``o = S_t^T q`` (Eq. 1), and dasc §3.1 Eq. 1
  ``S_t = S_{t-1} Diag(a) (I - b k k^T) + b v k^T`` with ``o = S q`` on the
  transposed state;
* invariants the update must satisfy exactly (identity, pure decay, exact
  write with a unit key, GDN as KDA with a constant decay vector);
* the GQA sharing rule of dasc Appendix B.1 (adjacent value heads share a key
  head);
* replay of n logged tokens equals n single steps (Serving recurrent
  attention, "Speculative decoding without state snapshots").
"""
import numpy as np
import pytest

import oracle as orc
from recurrent_state_gb300 import inputs as gen


def damp_eq2_step(S, q, k, v, a, beta):
    """DAMP §3.1 Eq. 1-2 in FP64: rows of S are key channels."""
    dk = k.size
    A = (np.eye(dk) - beta * np.outer(k, k)) @ np.diag(a)
    S = A @ S + beta * np.outer(k, v)
    return S, S.T @ q


def dasc_eq1_step(S1, q, k, v, a, beta):
    """dasc §3.1 Eq. 1 in FP64: S1 is dv x dk and o = S1 q."""
    dk = k.size
    S1 = S1 @ np.diag(a) @ (np.eye(dk) - beta * np.outer(k, k)) + beta * np.outer(v, k)
    return S1, S1 @ q


def rel(x, ref):
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


@pytest.fixture(scope="module")
def tiny():
    # The small GDN case: batch 4, 4 heads, d = 64, 16 steps, fp32 inputs.
    return gen.decode_workload(B=4, Hk=4, Hv=4, d=64, steps=16, per_channel=False,
                               in_dtype="f32", seed=0, tiny_gdn=True)


def test_page_forms_agree_with_each_other():
    """The two pages' statements are the same map up to transposition (FP64)."""
    g = gen.rng(1)
    dk, dv = 8, 6
    S = g.standard_normal((dk, dv))
    for _ in range(10):
        q, k = gen.l2_normalise(g.standard_normal(dk)), gen.l2_normalise(g.standard_normal(dk))
        q, k = q.astype(np.float64), k.astype(np.float64)
        v, a, beta = g.standard_normal(dv), g.uniform(0.2, 1.0, dk), g.uniform()
        S2, o2 = damp_eq2_step(S, q, k, v, a, beta)
        S1, o1 = dasc_eq1_step(S.T.copy(), q, k, v, a, beta)
        assert np.max(np.abs(S2 - S1.T)) < 1e-12
        assert np.max(np.abs(o2 - o1)) < 1e-12
        S = S2


@pytest.mark.parametrize("form", ["damp_eq2", "dasc_eq1"])
def test_oracle_matches_page_matrix_forms_fp64(tiny, form):
    """16 steps of the tiny GDN case, every head, against FP64 matrix forms."""
    w = tiny
    pool = w.state0.copy()
    ref = w.state0.astype(np.float64)
    worst_s = worst_o = 0.0
    for t in range(w.steps):
        o, st = orc.decode_f32(pool, w.slot_idx, w.q[t], w.k[t], w.v[t], w.alpha[t], w.beta[t])
        assert st == 0
        for b in range(w.B):
            s = w.slot_idx[b]
            for h in range(w.Hv):
                args = (w.q[t, b, h].astype(np.float64), w.k[t, b, h].astype(np.float64),
                        w.v[t, b, h].astype(np.float64),
                        np.full(w.dk, np.float64(w.alpha[t, b, h])), np.float64(w.beta[t, b, h]))
                if form == "damp_eq2":
                    ref[s, h], o_ref = damp_eq2_step(ref[s, h], *args)
                else:
                    S1, o_ref = dasc_eq1_step(ref[s, h].T.copy(), *args)
                    ref[s, h] = S1.T
                worst_o = max(worst_o, rel(o[b, h], o_ref))
                worst_s = max(worst_s, rel(pool[s, h], ref[s, h]))
    # FP32 against FP64 over 16 contracting steps of a 64 x 64 state
    assert worst_s < 2e-6, worst_s
    assert worst_o < 2e-5, worst_o


def test_kda_matches_page_form_fp64():
    """Per-channel decay (KDA, DAMP §3.1 Lambda = diag(exp g)), bf16 inputs,
    d = 128, GQA 2:1, 8 steps on a few heads."""
    w = gen.decode_workload(B=2, Hk=2, Hv=4, d=128, steps=8, per_channel=True,
                            in_dtype="bf16", seed=3, horizon=(2.0, 8192.0))
    pool = w.state0.copy()
    ref = w.state0.astype(np.float64)
    for t in range(w.steps):
        o, st = orc.decode_f32(pool, w.slot_idx, w.q[t], w.k[t], w.v[t], w.alpha[t], w.beta[t])
        assert st == 0
        for b in range(w.B):
            s = w.slot_idx[b]
            for h in range(w.Hv):
                g_ = h // (w.Hv // w.Hk)
                ref[s, h], o_ref = damp_eq2_step(
                    ref[s, h], w.q[t, b, g_].astype(np.float64), w.k[t, b, g_].astype(np.float64),
                    w.v[t, b, h].astype(np.float64), w.alpha[t, b, h].astype(np.float64),
                    np.float64(w.beta[t, b, h]))
                assert rel(o[b, h], o_ref) < 2e-5
    assert rel(pool, ref) < 2e-6


def test_gqa_uses_adjacent_key_head():
    """Value head h reads key head h // (Hv/Hk): poison every other key head's
    q/k with NaN and check that no output of head h turns NaN."""
    w = gen.decode_workload(B=1, Hk=4, Hv=8, d=16, steps=1, per_channel=False,
                            in_dtype="f32", seed=5)
    for g_ in range(w.Hk):
        q = w.q[0].copy()
        k = w.k[0].copy()
        others = [x for x in range(w.Hk) if x != g_]
        q[:, others] = np.nan
        k[:, others] = np.nan
        pool = w.state0.copy()
        o, _ = orc.decode_f32(pool, w.slot_idx, q, k, w.v[0], w.alpha[0], w.beta[0])
        for h in range(w.Hv):
            finite = np.all(np.isfinite(o[0, h]))
            assert finite == (h // 2 == g_), (g_, h)


def test_identity_when_alpha_one_beta_zero():
    g = gen.rng(2)
    S = g.standard_normal((32, 24)).astype(np.float32)
    S0 = S.copy()
    orc.step_tile(S, g.standard_normal(32), g.standard_normal(32), g.standard_normal(24),
                  np.float32(1.0), 0.0)
    assert np.array_equal(S.view(np.uint32), S0.view(np.uint32))


@pytest.mark.parametrize("per_channel", [False, True])
def test_beta_zero_is_pure_decay(per_channel):
    g = gen.rng(3)
    dk, dv = 48, 40
    S = g.standard_normal((dk, dv)).astype(np.float32)
    a = (g.uniform(0.1, 1.0, dk) if per_channel else np.array([0.83])).astype(np.float32)
    expect = (S * (a[:, None] if per_channel else a[0])).astype(np.float32)
    q = gen.l2_normalise(g.standard_normal(dk))
    o = orc.step_tile(S, q, gen.l2_normalise(g.standard_normal(dk)), g.standard_normal(dv), a, 0.0)
    assert np.array_equal(S.view(np.uint32), expect.view(np.uint32))
    assert rel(o, expect.astype(np.float64).T @ q.astype(np.float64)) < 1e-6


def test_unit_key_full_strength_writes_value():
    """alpha = 1, beta = 1, |k| = 1: afterwards S^T k = v (the delta rule
    replaces the association along k)."""
    g = gen.rng(4)
    dk, dv = 64, 64
    S = (g.standard_normal((dk, dv)) * 0.3).astype(np.float32)
    k = gen.l2_normalise(g.standard_normal(dk)).astype(np.float32)
    v = g.standard_normal(dv).astype(np.float32)
    orc.step_tile(S, k, k, v, np.float32(1.0), 1.0)
    pred = S.astype(np.float64).T @ k.astype(np.float64)
    assert np.max(np.abs(pred - v)) < 4e-6 * max(1.0, np.max(np.abs(v)))
    # FP64 statement: exact up to rounding of the inputs
    S64 = (g.standard_normal((dk, dv)))
    k64 = k.astype(np.float64) / np.linalg.norm(k.astype(np.float64))
    S64, _ = damp_eq2_step(S64, k64, k64, v.astype(np.float64), np.ones(dk), 1.0)
    assert np.max(np.abs(S64.T @ k64 - v)) < 1e-12


def test_gdn_equals_kda_with_constant_decay():
    w = gen.decode_workload(B=3, Hk=2, Hv=4, d=32, steps=4, per_channel=False,
                            in_dtype="bf16", seed=6)
    p1, p2 = w.state0.copy(), w.state0.copy()
    for t in range(w.steps):
        o1, _ = orc.decode_f32(p1, w.slot_idx, w.q[t], w.k[t], w.v[t], w.alpha[t], w.beta[t])
        a_vec = np.repeat(w.alpha[t][:, :, None], w.dk, axis=2).copy()
        o2, _ = orc.decode_f32(p2, w.slot_idx, w.q[t], w.k[t], w.v[t], a_vec, w.beta[t])
        assert np.array_equal(o1.view(np.uint32), o2.view(np.uint32))
    assert np.array_equal(p1.view(np.uint32), p2.view(np.uint32))


def test_zero_state_zero_strength_reads_zero():
    g = gen.rng(7)
    S = np.zeros((16, 16), np.float32)
    o = orc.step_tile(S, g.standard_normal(16), g.standard_normal(16), g.standard_normal(16),
                      np.float32(0.9), 0.0)
    assert np.all(o == 0.0)


def test_readout_is_transpose_of_updated_state():
    """o = S_t^T q with S_t the updated state (DAMP §3.1 Eq. 1), not S q and
    not the state before the update."""
    g = gen.rng(8)
    dk, dv = 24, 24
    S = g.standard_normal((dk, dv)).astype(np.float32)
    S_before = S.copy()
    q = gen.l2_normalise(g.standard_normal(dk))
    o = orc.step_tile(S, q, gen.l2_normalise(g.standard_normal(dk)), g.standard_normal(dv),
                      np.float32(0.7), 0.6)
    upd = S.astype(np.float64).T @ q
    assert rel(o, upd) < 1e-6
    assert rel(o, S.astype(np.float64) @ q) > 1e-2
    assert rel(o, S_before.astype(np.float64).T @ q) > 1e-2


@pytest.mark.parametrize("per_channel", [False, True])
def test_replay_equals_single_steps(per_channel):
    """Replaying n logged tokens is n decode steps, bit for bit; rows of o for
    t >= n are not written; n = 0 leaves the state untouched."""
    T_max = 8
    w = gen.decode_workload(B=6, Hk=2, Hv=4, d=32, steps=T_max, per_channel=per_channel,
                            in_dtype="bf16", seed=9)
    n_acc = np.array([0, 1, 3, 8, 5, 2], np.int32)
    q, k, v, a, b = gen.replay_view(w, T_max)
    pool_r = w.state0.copy()
    o_r = np.full((w.B, T_max, w.Hv, w.dv), -7.0, np.float32)
    _, st = orc.replay_f32(pool_r, w.slot_idx, n_acc, q, k, v, a, b, o=o_r)
    assert st == 0
    pool_s = w.state0.copy()
    for bb in range(w.B):
        one = np.array([w.slot_idx[bb]], np.int32)
        for t in range(n_acc[bb]):
            o1, _ = orc.decode_f32(pool_s, one, q[bb:bb + 1, t], k[bb:bb + 1, t],
                                   v[bb:bb + 1, t], a[bb:bb + 1, t], b[bb:bb + 1, t])
            assert np.array_equal(o1[0].view(np.uint32), o_r[bb, t].view(np.uint32))
        assert np.all(o_r[bb, n_acc[bb]:] == -7.0)
    assert np.array_equal(pool_r.view(np.uint32), pool_s.view(np.uint32))


def test_status_bits_skip_bad_items():
    w = gen.decode_workload(B=3, Hk=1, Hv=2, d=8, steps=2, per_channel=False,
                            in_dtype="f32", seed=10)
    pool = w.state0.copy()
    slots = np.array([0, 7, -1], np.int32)
    o = np.full((3, 2, 8), 5.0, np.float32)
    _, st = orc.decode_f32(pool, slots, w.q[0], w.k[0], w.v[0], w.alpha[0], w.beta[0], o=o)
    assert st == 1
    assert np.all(o[1:] == 5.0)
    q, k, v, a, b = gen.replay_view(w, 2)
    _, st = orc.replay_f32(w.state0.copy(), np.array([0, 1, 2], np.int32),
                           np.array([1, 3, -1], np.int32), q, k, v, a, b)
    assert st == 2
