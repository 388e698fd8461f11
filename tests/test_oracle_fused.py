"""Pins for the oracle's fused requantisation arithmetic (mode 1, CPU only).

The pages fix the quantiser (DAMP §3.2 Eq. 5-6; dasc Appendix E.1 Eq. 8:
s = max(a, 1e-8)/127, code = clip(round(x/s), -127, 127), FP32) and the step
(DAMP Appendix A.4: dequantise, decay and update in FP32, requantise), not how
a kernel evaluates x/s or where the decay's rounding falls.  Mode 1 is the
division-free reading: the code is the integer nearest to the exact product
x * RN(1/s) (ties to even); the step itself (dequantise c * s, decay, update)
is mode 0's, so only the rounding of the new codes differs.

Pins, each independent of the oracle's own formulas:
  - the code against exact rational arithmetic (``fractions.Fraction``),
    including exact ties and a double-rounding trap;
  - mode-1 codes differ from mode-0 (IEEE quotient) codes by at most one and
    only where the exact quotient lies within the acceptance allowance,
    1e-6 max(1, |x/s|), of a half-integer; a constructed row where they do
    differ keeps the check from being vacuous;
  - one mode-1 step against the FP64 update of the dequantised input (DAMP
    §3.1 Eq. 2), within the local quantisation error of DAMP §3.3 Eq. 9;
  - replay of one token equals a decode step, replay requantises once;
  - with any decay the two modes agree on every byte but codes at a tie,
    and a teacher-forced comparison of the two meets the acceptance rule;
  - the same for the DAMP-exact layout (INT8 groups of 32 along dv).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle as orc
from recurrent_state_gb300 import inputs as gen

from .acceptance import Tally, compare_tile, reference_step_mixed
from .test_oracle_mixed import damp_eq2_step, logical


def nearest_even(fr: Fraction) -> int:
    return round(fr)   # Fraction.__round__ rounds half to even


def rcp32(s) -> np.float32:
    return np.float32(1.0) / np.float32(s)   # IEEE binary32 division


def expected_rcp_code(x, s) -> int:
    y = rcp32(s)
    return max(-127, min(127, nearest_even(Fraction(float(np.float32(x))) * Fraction(float(y)))))


def expected_ieee_code(x, s) -> int:
    q = np.float32(x) / np.float32(s)
    return int(max(-127.0, min(127.0, float(np.rint(q)))))


def test_rcp_code_is_nearest_integer_to_exact_product():
    g = gen.rng(100)
    for _ in range(3000):
        s = np.float32(np.exp(g.uniform(np.log(1e-6), np.log(1e3))))
        x = np.float32(g.uniform(-127.0, 127.0) * s)
        assert orc.quant_code_rcp(x, rcp32(s)) == expected_rcp_code(x, s)
    # exact ties with a power-of-two scale (1/s exact): half to even
    for n2 in range(-253, 254, 2):          # x/s = n2 / 2, odd n2: a tie
        s = np.float32(2.0 ** -7)
        x = np.float32(n2 / 2.0) * s
        assert orc.quant_code_rcp(x, rcp32(s)) == nearest_even(Fraction(n2, 2))


def test_rcp_code_rounds_the_exact_product_once():
    """Find x, y with RN32(x*y) exactly on a tie while the exact product is
    not: the code must follow the exact product (one rounding)."""
    found = 0
    g = gen.rng(101)
    for _ in range(4000):
        y = np.float32(g.uniform(0.5, 1.0))
        x0 = np.float32(np.float32(2.5) / y)
        cands, up, dn = [x0], x0, x0
        for _k in range(40):
            up = np.nextafter(up, np.float32(np.inf))
            dn = np.nextafter(dn, np.float32(-np.inf))
            cands += [np.float32(up), np.float32(dn)]
        for x in cands:
            exact = Fraction(float(x)) * Fraction(float(y))
            if np.float32(x) * y == np.float32(2.5) and exact != Fraction(5, 2):
                assert orc.quant_code_rcp(x, y) == nearest_even(exact)
                found += 1
                break
        if found >= 5:
            break
    assert found >= 5


def test_fused_row_codes_follow_the_exact_product_rule():
    g = gen.rng(102)
    for trial in range(40):
        n = 128
        scale = np.exp(g.uniform(-12, 8))
        x = (g.standard_normal(n) * scale).astype(np.float32)
        c1, s1 = orc.quantise_row(x, mode=1)
        c0, s0 = orc.quantise_row(x, mode=0)
        a = np.max(np.abs(x))
        assert s1 == s0 == np.float32(max(a, np.float32(1e-8))) / np.float32(127.0)
        exp = np.array([expected_rcp_code(v, s1) for v in x], np.int8)
        assert np.array_equal(c1, exp), trial


def test_fused_nonfinite_rows_keep_the_ieee_quotient():
    for bad in (np.inf, -np.inf, np.nan):
        x = np.linspace(-3, 3, 32).astype(np.float32)
        x[7] = bad
        c1, s1 = orc.quantise_row(x, mode=1)
        c0, s0 = orc.quantise_row(x, mode=0)
        assert np.array_equal(c1, c0) and (s1 == s0 or (np.isnan(s1) and np.isnan(s0)))


def boundary_ok(x, s, c0, c1):
    """Mode-1 code c1 may differ from the IEEE code c0 only by one, and only
    where the exact quotient lies within 1e-6 max(1, |x/s|) of a half-integer."""
    if c0 == c1:
        return True
    if abs(int(c0) - int(c1)) != 1:
        return False
    q = Fraction(float(np.float32(x))) / Fraction(float(np.float32(s)))
    half = Fraction(min(int(c0), int(c1))) + Fraction(1, 2)
    return abs(q - half) <= Fraction(1, 10 ** 6) * max(1, abs(q))


def test_fused_codes_differ_from_ieee_only_at_boundaries():
    g = gen.rng(103)
    n_diff = 0
    rows = 0
    for _ in range(3000):
        x = (g.standard_normal(128) * np.exp(g.uniform(-6, 6))).astype(np.float32)
        c0, s = orc.quantise_row(x, mode=0)
        c1, s1 = orc.quantise_row(x, mode=1)
        assert s == s1
        rows += 1
        for i in np.nonzero(c0 != c1)[0]:
            assert boundary_ok(x[i], s, c0[i], c1[i]), (x[i], s, c0[i], c1[i])
            n_diff += 1
    assert n_diff <= 1e-4 * rows * 128   # a boundary case is rare


def test_constructed_row_where_the_modes_differ():
    """Near a tie the IEEE quotient and the reciprocal product can round to
    different integers; such a row exists and both modes stay within the
    boundary allowance on it."""
    g = gen.rng(104)
    for _ in range(20000):
        s = np.float32(np.exp(g.uniform(-8, 4)))
        n = int(g.integers(-126, 126))
        x0 = np.float32((n + 0.5) * float(s))
        cands, up, dn = [x0], x0, x0
        for _k in range(6):
            up = np.nextafter(up, np.float32(np.inf))
            dn = np.nextafter(dn, np.float32(-np.inf))
            cands += [np.float32(up), np.float32(dn)]
        for x in cands:
            e0, e1 = expected_ieee_code(x, s), expected_rcp_code(x, s)
            if e0 != e1:
                # a row whose absmax fixes the scale s exactly: 127 s is a value of the row
                a = np.float32(np.float32(127.0) * s)
                if np.float32(max(a, np.float32(1e-8))) / np.float32(127.0) != s:
                    continue
                row = np.array([a, x], np.float32)
                c0, _ = orc.quantise_row(row, mode=0)
                c1, _ = orc.quantise_row(row, mode=1)
                assert (c0[1], c1[1]) == (e0, e1)
                assert boundary_ok(x, s, e0, e1)
                return
    pytest.fail("no row found where the two quotients round differently")


def make_strong(seed, per_channel, B=3, Hk=2, Hv=4, d=32, khi=4, steps=4, mode=1):
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=d, steps=steps, per_channel=per_channel,
                            in_dtype="bf16", seed=seed)
    g = gen.rng(seed + 1000)
    # strong decays, so that a decay applied twice or not at all is far
    # outside the quantisation error
    w.alpha[...] = g.uniform(0.3, 0.9, w.alpha.shape).astype(np.float32)
    hi = gen.hi_rows(Hv, d, khi, seed=seed)
    pi = orc.row_map(hi, d)
    pool = orc.convert_pool_f32_to_mixed(w.state0, khi, pi, mode=mode)
    return w, pi, pool


@pytest.mark.parametrize("per_channel", [False, True])
def test_fused_step_within_local_quantisation_error(per_channel):
    d, khi = 32, 4
    w, pi, pool = make_strong(110, per_channel, d=d, khi=khi)
    for t in range(w.steps):
        S_in = logical(pool, d, khi, pi)
        o, st = orc.decode_mixed(pool, w.slot_idx, pi, khi, d, d, w.q[t], w.k[t], w.v[t],
                                 w.alpha[t], w.beta[t], mode=1)
        assert st == 0
        S_out = logical(pool, d, khi, pi)
        for b in range(w.B):
            s = w.slot_idx[b]
            for h in range(w.Hv):
                g_ = h // (w.Hv // w.Hk)
                a = w.alpha[t, b, h] if per_channel else np.full(d, w.alpha[t, b, h])
                S_ref, o_ref = damp_eq2_step(S_in[s, h], w.q[t, b, g_].astype(np.float64),
                                             w.k[t, b, g_].astype(np.float64),
                                             w.v[t, b, h].astype(np.float64),
                                             np.asarray(a, np.float64), np.float64(w.beta[t, b, h]))
                assert np.max(np.abs(o[b, h] - o_ref)) <= 2e-5 * max(1.0, np.max(np.abs(o_ref)))
                for r in range(d):
                    c = pi[h, r]
                    err = np.max(np.abs(S_out[s, h, c] - S_ref[c]))
                    slop = 4e-6 * max(1.0, np.max(np.abs(S_ref[c])))
                    if r < khi:
                        half_ulp = np.max(np.spacing(np.abs(S_ref[c]).astype(np.float16))
                                          .astype(np.float64)) / 2
                        assert err <= half_ulp + slop, (t, b, h, r)
                    else:
                        sc = np.max(np.abs(S_ref[c])) / 127.0
                        assert err <= sc * 0.5 * (1 + 1e-4) + slop, (t, b, h, r, err, sc)


@pytest.mark.parametrize("per_channel", [False, True])
def test_fused_replay_one_equals_decode(per_channel):
    d, khi = 32, 4
    w, pi, pool = make_strong(111, per_channel, d=d, khi=khi)
    q, k, v, a, b = gen.replay_view(w, 1)
    p1 = pool.copy()
    o1, _ = orc.decode_mixed(p1, w.slot_idx, pi, khi, d, d, w.q[0], w.k[0], w.v[0],
                             w.alpha[0], w.beta[0], mode=1)
    p2 = pool.copy()
    o2, st = orc.replay_mixed(p2, w.slot_idx, np.ones(w.B, np.int32), pi, khi, d, d,
                              q, k, v, a, b, mode=1)
    assert st == 0
    assert np.array_equal(p1, p2)
    assert np.array_equal(o1.view(np.uint32), o2[:, 0].view(np.uint32))


@pytest.mark.parametrize("per_channel", [False, True])
def test_fused_replay_requantises_once(per_channel):
    d, khi, T_max = 32, 4, 5
    w, pi, pool = make_strong(112, per_channel, d=d, khi=khi, steps=T_max)
    n_acc = np.array([0, 5, 2], np.int32)
    q, k, v, a, b = gen.replay_view(w, T_max)
    S_in = logical(pool, d, khi, pi)
    p = pool.copy()
    o_m, st = orc.replay_mixed(p, w.slot_idx, n_acc, pi, khi, d, d, q, k, v, a, b, mode=1)
    assert st == 0
    S_out = logical(p, d, khi, pi)
    for bb in range(w.B):
        s = w.slot_idx[bb]
        for h in range(w.Hv):
            g_ = h // (w.Hv // w.Hk)
            if n_acc[bb] == 0:
                assert np.array_equal(p[s, h], pool[s, h])
                continue
            S_ref = S_in[s, h].copy()
            for t in range(n_acc[bb]):
                aa = a[bb, t, h] if per_channel else np.full(d, a[bb, t, h])
                S_ref, o_ref = damp_eq2_step(S_ref, q[bb, t, g_].astype(np.float64),
                                             k[bb, t, g_].astype(np.float64),
                                             v[bb, t, h].astype(np.float64),
                                             np.asarray(aa, np.float64), np.float64(b[bb, t, h]))
                assert np.max(np.abs(o_m[bb, t, h] - o_ref)) <= 3e-5 * max(1, np.abs(o_ref).max())
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


def split_tile(tile, d, khi):
    hi = tile[..., :2 * khi * d]
    lo = tile[..., 2 * khi * d:2 * khi * d + (d - khi) * d]
    sc = tile[..., 2 * khi * d + (d - khi) * d:]
    return hi, lo, sc


@pytest.mark.parametrize("per_channel", [False, True])
def test_modes_agree_but_at_ties(per_channel):
    """Both modes run the same FP32 step (strong decays here) and differ only
    in how the new codes are rounded."""
    d, khi = 64, 8
    w, pi, pool = make_strong(113, per_channel, B=4, Hk=2, Hv=4, d=d, khi=khi, mode=0)
    p0, p1 = pool.copy(), pool.copy()
    o0, _ = orc.decode_mixed(p0, w.slot_idx, pi, khi, d, d, w.q[0], w.k[0], w.v[0], w.alpha[0],
                             w.beta[0], mode=0)
    o1, _ = orc.decode_mixed(p1, w.slot_idx, pi, khi, d, d, w.q[0], w.k[0], w.v[0], w.alpha[0],
                             w.beta[0], mode=1)
    assert np.array_equal(o0.view(np.uint32), o1.view(np.uint32))
    h0, l0, s0 = split_tile(p0, d, khi)
    h1, l1, s1 = split_tile(p1, d, khi)
    assert np.array_equal(h0, h1) and np.array_equal(s0, s1)
    diff = np.abs(l0.view(np.int8).astype(int) - l1.view(np.int8).astype(int))
    assert diff.max() <= 1 and np.count_nonzero(diff) <= 1e-3 * diff.size


# ---- DAMP-exact layout (INT8 groups of 32 along dv, value scaling) --------
DD, DKHI, DG = 64, 8, 32


def make_damp(seed, per_channel, B=2, Hk=2, Hv=2, steps=3):
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=DD, steps=steps, per_channel=per_channel,
                            in_dtype="f32", seed=seed)
    g = gen.rng(seed + 2000)
    w.alpha[...] = g.uniform(0.3, 0.9, w.alpha.shape).astype(np.float32)
    hi = gen.hi_rows(Hv, DD, DKHI, seed=seed)
    pi = orc.row_map(hi, DD)
    cs = gen.value_scales(Hv, DD, seed=seed, group=DG)
    pool = orc.convert_pool_f32_to_damp(w.state0, DKHI, DG, pi, cs, mode=1)
    return w, pi, cs, pool


@pytest.mark.parametrize("per_channel", [False, True])
def test_damp_fused_step_within_group_error(per_channel):
    w, pi, cs, pool = make_damp(121, per_channel)
    for t in range(w.steps):
        S_in = orc.convert_pool_damp_to_f32(pool, DD, DD, DKHI, DG, pi, cs).astype(np.float64)
        o, st = orc.decode_damp(pool, w.slot_idx, pi, cs, DKHI, DG, DD, DD, w.q[t], w.k[t], w.v[t],
                                w.alpha[t], w.beta[t], mode=1)
        assert st == 0
        S_out = orc.convert_pool_damp_to_f32(pool, DD, DD, DKHI, DG, pi, cs).astype(np.float64)
        for b in range(w.B):
            s = w.slot_idx[b]
            for h in range(w.Hv):
                g_ = h // (w.Hv // w.Hk)
                a = w.alpha[t, b, h] if per_channel else np.full(DD, w.alpha[t, b, h])
                S_ref, o_ref = damp_eq2_step(S_in[s, h], w.q[t, b, g_].astype(np.float64),
                                             w.k[t, b, g_].astype(np.float64),
                                             w.v[t, b, h].astype(np.float64),
                                             np.asarray(a, np.float64), np.float64(w.beta[t, b, h]))
                assert np.max(np.abs(o[b, h] - o_ref)) <= 3e-5 * max(1.0, np.max(np.abs(o_ref)))
                for r in range(DKHI, DD):
                    c = pi[h, r]
                    for gi in range(DD // DG):
                        sl = slice(gi * DG, (gi + 1) * DG)
                        # the group's step, in stored (value-scaled) coordinates
                        tgt = S_ref[c, sl] / cs[h, sl]
                        err = np.max(np.abs((S_out[s, h, c, sl] - S_ref[c, sl]) / cs[h, sl]))
                        slop = 1e-5 * max(1.0, np.max(np.abs(tgt)))
                        assert err <= np.max(np.abs(tgt)) / 127.0 * 0.5 * (1 + 1e-4) + slop


@pytest.mark.parametrize("per_channel", [False, True])
def test_damp_fused_replay_one_equals_decode(per_channel):
    w, pi, cs, pool = make_damp(122, per_channel)
    q, k, v, a, b = gen.replay_view(w, 1)
    p1, p2 = pool.copy(), pool.copy()
    o1, _ = orc.decode_damp(p1, w.slot_idx, pi, cs, DKHI, DG, DD, DD, w.q[0], w.k[0], w.v[0],
                            w.alpha[0], w.beta[0], mode=1)
    o2, st = orc.replay_damp(p2, w.slot_idx, np.ones(w.B, np.int32), pi, cs, DKHI, DG, DD, DD,
                             q, k, v, a, b, mode=1)
    assert st == 0 and np.array_equal(p1, p2)
    assert np.array_equal(o1.view(np.uint32), o2[:, 0].view(np.uint32))


# ---- mode 1 against the pages' quantiser under real decays ---------------
@pytest.mark.parametrize("layout", ["mixed", "damp"])
def test_reference_step_is_the_oracle_mode0_step(layout):
    """The teacher-forced reference (unpack, one FP32 step, IEEE requantise)
    is the oracle's batched mode-0 decode, byte for byte."""
    d, khi, Hv = 128, 16, 4
    group = DG if layout == "damp" else 0
    w = gen.decode_workload(B=3, Hk=2, Hv=Hv, d=d, steps=1, per_channel=True, in_dtype="bf16",
                            seed=41, horizon=(2.0, 8192.0))
    pi = orc.row_map(gen.hi_rows(Hv, d, khi, seed=41), d)
    cs = gen.value_scales(Hv, d, seed=41) if group else None
    if group:
        pool = orc.convert_pool_f32_to_damp(w.state0, khi, group, pi, cs)
        before = pool.copy()
        o, _ = orc.decode_damp(pool, w.slot_idx, pi, cs, khi, group, d, d, w.q[0], w.k[0], w.v[0],
                               w.alpha[0], w.beta[0])
    else:
        pool = orc.convert_pool_f32_to_mixed(w.state0, khi, pi)
        before = pool.copy()
        o, _ = orc.decode_mixed(pool, w.slot_idx, pi, khi, d, d, w.q[0], w.k[0], w.v[0],
                                w.alpha[0], w.beta[0])
    for b in range(w.B):
        s = w.slot_idx[b]
        for h in range(Hv):
            g_ = h // (Hv // w.Hk)
            tile, _, o_r = reference_step_mixed(before[s, h], pi[h], w.q[0, b, g_], w.k[0, b, g_],
                                                w.v[0, b, h], w.alpha[0, b, h], w.beta[0, b, h],
                                                d, d, khi, group, None if cs is None else cs[h])
            assert np.array_equal(tile, pool[s, h])
            assert np.array_equal(o_r.view(np.uint32), o[b, h].view(np.uint32))


@pytest.mark.parametrize("layout,per_channel", [("mixed", True), ("mixed", False), ("damp", True)])
def test_fused_mode_meets_the_acceptance_rule_under_decay(layout, per_channel):
    """Teacher-forced, with real decays (alpha != 1, so the two modes also
    round the decay differently): every step, one mode-1 step and one step of
    the pages' quantiser (mode 0) start from the same packed bytes; codes must
    be equal except +-1 within 1e-6 max(1, |x/s|) of a rounding boundary,
    scales and FP16 rows within one ulp, o within 1e-3 (dasc Appendix E.1
    Eq. 8; DAMP §3.2 Eq. 5-6)."""
    d, khi = 128, 16
    group = DG if layout == "damp" else 0
    Hk, Hv = (4, 4) if per_channel else (2, 4)
    w = gen.decode_workload(B=12, Hk=Hk, Hv=Hv, d=d, steps=6, per_channel=per_channel,
                            in_dtype="bf16", seed=43,
                            horizon=(2.0, 8192.0) if per_channel else (4.0, 4096.0))
    pi = orc.row_map(gen.hi_rows(Hv, d, khi, seed=43), d)
    cs = gen.value_scales(Hv, d, seed=43) if group else None
    if group:
        pool = orc.convert_pool_f32_to_damp(w.state0, khi, group, pi, cs, mode=1)
    else:
        pool = orc.convert_pool_f32_to_mixed(w.state0, khi, pi, mode=1)
    tally = Tally()
    for t in range(w.steps):
        before = pool.copy()
        if group:
            o1, st = orc.decode_damp(pool, w.slot_idx, pi, cs, khi, group, d, d, w.q[t], w.k[t],
                                     w.v[t], w.alpha[t], w.beta[t], mode=1)
        else:
            o1, st = orc.decode_mixed(pool, w.slot_idx, pi, khi, d, d, w.q[t], w.k[t], w.v[t],
                                      w.alpha[t], w.beta[t], mode=1)
        assert st == 0
        for b in range(w.B):
            s = w.slot_idx[b]
            for h in range(Hv):
                g_ = h // (Hv // Hk)
                ref, x, o_r = reference_step_mixed(before[s, h], pi[h], w.q[t, b, g_], w.k[t, b, g_],
                                                   w.v[t, b, h], w.alpha[t, b, h], w.beta[t, b, h],
                                                   d, d, khi, group, None if cs is None else cs[h])
                compare_tile(tally, pool[s, h], ref, x, o1[b, h], o_r, d, d, khi, group,
                             where=f"step {t} seq {b} head {h}")
    assert tally.ok(), tally.failures[:5]
    # the modes share the FP32 step: scales, FP16 rows and o agree exactly
    assert tally.scale_ulp_max == 0 and tally.fp16_ulp_max == 0 and tally.o_rel_max == 0.0
    assert tally.codes == w.steps * w.B * Hv * (d - khi) * d
