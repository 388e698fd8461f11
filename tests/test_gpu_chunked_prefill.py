"""GPU parity of the chunk-parallel prefill on the tensor cores
(rs_prefill_chunked_update; DAMP Appendix A.4 "Prefill path"; "Serving
recurrent attention", "Kernels follow the serving phase").

The oracle is the plain recurrence: every token one decode step in FP32
(the oracle's multi-token replay).  The chunked form reorders the sums and
runs the large products as tf32 pairs with fp32 accumulation, so the bar is
a tolerance, not bit-exactness: per (sequence, head) tile, the final state
and every output row within 1e-5 of the oracle's, normwise
(||x - x_ref||_inf / ||x_ref||_inf), as for the FP32 state after 64 decode
steps.  Cases: GDN and KDA, grouped key heads, ragged token counts (0, 1, 32,
33, L and between) over two 32-token groups with a partial last one, bf16
and fp32 inputs, strong decays, and the full batch-256 workload with 32 and
64 tokens on sampled sequences.  On the mixed FP16/INT8 layout the oracle is its
sequential mixed prefill from the same packed bytes (dequantise once, FP32
steps, requantise once): outputs within the same tolerance, INT8 codes at
most one step apart (and rarely), row scales within the state tolerance over
127, and the dequantised state within the tolerance of the tile norm plus one
quantisation step of the FP32 state the oracle requantises.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import recurrent_state_gb300 as rs
from recurrent_state_gb300 import _abi
from recurrent_state_gb300 import inputs as gen

from .gpu_util import dev, ensure_built, host, replay_inputs, sub_batch

pytestmark = pytest.mark.gpu

D = 128
TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def tile_rel(x, ref):
    """max over tiles of ||x - ref||_inf / ||ref||_inf (tiles: the last two axes)."""
    x = x.astype(np.float64)
    ref = ref.astype(np.float64)
    num = np.max(np.abs(x - ref), axis=(-2, -1))
    den = np.maximum(np.max(np.abs(ref), axis=(-2, -1)), 1e-30)
    return float(np.max(num / den))


def run_case(B, Hk, Hv, L, per_channel, in_dtype, seed, n_tok=None, decay_range=None):
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=L, per_channel=per_channel,
                            in_dtype=in_dtype, seed=seed,
                            horizon=(2.0, 8192.0) if per_channel else (4.0, 4096.0))
    if decay_range is not None:  # decays far from 1
        w.alpha[...] = gen.rng(seed + 5).uniform(*decay_range, w.alpha.shape).astype(np.float32)
    if n_tok is None:
        n_tok = np.full(B, L, np.int32)
    qd, kd, vd, ad, bd = replay_inputs(w, L)
    q, k, v, a, b = gen.replay_view(w, L)
    lay = rs.Layout("fp32", D, Hv, Hk)
    pool = dev(w.state0)
    o = torch.full((B, L, Hv, D), 3.0, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rs.prefill_update(lay, per_channel, pool, dev(w.slot_idx), qd, kd, vd, ad, bd, n_tokens=dev(n_tok),
                      o=o, status=status, chunked=True)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return w, n_tok, (q, k, v, a, b), host(pool), host(o)


def check_against_oracle(w, n_tok, inputs, pool_g, o_g, bsel=None):
    q, k, v, a, b = inputs
    if bsel is None:
        bsel = np.arange(w.B)
    ws = sub_batch(w, bsel)
    L = q.shape[1]
    ref = ws.state0.copy()
    o_r = np.full((len(bsel), L, w.Hv, D), 3.0, np.float32)
    pick = lambda x: np.ascontiguousarray(x[bsel])
    _, st = orc.replay_f32(ref, ws.slot_idx, np.ascontiguousarray(n_tok[bsel]), pick(q), pick(k), pick(v),
                           pick(a), pick(b), o=o_r)
    assert st == 0
    s_err = tile_rel(pool_g[w.slot_idx[bsel]], ref)
    assert s_err <= TOL, f"state {s_err:.3g}"
    worst = 0.0
    for i, bb in enumerate(bsel):
        n = int(n_tok[bb])
        if n:
            got = np.swapaxes(o_g[bb, :n], 0, 1)     # [Hv][n][D]: tiles per head
            exp = np.swapaxes(o_r[i, :n], 0, 1)
            worst = max(worst, tile_rel(got, exp))
        assert np.all(o_g[bb, n:] == 3.0), "rows past n_tokens must stay untouched"
    assert worst <= TOL, f"o {worst:.3g}"
    return s_err, worst


@pytest.mark.parametrize("per_channel,Hk,Hv", [(True, 4, 4), (False, 2, 4), (False, 4, 4)])
def test_chunked_prefill_ragged_counts(per_channel, Hk, Hv):
    B, L = 11, 37
    n_tok = gen.rng(3).integers(0, L + 1, B).astype(np.int32)
    n_tok[0], n_tok[1], n_tok[2], n_tok[3], n_tok[4], n_tok[5] = 0, L, 1, 16, 32, 33
    w, n_tok, inputs, pool_g, o_g = run_case(B, Hk, Hv, L, per_channel, "bf16", seed=61, n_tok=n_tok)
    check_against_oracle(w, n_tok, inputs, pool_g, o_g)


@pytest.mark.parametrize("per_channel", [True, False])
@pytest.mark.parametrize("decay_range", [(0.02, 0.6), (0.001, 0.03)])
def test_chunked_prefill_fp32_inputs_and_strong_decay(per_channel, decay_range):
    """Strong decays: products over a 32-token group reach about 1e-26 (the
    factored form) and fall far below 1e-30 (the running products the kernel
    then takes)."""
    B, L = 6, 80
    w, n_tok, inputs, pool_g, o_g = run_case(B, 2, 2, L, per_channel, "f32", seed=62,
                                             decay_range=decay_range)
    assert np.all(np.isfinite(pool_g)) and np.all(np.isfinite(o_g))
    check_against_oracle(w, n_tok, inputs, pool_g, o_g)


@pytest.mark.parametrize("L", [32, 64])
def test_chunked_prefill_full_size_sampled(L):
    """KDA, batch 256, 32 heads, chunks of 32 and 64 tokens; oracle on sampled
    sequences (all heads)."""
    w, n_tok, inputs, pool_g, o_g = run_case(256, 32, 32, L, True, "bf16", seed=63)
    s_err, o_err = check_against_oracle(w, n_tok, inputs, pool_g, o_g, bsel=np.array([0, 97, 255]))
    print(f"\nchunked prefill L={L}: state {s_err:.3g}, o {o_err:.3g} (normwise per tile)")


def test_chunked_prefill_gdn_full_size_sampled():
    """GDN, batch 256, 16 key heads shared by 32 value heads, 32 tokens."""
    w, n_tok, inputs, pool_g, o_g = run_case(256, 16, 32, 32, False, "bf16", seed=64)
    check_against_oracle(w, n_tok, inputs, pool_g, o_g, bsel=np.array([1, 128, 254]))


def test_chunked_prefill_f16_inputs():
    """fp16 q, k, v (widened exactly), FP32 state: the same bar."""
    w, n_tok, inputs, pool_g, o_g = run_case(5, 2, 2, 40, True, "f16", seed=66)
    check_against_oracle(w, n_tok, inputs, pool_g, o_g)


@pytest.mark.parametrize("kind", ["fp32", "mixed"])
def test_chunked_prefill_bf16_outputs(kind):
    """bf16 outputs: the FP32 readout rounded to nearest even -- within half a bf16 ulp (2^-8 of the
    value: bf16 keeps 7 explicit mantissa bits) of the oracle's readout, plus the chunked form's
    tolerance."""
    B, Hk, Hv, L = 6, 2, 4, 33
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=L, per_channel=False, in_dtype="bf16", seed=67,
                            horizon=(4.0, 4096.0))
    qd, kd, vd, ad, bd = replay_inputs(w, L)
    q, k, v, a, b = gen.replay_view(w, L)
    hi = gen.hi_rows(Hv, D, 16, seed=67)
    pi = orc.row_map(hi, D)
    if kind == "fp32":
        lay, pool = rs.Layout("fp32", D, Hv, Hk), dev(w.state0)
    else:
        lay = rs.Layout("mixed", D, Hv, Hk, k_hi=16, hi_rows=hi)
        pool = dev(orc.convert_pool_f32_to_mixed(w.state0, 16, pi))
    n_tok = np.full(B, L, np.int32)
    o = torch.full((B, L, Hv, D), 3.0, dtype=torch.bfloat16, device="cuda")
    rs.prefill_update(lay, False, pool, dev(w.slot_idx), qd, kd, vd, ad, bd, o=o, chunked=True)
    torch.cuda.synchronize()
    s0 = w.state0 if kind == "fp32" else orc.convert_pool_mixed_to_f32(
        orc.convert_pool_f32_to_mixed(w.state0, 16, pi), D, D, 16, pi)
    ref = s0.copy()
    o_r = np.zeros((B, L, Hv, D), np.float32)
    _, st = orc.replay_f32(ref, w.slot_idx, n_tok, q, k, v, a, b, o=o_r)
    assert st == 0
    og = o.float().cpu().numpy()
    for bb in range(B):
        err = tile_rel(np.swapaxes(og[bb], 0, 1), np.swapaxes(o_r[bb], 0, 1))
        assert err <= 2.0 ** -8 + TOL, err


KHI = 16


def mixed_case(B, Hk, Hv, L, per_channel, seed, quant, n_tok=None, in_dtype="bf16"):
    """Chunked prefill on the mixed FP16/INT8 layout from packed tiles the oracle wrote; returns
    the GPU's packed pool and outputs beside the oracle's sequential mixed prefill from the same
    bytes and the FP32 state it requantises."""
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=L, per_channel=per_channel, in_dtype=in_dtype,
                            seed=seed, horizon=(2.0, 8192.0) if per_channel else (4.0, 4096.0))
    if n_tok is None:
        n_tok = np.full(B, L, np.int32)
    hi = gen.hi_rows(Hv, D, KHI, seed=seed)
    pi = orc.row_map(hi, D)
    mode = 1 if quant == "fused" else 0
    lay = rs.Layout("mixed", D, Hv, Hk, k_hi=KHI, hi_rows=hi, quant=quant)
    packed0 = orc.convert_pool_f32_to_mixed(w.state0, KHI, pi, mode=mode)
    qd, kd, vd, ad, bd = replay_inputs(w, L)
    q, k, v, a, b = gen.replay_view(w, L)
    pool = dev(packed0)
    o = torch.full((B, L, Hv, D), 3.0, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rs.prefill_update(lay, per_channel, pool, dev(w.slot_idx), qd, kd, vd, ad, bd, n_tokens=dev(n_tok),
                      o=o, status=status, chunked=True)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return w, n_tok, pi, mode, packed0, (q, k, v, a, b), host(pool), host(o)


def check_mixed(w, n_tok, pi, mode, packed0, inputs, pool_g, o_g, bsel=None):
    q, k, v, a, b = inputs
    if bsel is None:
        bsel = np.arange(w.B)
    ws = sub_batch(w, bsel)
    pick = lambda x: np.ascontiguousarray(x[bsel])
    L = q.shape[1]
    n_sel = np.ascontiguousarray(n_tok[bsel])
    sel = w.slot_idx[bsel]                       # the sampled sequences' tiles, renumbered 0..
    slots = ws.slot_idx
    p0 = np.ascontiguousarray(packed0[sel])
    # the oracle: sequential mixed prefill (dequantise once, FP32 steps, requantise once) ...
    ref = p0.copy()
    o_r = np.full((len(bsel), L, w.Hv, D), 3.0, np.float32)
    _, st = orc.replay_mixed(ref, slots, n_sel, pi, KHI, D, D, pick(q), pick(k), pick(v), pick(a), pick(b),
                             o=o_r, mode=mode)
    assert st == 0
    # ... and the FP32 state it requantises
    s32 = orc.convert_pool_mixed_to_f32(p0, D, D, KHI, pi)
    _, st = orc.replay_f32(s32, slots, n_sel, pick(q), pick(k), pick(v), pick(a), pick(b))
    assert st == 0
    worst = 0.0
    for i, bb in enumerate(bsel):
        n = int(n_tok[bb])
        if n:
            worst = max(worst, tile_rel(np.swapaxes(o_g[bb, :n], 0, 1), np.swapaxes(o_r[i, :n], 0, 1)))
        assert np.all(o_g[bb, n:] == 3.0), "rows past n_tokens must stay untouched"
    assert worst <= TOL, f"o {worst:.3g}"
    g = pool_g[sel]
    r = ref
    S = s32.astype(np.float64)                                      # [n][Hv][u][v], key-channel order
    norm = np.max(np.abs(S), axis=(-2, -1))                          # per tile
    hb, lb = 2 * KHI * D, (D - KHI) * D
    # INT8 codes: one step apart at most, and rarely
    cg = g[..., hb:hb + lb].view(np.int8).astype(np.int32)
    cr = r[..., hb:hb + lb].view(np.int8).astype(np.int32)
    diff = np.abs(cg - cr)
    assert diff.max() <= 1
    frac = float(np.mean(diff != 0))
    assert frac <= 5e-3, frac
    # row scales: within the state's tolerance (absmax / 127) and a few ulps
    sg = g[..., hb + lb:].copy().view(np.float32).astype(np.float64)  # [n][Hv][D - KHI]
    sr = r[..., hb + lb:].copy().view(np.float32).astype(np.float64)
    assert np.all(np.abs(sg - sr) <= TOL * norm[..., None] / 127.0 + 4 * np.spacing(sr.astype(np.float32)))
    # dequantised states: within the tolerance of the tile norm plus one quantisation step
    dg = orc.convert_pool_mixed_to_f32(np.ascontiguousarray(g), D, D, KHI, pi).astype(np.float64)
    step = np.zeros_like(S)
    rows = np.asarray(pi).reshape(w.Hv, D)                           # physical row -> key channel
    for hh in range(w.Hv):
        for rr in range(KHI, D):
            step[:, hh, rows[hh, rr], :] = np.maximum(sg[:, hh, rr - KHI], sr[:, hh, rr - KHI])[:, None]
        for rr in range(KHI):
            step[:, hh, rows[hh, rr], :] = np.abs(S[:, hh, rows[hh, rr], :]) * 2.0 ** -10 + 2.0 ** -24
    err = np.abs(dg - S) - step
    assert np.all(err <= TOL * norm[..., None, None]), float(np.max(err / norm[..., None, None]))
    return worst, frac


@pytest.mark.parametrize("quant", ["ieee", "fused"])
@pytest.mark.parametrize("per_channel,Hk,Hv", [(True, 4, 4), (False, 2, 4)])
def test_chunked_prefill_mixed_ragged(quant, per_channel, Hk, Hv):
    B, L = 9, 37
    n_tok = gen.rng(5).integers(0, L + 1, B).astype(np.int32)
    n_tok[0], n_tok[1], n_tok[2], n_tok[3] = 0, L, 1, 32
    res = mixed_case(B, Hk, Hv, L, per_channel, 71, quant, n_tok=n_tok)
    check_mixed(*res)


@pytest.mark.parametrize("quant", ["ieee", "fused"])
@pytest.mark.parametrize("L", [32, 64])
def test_chunked_prefill_mixed_full_size_sampled(quant, L):
    """KDA, batch 256, 32 heads, mixed FP16/INT8 state, sampled sequences (all heads)."""
    res = mixed_case(256, 32, 32, L, True, 72, quant)
    o_err, frac = check_mixed(*res, bsel=np.array([2, 130, 255]))
    print(f"\nchunked prefill, mixed {quant}, L={L}: o {o_err:.3g}, codes off by one {frac:.2g}")


def check_damp(w, n_tok, pi, cs, mode, packed0, inputs, pool_g, o_g, bsel=None):
    """DAMP-exact tiles (INT8 groups of 32 columns, value scaling): the rule of the mixed layout, on
    the stored state T = S diag(c')^-1 of each tile (physical rows), scales per (row, group)."""
    q, k, v, a, b = inputs
    if bsel is None:
        bsel = np.arange(w.B)
    ws = sub_batch(w, bsel)
    pick = lambda x: np.ascontiguousarray(x[bsel])
    L = q.shape[1]
    n_sel = np.ascontiguousarray(n_tok[bsel])
    sel = w.slot_idx[bsel]
    slots = ws.slot_idx
    p0 = np.ascontiguousarray(packed0[sel])
    ref = p0.copy()
    o_r = np.full((len(bsel), L, w.Hv, D), 3.0, np.float32)
    _, st = orc.replay_damp(ref, slots, n_sel, pi, cs, KHI, 32, D, D, pick(q), pick(k), pick(v), pick(a), pick(b),
                            o=o_r, mode=mode)
    assert st == 0
    s32 = orc.convert_pool_damp_to_f32(p0, D, D, KHI, 32, pi, cs)    # S, key-channel order
    _, st = orc.replay_f32(s32, slots, n_sel, pick(q), pick(k), pick(v), pick(a), pick(b))
    assert st == 0
    worst = 0.0
    for i, bb in enumerate(bsel):
        n = int(n_tok[bb])
        if n:
            worst = max(worst, tile_rel(np.swapaxes(o_g[bb, :n], 0, 1), np.swapaxes(o_r[i, :n], 0, 1)))
        assert np.all(o_g[bb, n:] == 3.0), "rows past n_tokens must stay untouched"
    assert worst <= TOL, f"o {worst:.3g}"
    g = pool_g[sel]
    hb, lb = 2 * KHI * D, (D - KHI) * D
    cg = g[..., hb:hb + lb].view(np.int8).astype(np.int32)
    cr = ref[..., hb:hb + lb].view(np.int8).astype(np.int32)
    diff = np.abs(cg - cr)
    assert diff.max() <= 1
    frac = float(np.mean(diff != 0))
    assert frac <= 5e-3, frac
    rows = np.asarray(pi).reshape(w.Hv, D)                           # physical row -> key channel
    csa = np.asarray(cs, np.float64).reshape(w.Hv, D)
    n_t = len(bsel)
    sg = g[..., hb + lb:].copy().view(np.float32).astype(np.float64).reshape(n_t, w.Hv, D - KHI, D // 32)
    sr = ref[..., hb + lb:].copy().view(np.float32).astype(np.float64).reshape(n_t, w.Hv, D - KHI, D // 32)
    for hh in range(w.Hv):
        T = s32[:, hh].astype(np.float64) / csa[hh][None, None, :]   # [n][u][v], key-channel order
        Tp = T[:, rows[hh], :]                                       # physical rows
        norm = np.max(np.abs(Tp), axis=(-2, -1))
        assert np.all(np.abs(sg[:, hh] - sr[:, hh]) <=
                      TOL * norm[:, None, None] / 127.0 + 4 * np.spacing(sr[:, hh].astype(np.float32)))
        dq = np.stack([orc.damp_unpack(g[i, hh], D, D, KHI, 32) for i in range(n_t)]).astype(np.float64)
        step = np.empty_like(Tp)
        step[:, :KHI, :] = np.abs(Tp[:, :KHI, :]) * 2.0 ** -10 + 2.0 ** -24
        grp = np.repeat(np.maximum(sg[:, hh], sr[:, hh]), 32, axis=-1)  # [n][row - KHI][v]
        step[:, KHI:, :] = grp
        err = np.abs(dq - Tp) - step
        assert np.all(err <= TOL * norm[:, None, None]), float(np.max(err / norm[:, None, None]))
    return worst, frac


def damp_case(B, Hk, Hv, L, per_channel, seed, quant, n_tok=None):
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=L, per_channel=per_channel, in_dtype="bf16",
                            seed=seed, horizon=(2.0, 8192.0) if per_channel else (4.0, 4096.0))
    if n_tok is None:
        n_tok = np.full(B, L, np.int32)
    hi = gen.hi_rows(Hv, D, KHI, seed=seed)
    pi = orc.row_map(hi, D)
    cs = gen.value_scales(Hv, D, seed=seed)
    mode = 1 if quant == "fused" else 0
    lay = rs.Layout("damp", D, Hv, Hk, k_hi=KHI, hi_rows=hi, value_scales=cs, quant=quant)
    packed0 = orc.convert_pool_f32_to_damp(w.state0, KHI, 32, pi, cs, mode=mode)
    qd, kd, vd, ad, bd = replay_inputs(w, L)
    q, k, v, a, b = gen.replay_view(w, L)
    pool = dev(packed0)
    o = torch.full((B, L, Hv, D), 3.0, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rs.prefill_update(lay, per_channel, pool, dev(w.slot_idx), qd, kd, vd, ad, bd, n_tokens=dev(n_tok),
                      o=o, status=status, chunked=True)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return w, n_tok, pi, cs, mode, packed0, (q, k, v, a, b), host(pool), host(o)


@pytest.mark.parametrize("quant", ["ieee", "fused"])
@pytest.mark.parametrize("per_channel,Hk,Hv", [(True, 4, 4), (False, 2, 4)])
def test_chunked_prefill_damp_ragged(quant, per_channel, Hk, Hv):
    B, L = 9, 37
    n_tok = gen.rng(6).integers(0, L + 1, B).astype(np.int32)
    n_tok[0], n_tok[1], n_tok[2], n_tok[3] = 0, L, 1, 32
    check_damp(*damp_case(B, Hk, Hv, L, per_channel, 73, quant, n_tok=n_tok))


@pytest.mark.parametrize("quant", ["ieee", "fused"])
def test_chunked_prefill_damp_full_size_sampled(quant):
    """KDA, batch 256, 32 heads, DAMP-exact state, 32 tokens, sampled sequences (all heads)."""
    o_err, frac = check_damp(*damp_case(256, 32, 32, 32, True, 74, quant), bsel=np.array([5, 199]))
    print(f"\nchunked prefill, DAMP-exact {quant}, L=32: o {o_err:.3g}, codes off by one {frac:.2g}")


@pytest.mark.parametrize("kind", ["fp32", "mixed", "damp"])
def test_chunked_prefill_guards_and_layouts(kind):
    B, Hk, Hv, L = 4, 2, 2, 5
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=L, per_channel=True, in_dtype="bf16", seed=65)
    qd, kd, vd, ad, bd = replay_inputs(w, L)
    hi = gen.hi_rows(Hv, D, 16, seed=1)
    pi = orc.row_map(hi, D)
    if kind == "fp32":
        lay, start = rs.Layout("fp32", D, Hv, Hk), w.state0
    elif kind == "mixed":
        lay = rs.Layout("mixed", D, Hv, Hk, k_hi=16, hi_rows=hi)
        start = orc.convert_pool_f32_to_mixed(w.state0, 16, pi)
    else:
        cs = gen.value_scales(Hv, D, seed=1)
        lay = rs.Layout("damp", D, Hv, Hk, k_hi=16, hi_rows=hi, value_scales=cs)
        start = orc.convert_pool_f32_to_damp(w.state0, 16, 32, pi, cs)
    pool = dev(start)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = w.slot_idx.copy()
    slots[1] = 999                                 # out of range: skipped, bit 1
    n_tok = np.array([L, L, L + 1, 2], np.int32)   # n > L: skipped, bit 2
    rs.prefill_update(lay, True, pool, dev(slots), qd, kd, vd, ad, bd, n_tokens=dev(n_tok),
                      status=status, chunked=True)
    torch.cuda.synchronize()
    assert int(status.item()) == (_abi.RS_DEV_BAD_SLOT | _abi.RS_DEV_BAD_ACCEPT)
    got = host(pool)
    for bb in (1, 2):  # skipped sequences keep their state
        if slots[bb] < start.shape[0]:
            assert np.array_equal(got[slots[bb]], start[slots[bb]])
    for bb in (0, 3):  # the others changed
        assert not np.array_equal(got[slots[bb]], start[slots[bb]])
    hi32 = gen.hi_rows(Hv, D, 32, seed=1)
    wide = rs.Layout("mixed", D, Hv, Hk, k_hi=32, hi_rows=hi32)  # 32 FP16 rows: the chunked form is not built
    with pytest.raises(rs.RsError) as e:
        rs.prefill_update(wide, True, wide.empty_pool(B), dev(w.slot_idx), qd, kd, vd, ad, bd, chunked=True)
    assert e.value.status == _abi.RS_ERR_UNSUPPORTED


@pytest.mark.parametrize("kind", ["fp32", "mixed"])
def test_chunked_prefill_repeats_bit_for_bit(kind):
    """The tensor-core products are issued by several warps at once; each issuing thread has
    accumulator columns of its own and the parts are summed in a fixed order, so the same call on
    the same state gives the same bits every time (KDA, 64 sequences, 32 heads, 64 tokens)."""
    B, Hk, Hv, L = 64, 32, 32, 64
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=L, per_channel=True, in_dtype="bf16", seed=91,
                            horizon=(2.0, 8192.0))
    qd, kd, vd, ad, bd = replay_inputs(w, L)
    if kind == "fp32":
        lay, start = rs.Layout("fp32", D, Hv, Hk), w.state0
    else:
        hi = gen.hi_rows(Hv, D, KHI, seed=91)
        lay = rs.Layout("mixed", D, Hv, Hk, k_hi=KHI, hi_rows=hi, quant="fused")
        start = orc.convert_pool_f32_to_mixed(w.state0, KHI, orc.row_map(hi, D), mode=1)
    runs = []
    for _ in range(3):
        pool = dev(start)
        o = torch.zeros((B, L, Hv, D), device="cuda")
        rs.prefill_update(lay, True, pool, dev(w.slot_idx), qd, kd, vd, ad, bd, o=o, chunked=True)
        torch.cuda.synchronize()
        runs.append((host(pool), host(o)))
    for pool_r, o_r in runs[1:]:
        assert np.array_equal(pool_r.view(np.uint8), runs[0][0].view(np.uint8))
        assert np.array_equal(o_r.view(np.uint32), runs[0][1].view(np.uint32))
