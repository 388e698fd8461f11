"""GPU parity with IEEE half (fp16) q, k and v.

fp16 inputs widen to FP32 exactly, so every path must give the same bits as
the oracle fed the widened values: decode on the FP32 layout (dk = 64 and
128, GDN and KDA), on the mixed and DAMP-exact layouts in both
requantisation modes, speculative replay and prefill chunks.  The readout is
FP32.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import recurrent_state_gb300 as rs
from recurrent_state_gb300 import inputs as gen

from .gpu_util import dev, ensure_built, host, replay_inputs, same_bits, step_inputs

pytestmark = pytest.mark.gpu

KHI, G = 16, 32


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def to_packed(lay, state0, D, Hv, Hk):
    f32 = rs.Layout("fp32", D, Hv, Hk)
    dst = lay.empty_pool(state0.shape[0])
    rs.state_convert(f32, dev(state0), lay, dst, torch.arange(state0.shape[0], dtype=torch.int32, device="cuda"))
    return dst


@pytest.mark.parametrize("D,per_channel", [(64, False), (128, False), (128, True)])
def test_fp32_layout_decode_f16_inputs(D, per_channel):
    B, Hk, Hv, steps = 13, 2, 4, 3
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=steps, per_channel=per_channel, in_dtype="f16",
                            seed=60 + D)
    lay = rs.Layout("fp32", D, Hv, Hk)
    pool, ref = dev(w.state0), w.state0.copy()
    fn = rs.kda_decode_update if per_channel else rs.gdn_decode_update
    for t in range(steps):
        q, k, v, a, b = step_inputs(w, t)
        assert q.dtype == torch.float16
        o = torch.empty((B, Hv, D), device="cuda")
        fn(lay, pool, dev(w.slot_idx), q, k, v, a, b, o=o)
        o_r, st = orc.decode_f32(ref, w.slot_idx, w.q[t], w.k[t], w.v[t], w.alpha[t], w.beta[t])
        assert st == 0
        torch.cuda.synchronize()
        assert same_bits(host(o), o_r), t
    assert same_bits(host(pool), ref)


@pytest.mark.parametrize("kind,quant", [("mixed", "ieee"), ("mixed", "fused"), ("damp", "ieee"), ("damp", "fused")])
def test_packed_layout_decode_f16_inputs(kind, quant):
    B, Hk, Hv, D, steps = 11, 2, 4, 128, 2
    seed = 62
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=steps, per_channel=True, in_dtype="f16", seed=seed,
                            horizon=(2.0, 8192.0))
    hi = gen.hi_rows(Hv, D, KHI, seed=seed)
    pi = orc.row_map(hi, D)
    cs = gen.value_scales(Hv, D, seed=seed) if kind == "damp" else None
    lay = rs.Layout(kind, D, Hv, Hk, k_hi=KHI, hi_rows=hi, value_scales=cs, quant=quant)
    mode = 1 if quant == "fused" else 0
    pool = to_packed(lay, w.state0, D, Hv, Hk)
    if kind == "damp":
        ref = orc.convert_pool_f32_to_damp(w.state0, KHI, G, pi, cs, mode=mode)
    else:
        ref = orc.convert_pool_f32_to_mixed(w.state0, KHI, pi, mode=mode)
    for t in range(steps):
        q, k, v, a, b = step_inputs(w, t)
        o = torch.empty((B, Hv, D), device="cuda")
        rs.kda_decode_update(lay, pool, dev(w.slot_idx), q, k, v, a, b, o=o)
        if kind == "damp":
            o_r, _ = orc.decode_damp(ref, w.slot_idx, pi, cs, KHI, G, D, D, w.q[t], w.k[t], w.v[t],
                                     w.alpha[t], w.beta[t], mode=mode)
        else:
            o_r, _ = orc.decode_mixed(ref, w.slot_idx, pi, KHI, D, D, w.q[t], w.k[t], w.v[t],
                                      w.alpha[t], w.beta[t], mode=mode)
        torch.cuda.synchronize()
        assert same_bits(host(o), o_r), t
        assert same_bits(host(pool), ref), t


@pytest.mark.parametrize("path", ["replay_fp32", "replay_mixed", "prefill_fp32", "prefill_mixed", "prefill_damp"])
def test_multi_token_f16_inputs(path):
    B, Hk, Hv, D = 9, 2, 4, 128
    T = 8 if path.startswith("replay") else 11
    seed = 63
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=T, per_channel=True, in_dtype="f16", seed=seed,
                            horizon=(2.0, 8192.0))
    n_tok = gen.rng(seed).integers(0 if path.startswith("prefill") else 1, T + 1, B).astype(np.int32)
    qd, kd, vd, ad, bd = replay_inputs(w, T)
    q, k, v, a, b = gen.replay_view(w, T)
    o = torch.zeros((B, T, Hv, D), device="cuda")
    o_r = np.zeros((B, T, Hv, D), np.float32)
    hi = gen.hi_rows(Hv, D, KHI, seed=seed)
    pi = orc.row_map(hi, D)
    if path.endswith("fp32"):
        lay = rs.Layout("fp32", D, Hv, Hk)
        pool, ref = dev(w.state0), w.state0.copy()
        orc.replay_f32(ref, w.slot_idx, n_tok, q, k, v, a, b, o=o_r)
    elif path.endswith("damp"):
        cs = gen.value_scales(Hv, D, seed=seed)
        lay = rs.Layout("damp", D, Hv, Hk, k_hi=KHI, hi_rows=hi, value_scales=cs, quant="fused")
        pool = to_packed(lay, w.state0, D, Hv, Hk)
        ref = orc.convert_pool_f32_to_damp(w.state0, KHI, G, pi, cs, mode=1)
        orc.replay_damp(ref, w.slot_idx, n_tok, pi, cs, KHI, G, D, D, q, k, v, a, b, o=o_r, mode=1)
    else:
        lay = rs.Layout("mixed", D, Hv, Hk, k_hi=KHI, hi_rows=hi)
        pool = to_packed(lay, w.state0, D, Hv, Hk)
        ref = orc.convert_pool_f32_to_mixed(w.state0, KHI, pi)
        orc.replay_mixed(ref, w.slot_idx, n_tok, pi, KHI, D, D, q, k, v, a, b, o=o_r)
    if path.startswith("replay"):
        rs.spec_replay_update(lay, True, pool, dev(w.slot_idx), dev(n_tok), qd, kd, vd, ad, bd, o=o)
    else:
        rs.prefill_update(lay, True, pool, dev(w.slot_idx), qd, kd, vd, ad, bd, n_tokens=dev(n_tok), o=o)
    torch.cuda.synchronize()
    assert same_bits(host(o), o_r)
    assert same_bits(host(pool), ref)
