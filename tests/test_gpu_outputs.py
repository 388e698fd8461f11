"""GPU parity of the bf16 readout on every path that writes o.

The readout is computed in FP32 and rounded once to bf16 (nearest, ties to
even) when stored; the state is unaffected.  Each case compares o with the
oracle's FP32 readout rounded by torch's float -> bf16 conversion, and the
pool with the oracle's, bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import recurrent_state_gb300 as rs
from recurrent_state_gb300 import inputs as gen

from .gpu_util import dev, ensure_built, host, replay_inputs, same_bits, step_inputs

pytestmark = pytest.mark.gpu

D, KHI, G = 128, 16, 32


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def bf16_bits(o_f32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(o_f32)).to(torch.bfloat16).view(torch.int16).numpy()


def gpu_bf16_bits(o: torch.Tensor) -> np.ndarray:
    return o.view(torch.int16).cpu().numpy()


def packed(kind, Hv, Hk, seed, quant):
    hi = gen.hi_rows(Hv, D, KHI, seed=seed)
    cs = gen.value_scales(Hv, D, seed=seed) if kind == "damp" else None
    lay = rs.Layout(kind, D, Hv, Hk, k_hi=KHI, hi_rows=hi, value_scales=cs, quant=quant)
    return lay, orc.row_map(hi, D), cs


def to_packed(lay, state0, Hv, Hk):
    f32 = rs.Layout("fp32", D, Hv, Hk)
    dst = lay.empty_pool(state0.shape[0])
    rs.state_convert(f32, dev(state0), lay, dst, torch.arange(state0.shape[0], dtype=torch.int32, device="cuda"))
    return dst


@pytest.mark.parametrize("kind,quant", [("mixed", "ieee"), ("mixed", "fused"), ("damp", "ieee"), ("damp", "fused")])
def test_decode_bf16_readout(kind, quant):
    B, Hk, Hv = 21, 4, 8
    seed = 70
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=2, per_channel=True, in_dtype="bf16", seed=seed,
                            horizon=(2.0, 8192.0))
    lay, pi, cs = packed(kind, Hv, Hk, seed, quant)
    mode = 1 if quant == "fused" else 0
    pool = to_packed(lay, w.state0, Hv, Hk)
    if kind == "damp":
        ref = orc.convert_pool_f32_to_damp(w.state0, KHI, G, pi, cs, mode=mode)
    else:
        ref = orc.convert_pool_f32_to_mixed(w.state0, KHI, pi, mode=mode)
    for t in range(w.steps):
        q, k, v, a, b = step_inputs(w, t)
        o = torch.empty((B, Hv, D), dtype=torch.bfloat16, device="cuda")
        rs.kda_decode_update(lay, pool, dev(w.slot_idx), q, k, v, a, b, o=o)
        if kind == "damp":
            o_r, _ = orc.decode_damp(ref, w.slot_idx, pi, cs, KHI, G, D, D, w.q[t], w.k[t], w.v[t],
                                     w.alpha[t], w.beta[t], mode=mode)
        else:
            o_r, _ = orc.decode_mixed(ref, w.slot_idx, pi, KHI, D, D, w.q[t], w.k[t], w.v[t],
                                      w.alpha[t], w.beta[t], mode=mode)
        torch.cuda.synchronize()
        assert np.array_equal(gpu_bf16_bits(o), bf16_bits(o_r)), t
        assert same_bits(host(pool), ref), t


@pytest.mark.parametrize("path", ["replay_mixed", "prefill_fp32", "prefill_mixed", "prefill_damp"])
def test_multi_token_bf16_readout(path):
    B, Hk, Hv, T = 17, 2, 4, 8 if path == "replay_mixed" else 13
    seed = 71
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=T, per_channel=False, in_dtype="bf16", seed=seed,
                            horizon=(2.0, 8192.0))
    n_tok = gen.rng(seed).integers(0, T + 1, B).astype(np.int32)
    qd, kd, vd, ad, bd = replay_inputs(w, T)
    q, k, v, a, b = gen.replay_view(w, T)
    o = torch.zeros((B, T, Hv, D), dtype=torch.bfloat16, device="cuda")
    o_r = np.zeros((B, T, Hv, D), np.float32)
    if path == "prefill_fp32":
        lay = rs.Layout("fp32", D, Hv, Hk)
        pool = dev(w.state0)
        ref = w.state0.copy()
        rs.prefill_update(lay, False, pool, dev(w.slot_idx), qd, kd, vd, ad, bd, n_tokens=dev(n_tok), o=o)
        orc.replay_f32(ref, w.slot_idx, n_tok, q, k, v, a, b, o=o_r)
    elif path == "prefill_damp":
        lay, pi, cs = packed("damp", Hv, Hk, seed, "fused")
        pool = to_packed(lay, w.state0, Hv, Hk)
        ref = orc.convert_pool_f32_to_damp(w.state0, KHI, G, pi, cs, mode=1)
        rs.prefill_update(lay, False, pool, dev(w.slot_idx), qd, kd, vd, ad, bd, n_tokens=dev(n_tok), o=o)
        orc.replay_damp(ref, w.slot_idx, n_tok, pi, cs, KHI, G, D, D, q, k, v, a, b, o=o_r, mode=1)
    else:
        lay, pi, _ = packed("mixed", Hv, Hk, seed, "fused")
        pool = to_packed(lay, w.state0, Hv, Hk)
        ref = orc.convert_pool_f32_to_mixed(w.state0, KHI, pi, mode=1)
        if path == "replay_mixed":
            rs.spec_replay_update(lay, False, pool, dev(w.slot_idx), dev(n_tok), qd, kd, vd, ad, bd, o=o)
        else:
            rs.prefill_update(lay, False, pool, dev(w.slot_idx), qd, kd, vd, ad, bd, n_tokens=dev(n_tok), o=o)
        orc.replay_mixed(ref, w.slot_idx, n_tok, pi, KHI, D, D, q, k, v, a, b, o=o_r, mode=1)
    torch.cuda.synchronize()
    assert np.array_equal(gpu_bf16_bits(o), bf16_bits(o_r))
    assert same_bits(host(pool), ref)
