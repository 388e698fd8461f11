"""The hot-path calls inside CUDA graphs.

A serving engine captures its decode step once and replays it, so the
calls must capture: no synchronisation, no allocation, no host-side state
that a replay would miss.  Each case captures a few calls into a CUDA graph
on a side stream, replays the graph, and compares the pool and the outputs
with the same calls made directly, bit for bit.
"""
import numpy as np
import pytest
import torch

import recurrent_state_gb300 as rs
from recurrent_state_gb300 import inputs as gen

from .gpu_util import dev, ensure_built, host, replay_inputs, same_bits, step_inputs

pytestmark = pytest.mark.gpu

D, KHI = 128, 16


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def layouts(Hv, Hk, seed):
    hi = gen.hi_rows(Hv, D, KHI, seed=seed)
    return (rs.Layout("fp32", D, Hv, Hk),
            rs.Layout("mixed", D, Hv, Hk, k_hi=KHI, hi_rows=hi, quant="fused"))


def packed(f32, lay, state0):
    dst = lay.empty_pool(state0.shape[0])
    rs.state_convert(f32, dev(state0), lay, dst, torch.arange(state0.shape[0], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    return dst


def run_twice(calls, make_state):
    """Direct calls on one copy of the state; a captured graph replayed on
    another; returns both final states and output lists."""
    s_direct, outs_direct = make_state()
    calls(s_direct, outs_direct)
    torch.cuda.synchronize()
    s_graph, outs_graph = make_state()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        # warm-up outside capture on copies: kernel attributes are set on the first launch
        s_warm, outs_warm = make_state()
        calls(s_warm, outs_warm)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        calls(s_graph, outs_graph)
    g.replay()
    torch.cuda.synchronize()
    return (s_direct, outs_direct), (s_graph, outs_graph)


@pytest.mark.parametrize("kind", ["fp32", "mixed_fused"])
def test_decode_steps_in_a_graph(kind):
    B, Hk, Hv, steps = 19, 4, 8, 4
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=steps, per_channel=True, in_dtype="bf16", seed=80)
    f32, mix = layouts(Hv, Hk, 80)
    lay = f32 if kind == "fp32" else mix
    base = dev(w.state0) if kind == "fp32" else packed(f32, mix, w.state0)
    inputs = [step_inputs(w, t) for t in range(steps)]
    slots = dev(w.slot_idx)

    def make_state():
        return base.clone(), [torch.empty((B, Hv, D), device="cuda") for _ in range(steps)]

    def calls(pool, outs):
        for t in range(steps):
            q, k, v, a, b = inputs[t]
            rs.kda_decode_update(lay, pool, slots, q, k, v, a, b, o=outs[t])

    (sd, od), (sg, og) = run_twice(calls, make_state)
    assert same_bits(host(sd), host(sg))
    for x, y in zip(od, og):
        assert same_bits(host(x), host(y))


@pytest.mark.parametrize("path", ["replay", "prefill", "prefill_chunked", "prefill_chunked_fp32"])
def test_multi_token_calls_in_a_graph(path):
    B, Hk, Hv, T = 13, 2, 4, 8
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=T, per_channel=False, in_dtype="bf16", seed=81)
    f32, mix = layouts(Hv, Hk, 81)
    base = dev(w.state0) if path == "prefill_chunked_fp32" else packed(f32, mix, w.state0)
    qd, kd, vd, ad, bd = replay_inputs(w, T)
    n = dev(gen.n_accept(B, T, seed=81))
    slots = dev(w.slot_idx)

    def make_state():
        return base.clone(), [torch.zeros((B, T, Hv, D), device="cuda")]

    def calls(pool, outs):
        if path == "replay":
            rs.spec_replay_update(mix, False, pool, slots, n, qd, kd, vd, ad, bd, o=outs[0])
        elif path == "prefill":
            rs.prefill_update(mix, False, pool, slots, qd, kd, vd, ad, bd, n_tokens=n, o=outs[0])
        else:  # the chunk-parallel form: tensor maps encoded on the host at each call, passed by value
            rs.prefill_update(f32 if path == "prefill_chunked_fp32" else mix, False, pool, slots, qd, kd, vd, ad,
                              bd, n_tokens=n, o=outs[0], chunked=True)

    (sd, od), (sg, og) = run_twice(calls, make_state)
    assert same_bits(host(sd), host(sg))
    assert same_bits(host(od[0]), host(og[0]))


def test_checkpoint_pack_restore_in_a_graph():
    L, slots_n, Hv, d = 4, 3, 4, 64
    pool_np = gen.random_pool((L, slots_n, Hv, d, d), seed=82)
    keep = gen.keep_mask(L, Hv * d, 0.45, seed=82)
    lay = rs.Layout("fp32", d, Hv, 1)
    plan = rs.Plan(lay, keep, "channel").upload()
    src = torch.tensor([2, 0], dtype=torch.int32, device="cuda")
    dst = torch.tensor([1, 0], dtype=torch.int32, device="cuda")
    base = dev(pool_np)

    def make_state():
        return base.clone(), [plan.empty_ckpt_pool(2, device="cuda").zero_(), torch.zeros_like(base)]

    def calls(pool, outs):
        rs.ckpt_pack(plan, pool, src, dst, outs[0])
        rs.ckpt_restore(plan, outs[0], dst, outs[1], src)

    (sd, od), (sg, og) = run_twice(calls, make_state)
    assert same_bits(host(od[0]), host(og[0]))
    assert same_bits(host(od[1]), host(og[1]))
