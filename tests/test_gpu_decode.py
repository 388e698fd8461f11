"""GPU parity of the FP32-state decode step (GDN and KDA) against the oracle.

Acceptance for the FP32 path: max relative error <= 1e-5 in S and o after 64
steps.  The library fixes the FP32 evaluation order of every result (see the
header), so the tests also require bit-for-bit equality with the oracle.
Sizes: the small GDN case in full; mid-size cases with every tile checked
(several CTAs per launch, groups with a ragged tail of items); and the full
B = 256 workloads, run whole on the GPU in the launch configuration the
benchmark times, checked on sampled sequences (all heads of each).
"""
import numpy as np
import pytest
import torch

import oracle as orc
import recurrent_state_gb300 as rs
from recurrent_state_gb300 import inputs as gen

from .gpu_util import dev, ensure_built, host, max_rel, same_bits, step_inputs, sub_batch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def gpu_run(w, layout, steps, out_dtype=torch.float32, status=None):
    pool = dev(w.state0)
    slots = dev(w.slot_idx)
    outs = []
    fn = rs.kda_decode_update if w.per_channel else rs.gdn_decode_update
    for t in range(steps):
        q, k, v, a, b = step_inputs(w, t)
        o = torch.empty((w.B, w.Hv, w.dv), dtype=out_dtype, device="cuda")
        fn(layout, pool, slots, q, k, v, a, b, o=o, status=status)
        outs.append(o)
    torch.cuda.synchronize()
    return host(pool), [host(o.float()) for o in outs]


def oracle_run(w, steps):
    pool = w.state0.copy()
    outs = []
    for t in range(steps):
        o, st = orc.decode_f32(pool, w.slot_idx, w.q[t], w.k[t], w.v[t], w.alpha[t], w.beta[t])
        assert st == 0
        outs.append(o)
    return pool, outs


def check(gpu, ref, tol=1e-5):
    g_pool, g_o = gpu
    r_pool, r_o = ref
    assert max_rel(g_pool, r_pool) <= tol
    for t, (a, b) in enumerate(zip(g_o, r_o)):
        assert max_rel(a, b) <= tol, t
        assert same_bits(a, b), f"o differs from the oracle at step {t}"
    assert same_bits(g_pool, r_pool), "state differs from the oracle"


def test_tiny_gdn_all_steps():
    """Batch 4, 4 heads, d = 64, 16 steps, fp32 q/k/v, fixed per-head decay."""
    w = gen.decode_workload(B=4, Hk=4, Hv=4, d=64, steps=16, per_channel=False, in_dtype="f32",
                            seed=0, tiny_gdn=True)
    lay = rs.Layout("fp32", 64, 4, 4)
    check(gpu_run(w, lay, 16), oracle_run(w, 16))


@pytest.mark.parametrize("per_channel,Hk,Hv,in_dtype,d", [
    (False, 4, 8, "bf16", 128),
    (False, 2, 8, "bf16", 128),    # four value heads per key head
    (True, 8, 8, "bf16", 128),
    (False, 2, 4, "f32", 64),
    (True, 4, 4, "f32", 64),
])
def test_every_tile_mid_size(per_channel, Hk, Hv, in_dtype, d):
    """B * Hv items spread over more groups than there are CTAs' worth, with
    a ragged last round, every tile checked for 4 steps."""
    B = 301
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=d, steps=4, per_channel=per_channel,
                            in_dtype=in_dtype, seed=11, n_slots=B + 37,
                            horizon=(2.0, 8192.0) if per_channel else (4.0, 4096.0))
    lay = rs.Layout("fp32", d, Hv, Hk)
    check(gpu_run(w, lay, 4), oracle_run(w, 4))


FULL = {
    "gdn": dict(B=256, Hk=16, Hv=32, d=128, per_channel=False, horizon=(4.0, 4096.0)),
    "kda": dict(B=256, Hk=32, Hv=32, d=128, per_channel=True, horizon=(2.0, 8192.0)),
}


@pytest.mark.parametrize("name", ["gdn", "kda"])
def test_full_size_64_steps_sampled(name):
    """The B = 256, d = 128 workloads for 64 consecutive steps on the GPU;
    the oracle replays 6 sampled sequences (all 32 heads each)."""
    c = FULL[name]
    w = gen.decode_workload(steps=64, in_dtype="bf16", seed=1, **c)
    lay = rs.Layout("fp32", 128, c["Hv"], c["Hk"])
    g_pool, g_o = gpu_run(w, lay, 64)
    bsel = np.array([0, 1, 77, 128, 200, 255])
    ws = sub_batch(w, bsel)
    r_pool, r_o = oracle_run(ws, 64)
    check((g_pool[w.slot_idx[bsel]], [o[bsel] for o in g_o]), (r_pool, r_o))


def test_bf16_output_is_rounded_fp32_readout():
    w = gen.decode_workload(B=16, Hk=4, Hv=8, d=128, steps=2, per_channel=False, in_dtype="bf16",
                            seed=5)
    lay = rs.Layout("fp32", 128, 8, 4)
    g32 = gpu_run(w, lay, 2)
    g16 = gpu_run(w, lay, 2, out_dtype=torch.bfloat16)
    for a, b in zip(g32[1], g16[1]):
        ref = torch.from_numpy(a).to(torch.bfloat16).float().numpy()
        assert same_bits(b, ref)
    assert same_bits(g32[0], g16[0])


def test_bad_slots_are_skipped_and_reported():
    w = gen.decode_workload(B=6, Hk=2, Hv=4, d=64, steps=1, per_channel=False, in_dtype="f32",
                            seed=6)
    w.slot_idx[2] = 99
    w.slot_idx[4] = -3
    lay = rs.Layout("fp32", 64, 4, 2)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = dev(w.state0)
    q, k, v, a, b = step_inputs(w, 0)
    o = torch.full((6, 4, 64), 7.0, device="cuda")
    rs.gdn_decode_update(lay, pool, dev(w.slot_idx), q, k, v, a, b, o=o, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    oh = host(o)
    assert np.all(oh[[2, 4]] == 7.0)
    ref_pool = w.state0.copy()
    ok = np.array([0, 1, 3, 5])
    ref_o, _ = orc.decode_f32(ref_pool, w.slot_idx[ok], w.q[0][ok], w.k[0][ok], w.v[0][ok],
                              w.alpha[0][ok], w.beta[0][ok])
    assert same_bits(oh[ok], ref_o)
    assert same_bits(host(pool), ref_pool)


def test_zero_batch_is_a_no_op():
    lay = rs.Layout("fp32", 128, 4, 4)
    pool = torch.zeros((2, 4, 128, 128), device="cuda")
    e = torch.empty(0, device="cuda")
    rs.gdn_decode_update(lay, pool, torch.empty(0, dtype=torch.int32, device="cuda"), e, e, e, e, e)
    torch.cuda.synchronize()
    assert int(pool.abs().sum().item()) == 0


def test_guard_regions_untouched():
    """Canary words around the pool and the output stay intact."""
    w = gen.decode_workload(B=8, Hk=4, Hv=8, d=128, steps=1, per_channel=True, in_dtype="bf16",
                            seed=8)
    lay = rs.Layout("fp32", 128, 8, 4)
    n = w.state0.size
    big = torch.full((n + 2 * 4096,), -123.0, device="cuda")
    pool = big[4096:4096 + n].view(w.state0.shape)
    pool.copy_(dev(w.state0))
    obuf = torch.full((8 * 8 * 128 + 2 * 64,), -321.0, device="cuda")
    o = obuf[64:64 + 8 * 8 * 128].view(8, 8, 128)
    q, k, v, a, b = step_inputs(w, 0)
    rs.kda_decode_update(lay, pool, dev(w.slot_idx), q, k, v, a, b, o=o)
    torch.cuda.synchronize()
    hb = host(big)
    assert np.all(hb[:4096] == -123.0) and np.all(hb[4096 + n:] == -123.0)
    ho = host(obuf)
    assert np.all(ho[:64] == -321.0) and np.all(ho[64 + 8 * 8 * 128:] == -321.0)
