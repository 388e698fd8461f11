"""Decode on the packed layouts writes exactly the tiles of the batch.

The mixed and DAMP-exact decode kernels store each new word from registers
straight to the pool, so these tests surround the pool and the readout with
canary bytes and leave some pool slots out of the batch: the canaries, and
every byte of the slots that are not stepped, must be unchanged, and the
stepped slots must equal the oracle's step.  Both requantisation modes, GDN
and KDA.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import recurrent_state_gb300 as rs
from recurrent_state_gb300 import inputs as gen

from .gpu_util import dev, ensure_built, host, same_bits, step_inputs

pytestmark = pytest.mark.gpu

D, KHI, G = 128, 16, 32
PAD = 4096          # canary bytes on each side (keeps the pool 16-byte aligned)
CANARY = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def guarded(nbytes, fill):
    big = torch.full((nbytes + 2 * PAD,), fill, dtype=torch.uint8, device="cuda")
    return big, big[PAD:PAD + nbytes]


@pytest.mark.parametrize("kind", ["mixed", "damp"])
@pytest.mark.parametrize("quant", ["ieee", "fused"])
@pytest.mark.parametrize("per_channel", [True, False])
def test_packed_decode_touches_only_the_batch(kind, quant, per_channel):
    B, Hk, Hv, n_slots = 5, 2, 4, 9
    hi = gen.hi_rows(Hv, D, KHI, seed=21)
    pi = orc.row_map(hi, D)
    cs = gen.value_scales(Hv, D, seed=21) if kind == "damp" else None
    f32 = rs.Layout("fp32", D, Hv, Hk)
    lay = rs.Layout(kind, D, Hv, Hk, k_hi=KHI, hi_rows=hi, value_scales=cs, quant=quant)
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=1, per_channel=per_channel, in_dtype="bf16",
                            seed=21, n_slots=n_slots, horizon=(2.0, 8192.0))
    assert len(set(w.slot_idx.tolist())) == B < n_slots

    nbytes = n_slots * Hv * lay.head_bytes
    big, flat = guarded(nbytes, CANARY)
    pool = flat.view(n_slots, Hv, lay.head_bytes)
    rs.state_convert(f32, dev(w.state0), lay, pool, torch.arange(n_slots, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    before = host(pool).copy()

    on = B * Hv * D * 4
    obig = torch.full((on + 2 * PAD,), CANARY, dtype=torch.uint8, device="cuda")
    o = obig[PAD:PAD + on].view(torch.float32).view(B, Hv, D)
    q, k, v, a, b = step_inputs(w, 0)
    fn = rs.kda_decode_update if per_channel else rs.gdn_decode_update
    fn(lay, pool, dev(w.slot_idx), q, k, v, a, b, o=o)
    torch.cuda.synchronize()

    hb = host(big)
    assert np.all(hb[:PAD] == CANARY) and np.all(hb[PAD + nbytes:] == CANARY)
    ho = host(obig)
    assert np.all(ho[:PAD] == CANARY) and np.all(ho[PAD + on:] == CANARY)

    after = host(pool)
    stepped = set(w.slot_idx.tolist())
    for s in range(n_slots):
        if s not in stepped:
            assert np.array_equal(after[s], before[s]), f"slot {s} outside the batch was written"

    ref = before.copy()
    mode = 1 if quant == "fused" else 0
    if kind == "mixed":
        o_r, st = orc.decode_mixed(ref, w.slot_idx, pi, KHI, D, D, w.q[0], w.k[0], w.v[0], w.alpha[0],
                                   w.beta[0], mode=mode)
    else:
        o_r, st = orc.decode_damp(ref, w.slot_idx, pi, cs, KHI, G, D, D, w.q[0], w.k[0], w.v[0],
                                  w.alpha[0], w.beta[0], mode=mode)
    assert st == 0
    assert same_bits(after, ref)
    assert same_bits(host(o), o_r)
