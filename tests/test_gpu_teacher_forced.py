"""Teacher-forced acceptance of the packed-state decode on the GPU against the
pages' quantiser (the oracle's IEEE mode), at full size.

The GPU runs 64 decode steps of the whole batch on its own packed state.
Before each step the packed tiles of a few sampled sequences (all heads) are
copied out; one oracle step of the pages' arithmetic (dequantise, decay,
update in FP32, requantise with the IEEE quotient: DAMP §3.1 Eq. 1-2, §3.2
Eq. 5-6, Appendix A.4; dasc Appendix E.1 Eq. 8) starts from those same bytes,
and the GPU's packed result is held to the acceptance rule (tests/acceptance):
INT8 codes equal except +-1 within 1e-6 max(1, |x/s|) of a rounding boundary
of the oracle's value, scales and FP16 rows within one ulp, o within 1e-3.

Cases: the fused arithmetic (RS_QUANT_FUSED) on the one-scale-per-row layout
and on the DAMP-exact layout (INT8 groups of 32, value scaling), KDA with
real per-channel decays (batch 256, 32 heads, d = 128, 16 FP16 rows); the
fused arithmetic on GDN with grouped key heads (16 key heads, 32 value
heads); and the IEEE default, which must meet the rule trivially.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import recurrent_state_gb300 as rs
from recurrent_state_gb300 import inputs as gen

from .acceptance import Tally, compare_tile, reference_step_mixed
from .gpu_util import dev, ensure_built, host, step_inputs

pytestmark = pytest.mark.gpu

D, KHI, G = 128, 16, 32
STEPS = 64
SAMPLE = np.array([0, 41, 128, 200, 255])


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


CASES = [
    # (layout, quant, per_channel, Hk, Hv)
    ("mixed", "fused", True, 32, 32),
    ("damp", "fused", True, 32, 32),
    ("mixed", "fused", False, 16, 32),
    ("mixed", "ieee", True, 32, 32),
]


@pytest.mark.parametrize("kind,quant,per_channel,Hk,Hv", CASES)
def test_teacher_forced_full_size(kind, quant, per_channel, Hk, Hv):
    B = 256
    seed = 7
    hi = gen.hi_rows(Hv, D, KHI, seed=seed)
    pi = orc.row_map(hi, D)
    cs = gen.value_scales(Hv, D, seed=seed) if kind == "damp" else None
    group = G if kind == "damp" else 0
    f32 = rs.Layout("fp32", D, Hv, Hk)
    lay = rs.Layout(kind, D, Hv, Hk, k_hi=KHI, hi_rows=hi, value_scales=cs, quant=quant)
    w = gen.decode_workload(B=B, Hk=Hk, Hv=Hv, d=D, steps=STEPS, per_channel=per_channel,
                            in_dtype="bf16", seed=seed,
                            horizon=(2.0, 8192.0) if per_channel else (4.0, 4096.0))
    pool = lay.empty_pool(B)
    rs.state_convert(f32, dev(w.state0), lay, pool, torch.arange(B, dtype=torch.int32, device="cuda"))
    slots = dev(w.slot_idx)
    sampled_slots = torch.from_numpy(w.slot_idx[SAMPLE].astype(np.int64)).cuda()
    fn = rs.kda_decode_update if per_channel else rs.gdn_decode_update
    tally = Tally()
    for t in range(STEPS):
        before = host(pool.index_select(0, sampled_slots))
        q, k, v, a, b = step_inputs(w, t)
        o = torch.empty((B, Hv, D), device="cuda")
        fn(lay, pool, slots, q, k, v, a, b, o=o)
        after = host(pool.index_select(0, sampled_slots))
        o_g = host(o)[SAMPLE]
        for i, bb in enumerate(SAMPLE):
            for h in range(Hv):
                g_ = h // (Hv // Hk)
                ref, x, o_r = reference_step_mixed(
                    before[i, h], pi[h], w.q[t, bb, g_], w.k[t, bb, g_], w.v[t, bb, h],
                    w.alpha[t, bb, h], w.beta[t, bb, h], D, D, KHI, group,
                    None if cs is None else cs[h])
                compare_tile(tally, after[i, h], ref, x, o_g[i, h], o_r, D, D, KHI, group,
                             where=f"step {t} seq {bb} head {h}")
        if len(tally.failures) > 20:
            break
    print(f"\n{kind}/{quant}/{'KDA' if per_channel else 'GDN'}: {tally.tiles} tiles, "
          f"{tally.codes} codes, {tally.code_flips} boundary flips "
          f"(worst {tally.worst_flip_distance:.3g}), scales moved {tally.scale_moved} "
          f"(max {tally.scale_ulp_max} ulp), FP16 max {tally.fp16_ulp_max} ulp, "
          f"o max {tally.o_rel_max:.3g}")
    assert tally.ok(), tally.failures[:10]
    assert tally.tiles == STEPS * len(SAMPLE) * Hv
    # both modes run the pages' FP32 step: scales, FP16 rows and o agree
    # exactly; only a fused code at a rounding boundary may differ
    assert tally.scale_moved == 0 and tally.fp16_ulp_max == 0 and tally.o_rel_max == 0.0
    if quant == "ieee":  # the library's default is the pages' arithmetic itself
        assert tally.code_flips == 0
