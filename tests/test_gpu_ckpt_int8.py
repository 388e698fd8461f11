"""GPU parity of the dasc INT8 state checkpoint (dasc Appendix E.1 Eq. 8) and
of whole-head checkpoints of mixed FP16/INT8 pools (bit-exact).

INT8: every code byte and every scale of the checkpoint, and every FP32 value
of the restored pool, equal the oracle's -- head and key-channel units, dv =
128 and 64, rows with NaN or infinity (literal-division path), edge plans and
bad slot indices, and the full workload (36 layers x 64 checkpoints) on
sampled checkpoints.  Mixed heads: every byte of checkpoint and pool.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import recurrent_state_gb300 as rs
from recurrent_state_gb300 import inputs as gen

from .gpu_util import dev, ensure_built, host, same_bits, same_bits_nan

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def unit_name(unit):
    return "head" if unit == 0 else "channel"


@pytest.mark.parametrize("unit,p,d", [(0, 0.5, 128), (1, 0.45, 128), (1, 0.45, 64), (0, 0.3, 64)])
def test_int8_pack_restore_small_every_byte(unit, p, d):
    L, slots, Hv, n = 4, 7, 4, 5
    pool_np = gen.random_pool((L, slots, Hv, d, d), seed=10 + unit + d)
    pool_np[1, 2, 1, 5] *= 1e5                 # an outlier row
    pool_np[2, 3, 0, 7, 9] = np.nan            # a NaN row
    pool_np[3, 4, 2, 1, 3] = -np.inf           # an infinite row
    pool_np[0, 1, 3, 2] = 0.0                  # an all-zero row (scale floor)
    n_units = Hv if unit == 0 else Hv * d
    keep = gen.keep_mask(L, n_units, p, seed=20 + unit + d)
    keep[2, (0 if unit == 0 else 7)] = 1       # the special rows are retained
    keep[3, (2 if unit == 0 else 2 * d + 1)] = 1
    keep[1, (1 if unit == 0 else d + 5)] = 1
    keep[0, (3 if unit == 0 else 3 * d + 2)] = 1
    src = np.array([2, 3, 4, 1, 0], np.int32)
    dst = np.array([1, 4, 0, 2, 3], np.int32)
    lay = rs.Layout("fp32", d, Hv, 1)
    plan = rs.Plan(lay, keep, unit_name(unit)).upload()
    cb, sb = orc.ckpt_int8_layout(int(keep.sum()), unit, d, d)
    assert (plan.int8_codes_bytes, plan.int8_slot_bytes) == (cb, sb)
    ckpt = torch.full((n, sb), 0xCD, dtype=torch.uint8, device="cuda")
    pool = dev(pool_np)
    rs.ckpt_pack_int8(plan, pool, dev(src), dev(dst), ckpt)
    ref = np.full((n, sb), 0xCD, np.uint8)
    assert orc.ckpt_pack_int8(keep, unit, pool_np, src, dst, ref) == 0
    torch.cuda.synchronize()
    assert same_bits(host(ckpt), ref)
    out = torch.full_like(pool, float("nan"))
    rdst = np.array([6, 0, 3, 1, 5], np.int32)
    rs.ckpt_restore_int8(plan, ckpt, dev(dst), out, dev(rdst))
    out_ref = np.full_like(pool_np, np.nan)
    assert orc.ckpt_restore_int8(keep, unit, ref, dst, out_ref, rdst) == 0
    torch.cuda.synchronize()
    # the row with an infinite absmax restores as code * inf: +-inf, and NaN for code 0
    assert same_bits_nan(host(out), out_ref)
    assert np.isnan(out_ref[:, rdst]).sum() > 0


@pytest.mark.parametrize("unit", [0, 1])
def test_int8_all_and_none_kept(unit):
    L, slots, Hv, d = 3, 2, 2, 128
    pool_np = gen.random_pool((L, slots, Hv, d, d), seed=40 + unit)
    n_units = Hv if unit == 0 else Hv * d
    lay = rs.Layout("fp32", d, Hv, 1)
    one = torch.tensor([1], dtype=torch.int32, device="cuda")
    zero = torch.tensor([0], dtype=torch.int32, device="cuda")
    keep = np.ones((L, n_units), np.uint8)
    plan = rs.Plan(lay, keep, unit_name(unit)).upload()
    ckpt = torch.zeros((1, plan.int8_slot_bytes), dtype=torch.uint8, device="cuda")
    pool = dev(pool_np)
    rs.ckpt_pack_int8(plan, pool, one, zero, ckpt)
    ref = np.zeros((1, plan.int8_slot_bytes), np.uint8)
    orc.ckpt_pack_int8(keep, unit, pool_np, np.array([1], np.int32), np.array([0], np.int32), ref)
    torch.cuda.synchronize()
    assert same_bits(host(ckpt), ref)
    rs.ckpt_restore_int8(plan, ckpt, zero, pool, zero)
    back = pool_np.copy()
    orc.ckpt_restore_int8(keep, unit, ref, np.array([0], np.int32), back, np.array([0], np.int32))
    torch.cuda.synchronize()
    assert same_bits(host(pool), back)
    none = rs.Plan(lay, np.zeros((L, n_units), np.uint8), unit_name(unit)).upload()
    assert none.int8_slot_bytes == 0
    empty = torch.empty((1, 0), dtype=torch.uint8, device="cuda")
    rs.ckpt_restore_int8(none, empty, zero, pool, one)
    torch.cuda.synchronize()
    assert np.all(host(pool)[:, 1].view(np.uint32) == 0)


def test_int8_bad_slots_reported_and_skipped():
    L, slots, Hv, d = 2, 3, 2, 64
    pool_np = gen.random_pool((L, slots, Hv, d, d), seed=50)
    lay = rs.Layout("fp32", d, Hv, 1)
    plan = rs.Plan(lay, np.ones((L, Hv), np.uint8), "head").upload()
    ckpt = torch.full((2, plan.int8_slot_bytes), 7, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = dev(pool_np)
    rs.ckpt_pack_int8(plan, pool, dev(np.array([0, 9], np.int32)), dev(np.array([5, 1], np.int32)),
                      ckpt, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == (1 | 4)
    assert np.all(host(ckpt) == 7)
    status.zero_()
    rs.ckpt_restore_int8(plan, ckpt, dev(np.array([3], np.int32)), pool, dev(np.array([0], np.int32)),
                         status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 4
    assert same_bits(host(pool), pool_np)


@pytest.mark.parametrize("unit,p", [(0, 0.5), (1, 0.45)])
def test_int8_full_workload_sampled(unit, p):
    """36 layers, 64 checkpoints from 64 pool slots in a seeded permuted
    order, 32 heads of 128 x 128; checkpoints 0, 17 and 63 against the
    oracle, every byte, and their restores."""
    L, Hv, d, n = 36, 32, 128, 64
    g = torch.Generator(device="cuda").manual_seed(5 + unit)
    pool = torch.randn((L, n, Hv, d, d), device="cuda", generator=g) * 0.1
    n_units = Hv if unit == 0 else Hv * d
    keep = gen.keep_mask(L, n_units, p, seed=60 + unit)
    src, dst = gen.ckpt_slots(n, n, seed=70 + unit)
    lay = rs.Layout("fp32", d, Hv, 1)
    plan = rs.Plan(lay, keep, unit_name(unit)).upload()
    ckpt = plan.empty_int8_ckpt_pool(n)
    rs.ckpt_pack_int8(plan, pool, dev(src), dev(dst), ckpt)
    out = torch.full_like(pool, float("nan"))
    rs.ckpt_restore_int8(plan, ckpt, dev(dst), out, dev(src))
    torch.cuda.synchronize()
    used = plan.int8_codes_bytes + 4 * (plan.int8_codes_bytes // d)  # codes and scales, no padding
    for i in (0, 17, 63):
        pool_i = np.ascontiguousarray(host(pool[:, src[i]:src[i] + 1]))
        ref = np.zeros((1, plan.int8_slot_bytes), np.uint8)
        assert orc.ckpt_pack_int8(keep, unit, pool_i, np.array([0], np.int32),
                                  np.array([0], np.int32), ref) == 0
        assert same_bits(host(ckpt[dst[i]])[:used], ref[0, :used])
        back = np.zeros_like(pool_i)
        assert orc.ckpt_restore_int8(keep, unit, ref, np.array([0], np.int32), back,
                                     np.array([0], np.int32)) == 0
        assert same_bits(host(out[:, src[i]:src[i] + 1]), back)


def test_mixed_heads_pack_restore_every_byte():
    """Whole mixed heads (18,880 B: 36 chunks of 512 B and one of 448 B) in
    and out of checkpoints, against the oracle."""
    L, slots, Hv, d, khi, n = 3, 5, 4, 128, 16, 4
    hi = gen.hi_rows(Hv, d, khi, seed=3)
    f32 = rs.Layout("fp32", d, Hv, Hv)
    mix = rs.Layout("mixed", d, Hv, Hv, k_hi=khi, hi_rows=hi)
    pool = torch.empty((L, slots, Hv, mix.head_bytes), dtype=torch.uint8, device="cuda")
    allslots = torch.arange(slots, dtype=torch.int32, device="cuda")
    for l in range(L):
        src32 = dev(gen.random_pool((slots, Hv, d, d), seed=80 + l))
        rs.state_convert(f32, src32, mix, pool[l], allslots)
    keep = gen.keep_mask(L, Hv, 0.5, seed=4)
    plan = rs.Plan(mix, keep, "head").upload()
    assert plan.unit_bytes == 18880
    src = np.array([4, 0, 2, 1], np.int32)
    dst = np.array([2, 3, 0, 1], np.int32)
    ckpt = torch.full((n, plan.ckpt_slot_bytes), 0xEE, dtype=torch.uint8, device="cuda")
    rs.ckpt_pack(plan, pool, dev(src), dev(dst), ckpt)
    torch.cuda.synchronize()
    pool_np = host(pool).copy()
    ref = np.full((n, plan.ckpt_slot_bytes), 0xEE, np.uint8)
    assert orc.ckpt_pack_heads(keep, pool_np, src, dst, ref) == 0
    assert same_bits(host(ckpt), ref)
    out = torch.full_like(pool, 0x5A)
    rdst = np.array([3, 1, 4, 0], np.int32)
    rs.ckpt_restore(plan, ckpt, dev(dst), out, dev(rdst))
    out_ref = np.full_like(pool_np, 0x5A)
    assert orc.ckpt_restore_heads(keep, ref, dst, out_ref, rdst) == 0
    torch.cuda.synchronize()
    assert same_bits(host(out), out_ref)
