"""GPU parity of dasc checkpoint pack and restore (bit-exact).

A small plan with every byte compared against the oracle, the edge plans
(everything kept, nothing kept), bad slot indices, and the full workload:
36 layers, 64 checkpoints, GDN 32 heads of 128 x 128 keeping a seeded 50% of
heads, KDA 32 heads keeping a seeded 45% of key channels, source slots in a
seeded permuted order; sampled checkpoints compared with the oracle.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import recurrent_state_gb300 as rs
from recurrent_state_gb300 import inputs as gen

from .gpu_util import dev, ensure_built, host, same_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def unit_name(unit):
    return "head" if unit == 0 else "channel"


@pytest.mark.parametrize("unit,p,d", [(0, 0.5, 128), (1, 0.45, 128), (1, 0.45, 64), (0, 0.3, 64)])
def test_pack_restore_small_every_byte(unit, p, d):
    L, slots, Hv, n = 5, 7, 4, 5
    pool_np = gen.random_pool((L, slots, Hv, d, d), seed=unit + d)
    n_units = Hv if unit == 0 else Hv * d
    keep = gen.keep_mask(L, n_units, p, seed=unit + d)
    src, dst = gen.ckpt_slots(slots, n, seed=unit + d)
    lay = rs.Layout("fp32", d, Hv, 1)
    plan = rs.Plan(lay, keep, unit_name(unit)).upload()
    ckpt = torch.full((n, plan.ckpt_slot_bytes), 0xCD, dtype=torch.uint8, device="cuda")
    pool = dev(pool_np)
    rs.ckpt_pack(plan, pool, dev(src), dev(dst), ckpt)
    ref = np.full((n, plan.ckpt_slot_bytes), 0xCD, np.uint8)
    assert orc.ckpt_pack(keep, unit, pool_np, src, dst, ref) == 0
    torch.cuda.synchronize()
    assert same_bits(host(ckpt), ref)
    # restore into other slots of a pool pre-filled with NaN
    out = torch.full_like(pool, float("nan"))
    rdst = np.array([6, 0, 3, 1, 5], np.int32)
    rs.ckpt_restore(plan, ckpt, dev(dst), out, dev(rdst))
    out_ref = np.full_like(pool_np, np.nan)
    assert orc.ckpt_restore(keep, unit, ref, dst, out_ref, rdst) == 0
    torch.cuda.synchronize()
    assert same_bits(host(out), out_ref)


@pytest.mark.parametrize("unit", [0, 1])
def test_all_and_none_kept(unit):
    L, slots, Hv, d = 3, 2, 2, 64
    pool_np = gen.random_pool((L, slots, Hv, d, d), seed=40 + unit)
    n_units = Hv if unit == 0 else Hv * d
    lay = rs.Layout("fp32", d, Hv, 1)
    plan = rs.Plan(lay, np.ones((L, n_units), np.uint8), unit_name(unit)).upload()
    ckpt = plan.empty_ckpt_pool(1)
    pool = dev(pool_np)
    one = torch.tensor([1], dtype=torch.int32, device="cuda")
    zero = torch.tensor([0], dtype=torch.int32, device="cuda")
    rs.ckpt_pack(plan, pool, one, zero, ckpt)
    torch.cuda.synchronize()
    assert same_bits(host(ckpt)[0], pool_np[:, 1].reshape(-1).view(np.uint8))
    rs.ckpt_restore(plan, ckpt, zero, pool, zero)
    torch.cuda.synchronize()
    assert same_bits(host(pool)[:, 0], pool_np[:, 1])
    none = rs.Plan(lay, np.zeros((L, n_units), np.uint8), unit_name(unit)).upload()
    assert none.ckpt_slot_bytes == 0
    empty = torch.empty((1, 0), dtype=torch.uint8, device="cuda")
    rs.ckpt_restore(none, empty, zero, pool, one)
    torch.cuda.synchronize()
    assert np.all(host(pool)[:, 1].view(np.uint32) == 0)


def test_bad_slots_reported_and_skipped():
    L, slots, Hv, d = 2, 3, 2, 64
    pool_np = gen.random_pool((L, slots, Hv, d, d), seed=50)
    lay = rs.Layout("fp32", d, Hv, 1)
    plan = rs.Plan(lay, np.ones((L, Hv), np.uint8), "head").upload()
    ckpt = torch.zeros((2, plan.ckpt_slot_bytes), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rs.ckpt_pack(plan, dev(pool_np), dev(np.array([7, 0], np.int32)),
                 dev(np.array([0, 5], np.int32)), ckpt, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == (1 | 4)
    assert int(ckpt.sum().item()) == 0


@pytest.mark.parametrize("unit,p", [(0, 0.5), (1, 0.45)])
def test_full_workload_sampled(unit, p):
    """36 layers x 64 checkpoints; 64 pool slots (4.5 GiB of FP32 state)."""
    L, slots, Hv, d, n = 36, 64, 32, 128, 64
    n_units = Hv if unit == 0 else Hv * d
    keep = gen.keep_mask(L, n_units, p, seed=unit)
    src, dst = gen.ckpt_slots(slots, n, seed=unit)
    lay = rs.Layout("fp32", d, Hv, 1)
    plan = rs.Plan(lay, keep, unit_name(unit)).upload()
    g = torch.Generator(device="cuda").manual_seed(unit)
    pool = torch.randn((L, slots, Hv, d, d), device="cuda", generator=g)
    ckpt = plan.empty_ckpt_pool(n)
    rs.ckpt_pack(plan, pool, dev(src), dev(dst), ckpt)
    out = torch.full_like(pool, float("nan"))
    rs.ckpt_restore(plan, ckpt, dev(dst), out, dev(src))
    torch.cuda.synchronize()
    # the checkpoint of sampled pairs, and the restored slots, against the oracle
    for i in (0, 17, 63):
        pool_i = np.ascontiguousarray(host(pool[:, src[i]:src[i] + 1]))
        ref = np.zeros((1, plan.ckpt_slot_bytes), np.uint8)
        assert orc.ckpt_pack(keep, unit, pool_i, np.array([0], np.int32),
                             np.array([0], np.int32), ref) == 0
        assert same_bits(host(ckpt[dst[i]]), ref[0])
        out_ref = np.zeros_like(pool_i)
        assert orc.ckpt_restore(keep, unit, ref, np.array([0], np.int32), out_ref,
                                np.array([0], np.int32)) == 0
        assert same_bits(host(out[:, src[i]:src[i] + 1]), out_ref)
