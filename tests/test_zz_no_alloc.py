"""The pack entry point for callers that cannot allocate device memory.

rs_ckpt_pack_noalloc must produce the same checkpoint bytes as rs_ckpt_pack
(pack is a byte copy: the tolerance is bit-exactness), on two calls in a row
with different plans, so that the second call really replaces the table the
first one left in the library's fixed device array.  This file is collected
last; it also passes when run on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import recurrent_state_gb300 as rs
from recurrent_state_gb300 import _abi
from recurrent_state_gb300 import inputs as gen

from .gpu_util import dev, ensure_built, host, same_bits

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _pack_noalloc(plan, pool, src, dst, ckpt, status):
    n_pool = pool.shape[1]
    stride = pool[0].numel() * pool.element_size()
    return _abi.lib().rs_ckpt_pack_noalloc(
        plan._h, _p(pool), stride, n_pool, _p(src), _p(dst), src.numel(), _p(ckpt),
        ckpt.shape[0], _p(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_pack_matches_pack_on_two_calls():
    ensure_built()
    L, slots, Hv, d, n = 6, 9, 8, 128, 7
    pool = torch.randn((L, slots, Hv, d, d), device="cuda")
    lay = rs.Layout("fp32", d, Hv, 1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    plans = [(0, gen.keep_mask(L, Hv, 0.5, seed=21), "head"),
             (1, gen.keep_mask(L, Hv * d, 0.45, seed=22), "channel")]
    for call, (unit, keep, name) in enumerate(plans):
        src, dst = gen.ckpt_slots(slots, n, seed=30 + call)
        src_d, dst_d = dev(src), dev(dst)
        ref_plan = rs.Plan(lay, keep, name).upload()
        ref = torch.zeros((n, ref_plan.ckpt_slot_bytes), dtype=torch.uint8, device="cuda")
        rs.ckpt_pack(ref_plan, pool, src_d, dst_d, ref)
        plan = rs.Plan(lay, keep, name)  # never uploaded: the call needs no allocation
        out = torch.full((n, plan.ckpt_slot_bytes), 0xEE, dtype=torch.uint8, device="cuda")
        assert _pack_noalloc(plan, pool, src_d, dst_d, out, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert same_bits(host(out), host(ref)), f"call {call + 1} differs from rs_ckpt_pack"


def test_noalloc_pack_at_exactly_the_table_size():
    """A plan retaining exactly 262,144 units fills every entry of the fixed
    table: the call is accepted and its bytes equal rs_ckpt_pack's."""
    ensure_built()
    L, slots, Hv, d, n = 64, 2, 64, 64, 2
    lay = rs.Layout("fp32", d, Hv, 1)
    keep = np.ones((L, Hv * d), np.uint8)  # 64 layers x 4,096 key channels = 262,144
    g = torch.Generator(device="cuda").manual_seed(5)
    pool = torch.randn((L, slots, Hv, d, d), device="cuda", generator=g)
    src_d = dev(np.array([1, 0], np.int32))
    dst_d = dev(np.array([0, 1], np.int32))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_plan = rs.Plan(lay, keep, "channel").upload()
    assert ref_plan.ckpt_slot_bytes == 262144 * d * 4
    ref = torch.zeros((n, ref_plan.ckpt_slot_bytes), dtype=torch.uint8, device="cuda")
    rs.ckpt_pack(ref_plan, pool, src_d, dst_d, ref)
    plan = rs.Plan(lay, keep, "channel")
    out = torch.full((n, plan.ckpt_slot_bytes), 0xEE, dtype=torch.uint8, device="cuda")
    assert _pack_noalloc(plan, pool, src_d, dst_d, out, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out, ref)


def test_noalloc_pack_rejects_plans_beyond_the_table():
    ensure_built()
    lay = rs.Layout("fp32", 128, 64, 1)
    keep = np.ones((33, 64 * 128), np.uint8)  # 270,336 retained units > 262,144
    plan = rs.Plan(lay, keep, "channel")
    t = torch.zeros(16, dtype=torch.uint8, device="cuda")
    i = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = _abi.lib().rs_ckpt_pack_noalloc(plan._h, _p(t), 0, 1, _p(i), _p(i), 1, _p(t), 1, None,
                                         None)
    assert st == _abi.RS_ERR_UNSUPPORTED
