"""GB300-native recurrent-state library (sm_103a).

Batched decode-step update of gated delta-rule linear attention (GDN and KDA)
on FP32 or mixed FP16/INT8 state pools, speculative-token replay, and ragged
dasc checkpoint pack/restore (verbatim units, or the INT8 checkpoint).  Every step runs in the CUDA library built from
``csrc/`` and reached through the C ABI of ``include/recurrent_state.h``;
this package only marshals torch tensors into that ABI (PyTorch provides
device memory and streams).

Submodules are imported lazily so that ``recurrent_state_gb300.inputs`` (the
seeded synthetic workloads) can be used without torch or a GPU.
"""
from __future__ import annotations

import importlib

__all__ = [
    "Layout", "Plan", "gdn_decode_update", "kda_decode_update", "spec_replay_update", "prefill_update",
    "state_convert", "ckpt_pack", "ckpt_restore", "ckpt_pack_int8", "ckpt_restore_int8", "RsError",
    "build", "inputs", "plans",
]

_LAZY = {
    "Layout": "api", "Plan": "api", "gdn_decode_update": "api", "kda_decode_update": "api",
    "spec_replay_update": "api", "prefill_update": "api", "state_convert": "api", "ckpt_pack": "api",
    "ckpt_restore": "api", "ckpt_pack_int8": "api", "ckpt_restore_int8": "api", "RsError": "_abi",
}


def __getattr__(name):
    if name in _LAZY:
        mod = importlib.import_module(f".{_LAZY[name]}", __name__)
        return getattr(mod, name)
    if name in ("build", "inputs", "api", "_abi", "plans"):
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
