"""The oracle's pins must catch plausible mistakes.

Each case below plants one mistake in a copy of the oracle's C source (a
dropped term, a wrong sign, a transposed index, a wrong rounding rule, a
wrong offset, a missed permutation...), builds it with the same flags on the
CPU, routes the oracle module through it, and runs the pin checks of the
other ``test_oracle_*`` modules.  At least one pin must fail for every
mistake; the real oracle passes them all (the other test modules).
"""
import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest

import oracle as orc
from recurrent_state_gb300 import inputs as gen

from . import test_oracle_ckpt as ck
from . import test_oracle_ckpt_int8 as i8
from . import test_oracle_damp as dm
from . import test_oracle_error_propagation as ep
from . import test_oracle_fused as fz
from . import test_oracle_mixed as mx
from . import test_oracle_quant as qt
from . import test_oracle_recurrence as rc
from . import test_oracle_row_map as rm


def _tiny():
    return gen.decode_workload(B=4, Hk=4, Hv=4, d=64, steps=16, per_channel=False,
                               in_dtype="f32", seed=0, tiny_gdn=True)


# Quick pin checks, cheapest first.
CHECKS = [
    ("quant_golden", qt.test_golden_tie_rows),
    ("quant_zero", qt.test_zero_row_uses_floor),
    ("quant_single", lambda: qt.test_single_nonzero_maps_to_full_scale(-0.001)),
    ("quant_bound", qt.test_error_bound_and_range),
    ("readout", rc.test_readout_is_transpose_of_updated_state),
    ("unit_key", rc.test_unit_key_full_strength_writes_value),
    ("pure_decay", lambda: rc.test_beta_zero_is_pure_decay(True)),
    ("gqa", rc.test_gqa_uses_adjacent_key_head),
    ("page_form", lambda: rc.test_oracle_matches_page_matrix_forms_fp64(_tiny(), "damp_eq2")),
    ("replay", lambda: rc.test_replay_equals_single_steps(True)),
    ("ckpt_golden", ck.test_golden_offsets_and_order),
    ("ckpt_numpy", lambda: ck.test_pack_matches_numpy_statement(1, 0.45)),
    ("ckpt_restore", lambda: ck.test_restore_zero_fills_and_roundtrips(0, 0.5)),
    ("row_map_golden", rm.test_hand_worked_row_maps),
    ("mixed_perm", mx.test_permutation_is_applied_to_inputs),
    ("mixed_bound", lambda: mx.test_mixed_step_within_local_quantisation_error(True)),
    ("mixed_replay", lambda: mx.test_mixed_replay_requantises_once(True)),
    ("int8_closed", lambda: i8.test_constant_rows_closed_form_and_order(1)),
    ("int8_roundtrip", lambda: i8.test_roundtrip_error_bound_and_zero_fill(0)),
    ("heads", i8.test_whole_head_pack_matches_fp32_pack),
    ("damp_groups", dm.test_constant_groups_closed_form),
    ("damp_bound", dm.test_group_error_bound),
    ("damp_pow2", lambda: dm.test_pow2_value_scaling_equivariance(True)),
    ("damp_fp64", dm.test_transformed_step_matches_original_map_fp64),
    ("fused_code", fz.test_rcp_code_is_nearest_integer_to_exact_product),
    ("fused_once", fz.test_rcp_code_rounds_the_exact_product_once),
    ("fused_constructed", fz.test_constructed_row_where_the_modes_differ),
    ("fused_bound", lambda: fz.test_fused_step_within_local_quantisation_error(True)),
    ("fused_replay", lambda: fz.test_fused_replay_one_equals_decode(True)),
    ("fused_acceptance", lambda: fz.test_fused_mode_meets_the_acceptance_rule_under_decay("mixed", True)),
    ("error_recursion", lambda: ep.test_error_recursion_eq12_eq13(0)),
]

READOUT_BLOCK = """    /* readout o = S^T q on the updated state */
    if (o) {
        for (c = 0; c < dv; ++c) {
            float acc = 0.0f;
            for (u = 0; u < dk; ++u)
                acc = fmaf(S[(size_t)u * dv + c], q[u], acc);
            o[c] = acc;
        }
    }
"""
WRITE_BLOCK = """    /* rank-1 delta-rule write S <- S + beta k e^T */
    for (u = 0; u < dk; ++u) {
        float bk = beta * k[u];
        for (c = 0; c < dv; ++c)
            S[(size_t)u * dv + c] = fmaf(bk, e[c], S[(size_t)u * dv + c]);
    }
"""

MUTATIONS = {
    "error_sign": [("e[c] = v[c] - p;", "e[c] = p - v[c];")],
    "decay_dropped": [("S[(size_t)u * dv + c] = S[(size_t)u * dv + c] * au;",
                       "S[(size_t)u * dv + c] = S[(size_t)u * dv + c];")],
    "decay_index": [("float au = a[(size_t)u * (size_t)a_stride];",
                     "float au = a[(size_t)(dk - 1 - u) * (size_t)a_stride];")],
    "prediction_with_q": [("p = fmaf(S[(size_t)u * dv + c], k[u], p);",
                           "p = fmaf(S[(size_t)u * dv + c], q[u], p);")],
    "beta_dropped": [("float bk = beta * k[u];", "float bk = k[u];")],
    "write_wrong_index": [("fmaf(bk, e[c], S[(size_t)u * dv + c]);",
                           "fmaf(bk, e[u], S[(size_t)u * dv + c]);")],
    "readout_transposed": [("acc = fmaf(S[(size_t)u * dv + c], q[u], acc);",
                            "acc = fmaf(S[(size_t)c * dv + u], q[u], acc);")],
    "readout_before_write": [(WRITE_BLOCK + READOUT_BLOCK, READOUT_BLOCK + WRITE_BLOCK)],
    "gqa_modulo": [("{ return h / (Hv / Hk); }", "{ return h % Hk; }")],
    "round_half_away": [("float r = rintf(x / s);", "float r = roundf(x / s);")],
    "scale_128": [("return fmaxf(row_absmax(n, x), 1e-8f) / 127.0f;",
                   "return fmaxf(row_absmax(n, x), 1e-8f) / 128.0f;")],
    "abs_dropped": [("float ax = fabsf(x[i]);", "float ax = x[i];")],
    "offsets_not_cumulative": [("offsets[l] = offsets[l - 1] + r;", "offsets[l] = r;")],
    "pack_reversed_in_layer": [
        ("memcpy(ckpt + ((size_t)d * off[L] + (size_t)(off[l] + j)) * ub,",
         "memcpy(ckpt + ((size_t)d * off[L] + (size_t)(off[l + 1] - 1 - j)) * ub,")],
    "restore_no_zero_fill": [("memset(dst, 0, ub);", "(void)dst;")],
    "row_map_rest_descending": [("for (c = 0; c < dk; ++c)        /* then the rest, ascending */",
                                 "for (c = dk - 1; c >= 0; --c)  /* then the rest, ascending */")],
    "row_map_selection_last": [("    for (c = 0; c < dk; ++c)        /* the selected region, ascending */\n"
                                "        if (chosen[c]) pi[r++] = (int16_t)c;\n"
                                "    for (c = 0; c < dk; ++c)        /* then the rest, ascending */\n"
                                "        if (!chosen[c]) pi[r++] = (int16_t)c;",
                                "    for (c = 0; c < dk; ++c)        /* then the rest, ascending */\n"
                                "        if (!chosen[c]) pi[r++] = (int16_t)c;\n"
                                "    for (c = 0; c < dk; ++c)        /* the selected region, ascending */\n"
                                "        if (chosen[c]) pi[r++] = (int16_t)c;")],
    "mixed_q_unpermuted": [("qp[r] = qh[ph[r]];", "qp[r] = qh[r];")],
    "mixed_alpha_unpermuted": [("? alpha[((size_t)b * Hv + h) * dk + ph[r]]",
                                "? alpha[((size_t)b * Hv + h) * dk + r]")],
    "replay_requant_each_token": [
        ("beta[bt * Hv + h], o ? o + (bt * Hv + h) * dv : NULL);\n        }\n"
         "        orc_mixed_pack_m(dk, dv, khi, mode, T, tile);",
         "beta[bt * Hv + h], o ? o + (bt * Hv + h) * dv : NULL);\n"
         "            orc_mixed_pack_m(dk, dv, khi, mode, T, tile);\n"
         "            orc_mixed_unpack(dk, dv, khi, tile, T);\n        }\n"
         "        orc_mixed_pack_m(dk, dv, khi, mode, T, tile);")],
    "fused_double_rounding": [("double r = rint((double)x * (double)y);",
                               "double r = rint((double)(x * y));")],
    "fused_mode_ignored": [("if (mode == 1 && a <= FLT_MAX) {", "if (0) {")],
    "replay_skips_first": [("for (t = 0; t < n; ++t) {", "for (t = 1; t < n; ++t) {")],
    "int8_scale_per_unit": [
        ("memcpy(ckpt + (size_t)d * sb + (size_t)cb + (size_t)row * 4, &sc, 4);",
         "memcpy(ckpt + (size_t)d * sb + (size_t)cb + (size_t)(off[l] + j) * 4, &sc, 4);")],
    "int8_restore_no_zero_fill": [("memset(dst, 0, (size_t)R * dv * 4);", "(void)dst;")],
    "int8_dequant_unscaled": [("                                       sc, dst + (size_t)r * dv);",
                               "                                       1.0f, dst + (size_t)r * dv);")],
    "damp_value_scale_multiplied": [("vp[c] = v[c] / cs[c];", "vp[c] = v[c] * cs[c];")],
    "damp_readout_unscaled": [("o[c] = cs[c] * op[c];", "o[c] = op[c];")],
    "damp_group_scale_index": [("memcpy(&s, sc + ((size_t)(r - khi) * ng + gi) * 4, 4);",
                                "memcpy(&s, sc + ((size_t)(r - khi) * ng) * 4, 4);")],
    "damp_convert_multiplies": [("T[(size_t)r * dv + c] = S[(size_t)pi[r] * dv + c] / cs[c];",
                                 "T[(size_t)r * dv + c] = S[(size_t)pi[r] * dv + c] * cs[c];")],
    "heads_unit_is_fp32_head": [("size_t ub = (size_t)head_bytes, slot_bytes = (size_t)Hv * ub;\n    int status = 0, i, l, x;\n    if (L > 1024) return -1;\n    orc_plan_offsets(L, Hv, 1, 0, keep, off);\n    for (i = 0; i < n; ++i) {\n        int32_t s = src_slots[i]",
                                 "size_t ub = (size_t)head_bytes, slot_bytes = (size_t)Hv * ub * 2;\n    int status = 0, i, l, x;\n    if (L > 1024) return -1;\n    orc_plan_offsets(L, Hv, 1, 0, keep, off);\n    for (i = 0; i < n; ++i) {\n        int32_t s = src_slots[i]")],
}


def _mutant_source(edits):
    src = orc.source()
    for old, new in edits:
        assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
        src = src.replace(old, new)
    return src


@pytest.fixture(scope="module")
def workdir():
    with tempfile.TemporaryDirectory(prefix="orc_mut_") as d:
        yield d


def first_failing_check(path, checks=None):
    """Run the pin checks against the library at ``path``; return the name of
    the first one that fails, or None.  Called in a child process."""
    caught = None
    with orc.use_library(path):
        np.seterr(all="ignore")
        for check_name, fn in CHECKS:
            if checks and check_name not in checks:
                continue
            try:
                fn()
            except (AssertionError, ValueError, FloatingPointError):
                caught = check_name
                break
    return caught


_CHILD = """
import sys
from tests.test_oracle_mutations import first_failing_check
name = first_failing_check(sys.argv[1])
print("CAUGHT:" + str(name))
"""


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, workdir):
    # Each mutant runs in its own process: a planted indexing mistake may
    # write outside the buffers the checks sized, and must not take the test
    # process down with it.
    path = orc.build_variant(_mutant_source(MUTATIONS[name]),
                             os.path.join(workdir, f"lib_{name}.so"))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _CHILD, path], cwd=root,
                       capture_output=True, text=True, timeout=300)
    caught = [ln for ln in r.stdout.splitlines() if ln.startswith("CAUGHT:")]
    assert r.returncode == 0 and caught, (r.returncode, r.stdout[-2000:], r.stderr[-2000:])
    assert caught[-1] != "CAUGHT:None", f"no pin caught the planted mistake {name!r}"
