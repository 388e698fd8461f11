"""The acceptance rule for packed (FP16 rows + INT8 rows) states, applied
teacher-forced: a step under test and one step of the pages' quantiser (the
oracle's IEEE mode) start from the same packed bytes, and their packed
results are compared field by field.

The rule (stated for this path: INT8 codes bit-exact except that a code may
differ by one where the FP32 value before quantisation lies within 1e-6 of a
rounding boundary; o within 1e-3):

* INT8 codes are equal, except +-1 where, for the reference's value x and
  scale s, |x/s - (n + 1/2)| <= 1e-6 max(1, |x/s|), n + 1/2 being the
  boundary between the two codes.  A scale that moved by one ulp may flip
  several codes of its row; each flip is judged by the same rule.
* INT8 scales are within one ulp.
* FP16 rows are within one ulp.
* o is within 1e-3 of the reference, normwise per head.

The reference values come from the oracle only (dasc Appendix E.1 Eq. 8 and
DAMP §3.2 Eq. 5-6 for the quantiser; DAMP §3.1 Eq. 1-2 for the step).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

import oracle as orc

BOUNDARY_TOL = 1e-6
O_TOL = 1e-3


def split_tile(tile: np.ndarray, dk: int, dv: int, khi: int, group: int = 0):
    """Packed tile bytes -> (fp16 bits [khi][dv] uint16, codes [dk-khi][dv]
    int8, scales [dk-khi][n_groups] float32), rows in physical order.  The
    byte order is the word-interleaved one of the mixed layouts: FP16 value
    (r, c) at half ((r/2) dv + c) 2 + r%2, INT8 value (r, c) at byte
    ((q/4) dv + c) 4 + q%4 with q = r - khi; scales row-major after the
    codes (one per row, or dv/group per row)."""
    t = np.ascontiguousarray(tile, np.uint8)
    hb = 2 * khi * dv
    nlo = dk - khi
    ng = 1 if group == 0 else dv // group
    fp16 = t[:hb].copy().view(np.uint16).reshape(khi // 2, dv, 2).transpose(0, 2, 1).reshape(khi, dv)
    codes = (t[hb:hb + nlo * dv].copy().view(np.int8)
             .reshape(nlo // 4, dv, 4).transpose(0, 2, 1).reshape(nlo, dv))
    scales = t[hb + nlo * dv: hb + nlo * dv + 4 * nlo * ng].copy().view(np.float32).reshape(nlo, ng)
    return fp16, codes, scales


def _ordered(bits: np.ndarray, sign: int) -> np.ndarray:
    b = bits.astype(np.int64)
    return np.where(b & sign, -(b & (sign - 1)), b)


def ulp_diff_f32(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.abs(_ordered(a.view(np.uint32), 1 << 31) - _ordered(b.view(np.uint32), 1 << 31))


def ulp_diff_f16(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    return np.abs(_ordered(a_bits, 1 << 15) - _ordered(b_bits, 1 << 15))


@dataclass
class Tally:
    """What one or more comparisons saw (for the report and the asserts)."""
    tiles: int = 0
    codes: int = 0
    code_flips: int = 0
    worst_flip_distance: float = 0.0   # max |x/s - (n+1/2)| / max(1, |x/s|) over flips
    scale_ulp_max: int = 0
    scale_moved: int = 0
    fp16_ulp_max: int = 0
    o_rel_max: float = 0.0
    failures: list = field(default_factory=list)

    def ok(self) -> bool:
        return not self.failures


def reference_step_mixed(tile, pi_h, q_g, k_g, v_h, a_h, beta, dk, dv, khi, group=0, cs_h=None):
    """One step of the pages' quantiser (the oracle's IEEE mode) on one packed
    tile: returns (new tile bytes, FP32 tile before requantisation in physical
    rows, o).  a_h: scalar (GDN) or [dk] per logical channel (KDA)."""
    pi_h = np.asarray(pi_h)
    qp = np.ascontiguousarray(np.asarray(q_g, np.float32)[pi_h])
    kp = np.ascontiguousarray(np.asarray(k_g, np.float32)[pi_h])
    a = np.asarray(a_h, np.float32)
    ap = np.ascontiguousarray(a[pi_h] if a.ndim == 1 else np.full(dk, a, np.float32))
    v = np.asarray(v_h, np.float32)
    if group:
        T = orc.damp_unpack(tile, dk, dv, khi, group)
        vp = (v / np.asarray(cs_h, np.float32)).astype(np.float32)
        op = orc.step_tile(T, qp, kp, vp, ap, beta)
        o = (np.asarray(cs_h, np.float32) * op).astype(np.float32)
        return orc.damp_pack(T, khi, group, 0), T, o
    T = orc.mixed_unpack(tile, dk, dv, khi)
    o = orc.step_tile(T, qp, kp, v, ap, beta)
    return orc.mixed_pack(T, khi, 0), T, o


def compare_tile(tally: Tally, got_tile, ref_tile, x_ref, o_got, o_ref, dk, dv, khi, group=0,
                 where=""):
    """Apply the rule to one tile; record into ``tally``."""
    tally.tiles += 1
    fg, cg, sg = split_tile(got_tile, dk, dv, khi, group)
    fr, cr, sr = split_tile(ref_tile, dk, dv, khi, group)
    # FP16 rows
    du = ulp_diff_f16(fg, fr)
    tally.fp16_ulp_max = max(tally.fp16_ulp_max, int(du.max(initial=0)))
    if du.max(initial=0) > 1:
        tally.failures.append(f"{where}: FP16 row off by {int(du.max())} ulp")
    # scales
    ds = ulp_diff_f32(sg, sr)
    tally.scale_ulp_max = max(tally.scale_ulp_max, int(ds.max(initial=0)))
    tally.scale_moved += int(np.count_nonzero(ds))
    if ds.max(initial=0) > 1:
        tally.failures.append(f"{where}: scale off by {int(ds.max())} ulp")
    # codes, judged against the reference's value before quantisation
    ng = sr.shape[1]
    s_elem = np.repeat(sr, dv // ng, axis=1).astype(np.float64)
    x = x_ref[khi:].astype(np.float64)
    tally.codes += cg.size
    diff = cg.astype(np.int32) - cr.astype(np.int32)
    flips = diff != 0
    if flips.any():
        tally.code_flips += int(np.count_nonzero(flips))
        if np.abs(diff[flips]).max() > 1:
            tally.failures.append(f"{where}: a code differs by {int(np.abs(diff[flips]).max())}")
        r = x[flips] / s_elem[flips]
        boundary = (cg[flips].astype(np.float64) + cr[flips].astype(np.float64)) / 2.0
        dist = np.abs(r - boundary) / np.maximum(1.0, np.abs(r))
        tally.worst_flip_distance = max(tally.worst_flip_distance, float(dist.max()))
        if dist.max() > BOUNDARY_TOL:
            i = int(np.argmax(dist))
            tally.failures.append(
                f"{where}: code {int(cg[flips][i])} vs {int(cr[flips][i])} at x/s = {r[i]!r}, "
                f"{dist[i]:.3g} from the boundary")
    # o
    if o_got is not None:
        den = max(float(np.max(np.abs(o_ref))), 1e-30)
        rel = float(np.max(np.abs(o_got.astype(np.float64) - o_ref))) / den
        tally.o_rel_max = max(tally.o_rel_max, rel)
        if rel > O_TOL:
            tally.failures.append(f"{where}: o off by {rel:.3g} (normwise)")
