"""The library's host plan builders against the oracle (CPU only).

dasc §3.3 Eq. 2-3, §4.1, §4.2 Eq. 7; DAMP §5.1 Eq. 14-15 and top-K_hi.
Masks, windows and selections must equal the oracle's exactly; horizons and
risk scores agree to fp64 rounding.  Inputs are seeded synthetic gate
parameters and calibration trajectories with the pages' shapes (d = 128,
H = 256 decays after each anchor, 6 anchors).
"""
import numpy as np
import pytest

from oracle import plans as oplans
from recurrent_state_gb300 import build as rsbuild
from recurrent_state_gb300 import inputs as gen
from recurrent_state_gb300 import plans


@pytest.fixture(scope="module", autouse=True)
def _built():
    rsbuild.build()


@pytest.mark.parametrize("gate,a_s", [("std", -0.3), ("k3", 0.8)])
def test_horizons_masks_windows(gate, a_s):
    g = gen.rng(3)
    n = 32 * 128
    A = g.uniform(-4, 2, n).astype(np.float32)
    d = g.uniform(-8, 8, n).astype(np.float32)
    H = plans.dasc_horizons(gate, A, d, a_s)
    ref = oplans.static_horizons(gate, A, d, a_s)
    assert np.allclose(H, ref, rtol=1e-13, atol=0)
    for W in (16, 64, 128, 512):
        keep = plans.dasc_keep(H, W)
        assert np.array_equal(keep, oplans.retention_mask(ref, W))
        for n_p in (0, 5, 100, 10**6):
            assert plans.dasc_refresh_window(H, keep, W, n_p) == oplans.replay_window(ref, keep, W, n_p)
    assert plans.dasc_refresh_window(H, np.ones_like(keep), 64, 100) == 0


def test_risk_scores_and_selection():
    g = gen.rng(4)
    N, dk, dv, Hn = 6, 128, 128, 256
    S = (g.standard_normal((N, dk, dv)) * 10.0 ** g.uniform(-2, 1, (N, dk, 1))).astype(np.float32)
    S[:, 5, 7] = 50.0                               # an outlier in channel 5
    a = 1.0 / (1.0 + np.exp(-g.normal(3.0, 2.0, (1, 1, dk))))       # per-channel decay level
    dec = np.clip(a + g.normal(0, 0.01, (N, Hn, dk)), 0, 1).astype(np.float32)
    C = plans.damp_risk_scores(S, dec)
    ref = oplans.risk_scores(S, dec)
    assert np.allclose(C, ref, rtol=1e-12, atol=0)
    for k in (0, 1, 16, 128):
        assert np.array_equal(plans.damp_select_hi_rows(C, k)[0], oplans.select_high_precision(ref, k))


def test_selection_ties_and_errors():
    C = np.array([[0.1, 5.0, 3.0, 5.0, 0.0, 2.0], [1, 1, 1, 1, 1, 1]], np.float64)
    out = plans.damp_select_hi_rows(C, 2)
    assert out.tolist() == [[1, 3], [0, 1]]
    with pytest.raises(Exception):
        plans.damp_select_hi_rows(np.array([np.nan, 1.0]), 1)
    with pytest.raises(Exception):
        plans.damp_select_hi_rows(C, 7)
