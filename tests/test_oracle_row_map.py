"""Pins of the oracle's row map (DAMP Appendix A.2, Algorithm 1, last step;
Appendix A.3 Eq. 17): physical row r of a mixed state holds logical key
channel pi[r], the selected channels first, each region ascending."""
import json
import os

import numpy as np
import pytest

import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "row_map.json")


def test_hand_worked_row_maps():
    for case in json.load(open(GOLDEN))["cases"]:
        sel = np.array([case["selected"]], np.int16).reshape(1, -1)
        pi = orc.row_map(sel, case["dk"])
        assert pi[0].tolist() == case["pi"], case


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_row_map_is_a_permutation_with_the_selection_first(seed):
    g = np.random.default_rng(seed)
    dk, khi = 128, 16
    sel = np.stack([g.permutation(dk)[:khi] for _ in range(6)]).astype(np.int16)  # unsorted
    pi = orc.row_map(sel, dk)
    for h in range(sel.shape[0]):
        assert sorted(pi[h].tolist()) == list(range(dk))
        assert pi[h, :khi].tolist() == sorted(sel[h].tolist())
        rest = pi[h, khi:]
        assert np.all(np.diff(rest) > 0) and not set(rest.tolist()) & set(sel[h].tolist())


def test_row_map_rejects_repeated_or_out_of_range_channels():
    with pytest.raises(ValueError):
        orc.row_map(np.array([[3, 3]], np.int16), 8)
    with pytest.raises(ValueError):
        orc.row_map(np.array([[3, 8]], np.int16), 8)
