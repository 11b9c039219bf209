"""CPU checks of the parity helper the GPU tests use: a single wrong token
row, a wrong short sequence, a wrong head, a wrong state or a NaN must fail it,
even where the whole-tensor relative L2 stays under the tolerance."""
from __future__ import annotations

import numpy as np
import pytest

from parity_util import TOL, assert_parity, parity_report, rel_l2

LENGTHS = [0, 1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 200]


def _pair(seed=0, H=3, d=128, noise=5e-3):
    """Reference outputs of the ragged test's shape and a copy with the kind of
    relative rounding noise a correct bf16 kernel shows."""
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(LENGTHS)])
    ref = rng.standard_normal((cu[-1], H, d))
    got = ref * (1.0 + noise * rng.standard_normal(ref.shape))
    return got, ref, cu


def test_correct_outputs_pass():
    got, ref, cu = _pair()
    rep = assert_parity(got, ref, TOL["bf16"], cu=cu)
    assert rep["whole"] < 6e-3 and rep["row"] < 2e-2 and rep["slice"] < 1e-2


@pytest.mark.parametrize("where", ["length-1 sequence", "last row of a ragged chunk",
                                   "first row of a sequence"])
def test_one_wrong_row_fails_although_the_whole_tensor_passes(where):
    got, ref, cu = _pair()
    row = {"length-1 sequence": cu[1], "last row of a ragged chunk": cu[11] - 1,
           "first row of a sequence": cu[13]}[where]
    got[row, 1] = 1.5 * ref[row, 1]                 # one (token, head) row 50 % off
    assert rel_l2(got, ref) <= TOL["bf16"]          # hidden in the whole-tensor figure
    with pytest.raises(AssertionError):
        assert_parity(got, ref, TOL["bf16"], cu=cu)
    rep = parity_report(got, ref, cu)
    assert rep["row_at"]["head"] == 1
    assert cu[rep["row_at"]["sequence"]] + rep["row_at"]["row_in_sequence"] == row


def test_slightly_wrong_slice_fails():
    """A whole (sequence, head) slice 5 % off: each row is near the bound but the
    slice's own relative L2 catches it."""
    got, ref, cu = _pair()
    a, b = cu[14], cu[15]
    got[a:b, 2] = ref[a:b, 2] * 1.05
    assert rel_l2(got, ref) <= TOL["bf16"]
    rep = parity_report(got, ref, cu)
    assert rep["slice"] > TOL["bf16"] and rep["slice_at"] == {"sequence": 14, "head": 2}


def test_wrong_state_fails():
    rng = np.random.default_rng(1)
    ref = rng.standard_normal((6, 4, 128, 128))
    got = ref * (1 + 1e-3 * rng.standard_normal(ref.shape))
    assert_parity(got, ref, TOL["bf16"])
    got[4, 3, 17] *= 1.5                             # one key row of one state, 50 % off
    assert rel_l2(got, ref) <= TOL["bf16"]
    with pytest.raises(AssertionError):
        assert_parity(got, ref, TOL["bf16"])


def test_nan_fails():
    got, ref, cu = _pair()
    got[5, 0, 3] = np.nan
    with pytest.raises(AssertionError):
        assert_parity(got, ref, TOL["bf16"], cu=cu)


def test_low_signal_slice_is_bounded_row_wise():
    """A one-token sequence whose reference row is tiny (q nearly orthogonal to
    k): its relative error may be large, but it is held to the head's RMS."""
    got, ref, cu = _pair()
    r = cu[1]
    ref[r, 0] *= 1e-3
    got[r, 0] = ref[r, 0] + 1e-3 * np.linalg.norm(ref[r + 1, 0]) / np.sqrt(128)
    assert_parity(got, ref, TOL["bf16"], cu=cu)            # skipped as a slice, fine as a row
    got[r, 0] = ref[r, 0] + 0.1 * np.linalg.norm(ref[r + 1, 0]) / np.sqrt(128) * 5
    with pytest.raises(AssertionError):
        assert_parity(got, ref, TOL["bf16"], cu=cu)
