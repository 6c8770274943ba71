"""The GPU parity checks themselves, on planted errors (CPU only).

A norm over a whole call, or even over one token's output, can hide a few
wrong output rows: 5 unwritten rows of a 16384-row map change a token's
relative L2 error by only sqrt(5 / 16384) ~ 1.7%, inside the bf16 bound of
2e-2.  The element-against-row-RMS bound must catch them.
"""
import numpy as np
import pytest

from tests.gpu_util import per_token_rel


def _case(seed=0, T=26, d_out=16384):
    rs = np.random.default_rng(seed)
    ref = rs.standard_normal((T, d_out))
    return ref, ref + 1e-4 * rs.standard_normal((T, d_out))


def test_clean_output_passes():
    ref, y = _case()
    assert per_token_rel(y, ref, 2e-2) < 1e-3


def test_unwritten_row_tail_is_caught():
    ref, y = _case()
    y[:, -5:] = 0.0  # the last CTA's 5 rows of every token left unwritten
    assert np.linalg.norm(y - ref) / np.linalg.norm(ref) <= 2e-2       # whole call: hidden
    assert np.median(np.linalg.norm(y - ref, axis=1) / np.linalg.norm(ref, axis=1)) <= 2e-2  # most tokens too
    with pytest.raises(AssertionError, match="per-token|element error"):
        per_token_rel(y, ref, 2e-2)


def test_one_unwritten_row_is_caught_by_the_element_bound():
    ref, y = _case()
    o = int(np.argmin(np.abs(np.abs(ref[5]) - 1.5)))  # an output row of token 5 with |y| ~ 1.5 RMS
    y[5, o] = 0.0
    assert np.max(np.linalg.norm(y - ref, axis=1) / np.linalg.norm(ref, axis=1)) <= 2e-2
    with pytest.raises(AssertionError, match="element error"):
        per_token_rel(y, ref, 2e-2)


def test_one_wrong_token_is_caught():
    ref, y = _case()
    y[3, -40:] *= -1.0  # one token's tail with the wrong sign
    assert np.linalg.norm(y - ref) / np.linalg.norm(ref) <= 2e-2       # whole call: hidden
    with pytest.raises(AssertionError, match="per-token"):
        per_token_rel(y, ref, 2e-2)


def test_zero_reference_rows_must_be_zero():
    ref, y = _case(T=4, d_out=64)
    ref[2] = 0.0
    y[2] = 0.0
    per_token_rel(y, ref, 2e-2)
    y[2, 7] = 1.0
    with pytest.raises(AssertionError, match="should be zero"):
        per_token_rel(y, ref, 2e-2)


def test_nonfinite_reference_rows_are_skipped():
    ref, y = _case(T=4, d_out=64)
    ref[1, 3] = np.nan
    y[1] = 5.0
    assert per_token_rel(y, ref, 2e-2) < 1e-3
