"""Disagreements between the library and the oracle over the whole GPU
parity suite (collected after the other parity tests).

Every parity comparison of the session adds its rows and its rows that
differ (all of them inside the declared near-tie band -- differences
outside it fail at once) to a tally by vocabulary class.  Small vocabularies
(V <= 4096) must stay under 0.01% of the rows; at V >= 128k the bound is
0.3% (see tests/parity.py for the reason)."""

import pytest

from tests.parity import FRAC, TALLY

pytestmark = pytest.mark.gpu


def test_suite_wide_disagreement_share():
    for cls, (rows, dis) in TALLY.items():
        if rows == 0:
            continue
        print(f"{cls} vocabularies: {dis} disagreements in {rows} rows ({dis / rows:.2e})")
        assert dis <= FRAC[cls] * rows, (cls, dis, rows)
