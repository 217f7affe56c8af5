"""CPU check of the tie fixtures used by the GPU tie tests: the expected ids
worked out by hand agree with the oracle's selection."""
from __future__ import annotations

import numpy as np

import oracle
from tie_cases import KINDS, expected_ids_t1, tie_bias


def test_tie_expectations_match_the_oracle():
    """The hand-made expectations above agree with the oracle's selection (a
    CPU check of the test's own fixtures)."""
    for E in (256, 1024):
        for kind in KINDS:
            bias = tie_bias(E, 8, kind)
            logits = np.zeros((1, E), np.float32)
            ids, _ = oracle.select(logits, bias, 8, 8, 4, 2.5)
            assert list(ids[0]) == expected_ids_t1(kind, E, 8, 8), (E, kind)
