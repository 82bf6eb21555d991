"""The CPU oracle against its pins (closed forms, invariants, brute force)."""
import pytest

import oracle
from oracle_pins import ORACLE_PINS, pin_materialised_rows_sum_to_one


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", ORACLE_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(orc, pin):
    pin(orc)


def test_materialised_rows_sum_to_one():
    pin_materialised_rows_sum_to_one()


def test_oracle_rejects_bad_arguments(orc):
    import numpy as np
    q = np.zeros((1, 4, 3, 8), np.uint16)
    k = np.zeros((1, 4, 2, 8), np.uint16)  # 3 % 2 != 0
    with pytest.raises(ValueError):
        orc.attn_rows(q, k, k, "fp16", True, -1, 1.0, np.array([0]))
    k = np.zeros((1, 4, 1, 8), np.uint16)
    with pytest.raises(ValueError):  # row id out of range
        orc.attn_rows(q, k, k, "fp16", True, -1, 1.0, np.array([12]))
    with pytest.raises(ValueError):  # window below -1
        orc.attn_rows(q, k, k, "fp16", True, -2, 1.0, np.array([0]))
