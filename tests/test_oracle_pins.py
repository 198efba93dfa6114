"""The oracle against what the pages and the mathematics fix (CPU only)."""
import pytest

import oracle
from tests import oracle_checks as oc


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("check", oc.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(orc, check):
    if check is oc.check_frequencies_high_precision:
        pytest.importorskip("mpmath")
    check(orc)


def test_oracle_rejects_bad_axes(orc):
    import numpy as np

    with pytest.raises(ValueError):
        orc.rope_tables(np.zeros((2, 2), np.int32), (3, 5), 2000.0)
    q = np.zeros((1, 2, 1, 8))
    with pytest.raises(ValueError):
        orc.joint_rope_attention(q, q, q, None, np.zeros((2, 2), np.int32), (2, 2), 10.0)
