"""The fp64 oracle against what the pages and mathematics fix (no GPU)."""
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_capacity_example_sizes():
    """The sizes the bench's byte model uses agree with the pages' capacity
    example at N=32768, d=dv=64 in fp16."""
    g = pins.golden("capacity_s1.json")
    n, d, dv, r, e = g["N"], g["d"], g["dv"], g["r"], g["bytes_per_element"]
    assert n * n * e == g["nxn_gib"] * 2**30
    assert n * (d + dv) * e == g["kv_mib"] * 2**20
    assert abs((r * dv + r) * e / 1024 - g["state_kib_approx"]) < 0.05


def test_rejects_bad_arguments(orc):
    import numpy as np

    q = np.zeros((1, 1, 4, 2))
    with pytest.raises(oracle.OracleError):
        orc.forward(q, q, q, causal=False, gamma=np.array([0.5]))
