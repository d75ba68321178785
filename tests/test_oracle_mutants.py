"""Plant a mistake in the oracle (on the CPU) and check that the pins see it.

Each ORC_PLANT_* switch in oracle/la_oracle.c builds a variant with one
plausible slip.  A pin set that let any of them pass would not be pinning the
oracle; every variant must fail at least one pin.
"""
import pytest

import oracle
import pins

PLANTS = [
    "ORC_PLANT_PHI_NO_PLUS_ONE",     # elu without the +1
    "ORC_PLANT_READ_BEFORE_WRITE",   # exclusive prefix: token t does not see itself
    "ORC_PLANT_DECAY_AFTER_WRITE",   # gamma applied to the fresh record too
    "ORC_PLANT_TRANSPOSED_UPDATE",   # key feature paired with the wrong value channel
    "ORC_PLANT_Z_NO_DECAY",          # normaliser left undecayed
    "ORC_PLANT_DROP_NORMALISER",     # division by phi(q)^T z dropped
    "ORC_PLANT_GLA_ALONG_VALUES",    # per-channel decay applied along the values
    "ORC_PLANT_IGNORE_Z0",           # the initial normaliser state dropped
    "ORC_PLANT_FAVOR_NO_NORM",       # random features without the -|x|^2/2 term
]


@pytest.mark.parametrize("plant", PLANTS)
def test_planted_mistake_is_caught(plant, tmp_path_factory):
    mutant = oracle.load((plant,), out_dir=tmp_path_factory.mktemp("mutant"))
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, oracle.OracleError):
            failed.append(pin.__name__)
    assert failed, f"{plant}: no pin failed"
