"""CPU: the fp64 oracle against closed forms, invariants, brute force and a golden example."""
import pytest

from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle):
    pin(oracle)


def test_oracle_rejects_bad_arguments(oracle):
    import numpy as np
    q = np.zeros((1, 3, 4, 8))
    k = np.zeros((1, 2, 4, 8))
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, k, k, 1.0)  # Hq % Hkv != 0
    bt = np.array([[5]], dtype=np.int32)
    with pytest.raises(ValueError):
        oracle.attn_decode(np.zeros((1, 2, 8)), np.zeros((2, 1, 4, 8)), np.zeros((2, 1, 4, 8)), bt,
                           np.array([3], dtype=np.int32), 1.0)  # block id 5 >= num_blocks
