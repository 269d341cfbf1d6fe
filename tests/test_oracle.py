"""The FP64 oracle against its pins (brute force, float64 SDPA, closed forms,
invariants). CPU only."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(orc, pin):
    pin(orc)


def test_oracle_rejects_bad_arguments(orc):
    import numpy as np
    q = np.zeros((1, 4, 3, 8), dtype=np.uint16)
    k = np.zeros((1, 4, 2, 8), dtype=np.uint16)      # Hq % Hkv != 0
    with pytest.raises(ValueError):
        orc.attention(q, k, k, mask_kind=0)
    with pytest.raises(ValueError):                   # additive kind needs a mask
        orc.attention(q, q, q, mask_kind=2)
