"""The oracle against its pins (no GPU): hand-derived worked blocks, exhaustive
scalar decoders, independent numpy dequantizers, brute-force routing, dense
numpy fp64 FFNs and layer invariants.  See tests/oracle_pins.py."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)
