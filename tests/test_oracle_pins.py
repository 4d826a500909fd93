"""The oracle against its pins, and planted mistakes against the pins (CPU)."""
import pytest

import _pins

PLANTS = ["PLANT_TRANSPOSE", "PLANT_SLOT", "PLANT_APPEND_HEAD", "PLANT_OFFSET", "PLANT_NO_SCALE",
          "PLANT_DROP_LAST_V", "PLANT_GQA", "PLANT_WINDOW", "PLANT_CAUSAL", "PLANT_PREFIX_CAP",
          "PLANT_E4M3_TIES", "PLANT_FP8_VPERM"]


@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


@pytest.mark.parametrize("plant", PLANTS)
def test_planted_mistake_is_caught(plant):
    import oracle
    bad = oracle.load_planted([plant])
    caught = []
    for pin in _pins.ALL_PINS:
        try:
            pin(bad)
        except pytest.skip.Exception:
            continue
        except Exception as e:  # an assertion, or the oracle refusing a bad read
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"{plant} passed every pin"
