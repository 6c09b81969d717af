"""Each planted mistake in the oracle fails at least one pin (no GPU).

The oracle is built again with ORACLE_MUTATION=k; every k is one plausible
mistake (a square not rounded to binary32, a float accumulator, the psnr
noise formed from a frame total instead of rows, a dropped column, the
columns walked first, a wrong divisor or scaler, a row accumulator that is
not reset, swapped planes, a float division). The pins of
``oracle_pins.py`` must reject every one of them.
"""

import pytest

import oracle_pins as pins

MUTATIONS = {
    1: "square in double, not rounded to binary32",
    2: "second moment accumulated in float",
    3: "psnr noise adds every term into one double",
    4: "psnr rows added exactly and rounded once",
    5: "last column dropped",
    6: "second moment walks columns first",
    7: "divides by the pixel count minus one",
    8: "scaler 2^(bpc-7)",
    9: "first moment accumulated in float",
    10: "psnr row accumulator not reset per row",
    11: "ref and dis outputs swapped",
    13: "mse divided in float",
    14: "integer_psnr adds |d| instead of d^2",
    15: "integer_psnr divides by the width only",
}


@pytest.mark.parametrize("k", sorted(MUTATIONS), ids=lambda k: f"mut{k}")
def test_mutation_is_caught(k):
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(mutation=k)
        except AssertionError as exc:
            caught.append(pin.__name__)
            break
    assert caught, f"planted mistake {k} ({MUTATIONS[k]}) passed every pin"
