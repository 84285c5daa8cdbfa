"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_chi_square_recipe_matches_its_alpha():
    """The page's critical value 25.7448 is the alpha = 1e-4 quantile of a
    chi-square with 5 degrees of freedom."""
    stats = pytest.importorskip("scipy.stats")
    g = oracle_pins.golden("chi_square_recipe.json")
    assert abs(stats.chi2.isf(g["alpha"], g["dof"]) - g["critical"]) < 1e-4
