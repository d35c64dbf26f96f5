"""Each planted mistake in the oracle (built with -DORACLE_MUTATION=k) fails
at least one pin, so the pins are able to see that class of error."""
import pytest

from oracle_pins import MUTATIONS, PINS


@pytest.mark.parametrize("mutation", sorted(MUTATIONS), ids=[MUTATIONS[k] for k in sorted(MUTATIONS)])
def test_mutation_is_caught(mutation):
    failed = [p.__name__ for p in PINS if not p(mutation)]
    assert failed, f"planted mistake '{MUTATIONS[mutation]}' passed every pin"
