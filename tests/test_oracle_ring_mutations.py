"""Mutation check of the ring-decode pins: plausible mistakes planted in a copy
of the oracle's sliding-window decode (its source text, rebound in this
process only) must each make one of the ring pins fail."""
import inspect
import textwrap

import pytest

import oracle
from tests import test_oracle_decode_rope as pins

RING_PINS = [pins.test_ring_decode_one_row_ring_returns_the_newest_value,
             pins.test_ring_decode_ignores_tokens_outside_the_window,
             pins.test_ring_decode_matches_brute_force_on_the_window,
             pins.test_ring_at_least_as_long_as_the_history_is_plain_decode]

MUTATIONS = {
    # the window starts one token late (keeps capacity - 1 tokens)
    "window_one_short": ("lo = max(0, int(n[b]) - capacity)", "lo = max(0, int(n[b]) - capacity + 1)"),
    # the oldest tokens instead of the newest once the ring has wrapped
    "oldest_tokens": ("lo = max(0, int(n[b]) - capacity)", "lo = 0"),
    # the newest token left out (window ends one early)
    "drops_newest": ("kc[b, :, :lens[b]] = k_tokens[b, :, lo:n[b]]",
                     "kc[b, :, :lens[b]] = k_tokens[b, :, max(0, lo - 1):n[b] - 1]"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_ring_pins_catch_planted_mistake(name, monkeypatch):
    before, after = MUTATIONS[name]
    src = textwrap.dedent(inspect.getsource(oracle.decode_ring))
    assert src.count(before) == 1, f"mutation site for {name} not found"
    ns = dict(vars(oracle))
    exec(compile(src.replace(before, after), f"<mutated decode_ring: {name}>", "exec"), ns)
    monkeypatch.setattr(oracle, "decode_ring", ns["decode_ring"])
    failed = 0
    for pin in RING_PINS:
        try:
            pin()
        except (AssertionError, ValueError):
            failed += 1
    assert failed > 0, f"no ring pin caught mutation {name}"


def test_ring_pins_pass_on_the_unmutated_oracle():
    for pin in RING_PINS:
        pin()
