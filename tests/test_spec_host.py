"""Host logic of speculative decoding through the C ABI (no GPU): prompt lookup and the
acceptance gate, on hand-built cases whose answers follow from the rules stated on the
Rust page ("Speculative decoding without a draft model")."""
import pytest

mie = pytest.importorskip("memory_bound_decode_dequant_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    try:
        mie.lib()
    except RuntimeError as e:  # not built in this checkout
        pytest.skip(str(e))


def test_lookup_proposes_what_followed_the_earlier_occurrence():
    # the last 3 tokens (5 6 7) occurred at the start; 8 5 6 followed them
    assert mie.mie_lookup_propose([5, 6, 7, 8, 5, 6, 7], 2, 4, 3) == [8, 5, 6]


def test_lookup_takes_the_most_recent_occurrence():
    # "1 2" occurs at 0 (then 9) and at 3 (then 8): the later one wins
    assert mie.mie_lookup_propose([1, 2, 9, 1, 2, 8, 1, 2], 2, 4, 2) == [8, 1]


def test_lookup_prefers_the_longest_match():
    # "1 2 3" (then 7) beats the more recent "2 3" (then 8)
    assert mie.mie_lookup_propose([1, 2, 3, 7, 2, 3, 8, 1, 2, 3], 2, 4, 1) == [7]


def test_lookup_needs_two_tokens_and_stops_at_the_end():
    assert mie.mie_lookup_propose([4, 9, 4], 2, 4, 3) == []  # a one-token match does not count
    assert mie.mie_lookup_propose([4, 9, 4], 1, 4, 3) == [9, 4]
    # the earlier occurrence may not overlap the suffix; guesses never pass the end
    assert mie.mie_lookup_propose([1, 2, 1, 2], 2, 4, 4) == [1, 2]
    assert mie.mie_lookup_propose([1, 1, 1], 2, 4, 4) == []
    assert mie.mie_lookup_propose([3], 2, 4, 4) == []


def test_gate_pauses_and_doubles_then_resets():
    g = mie.SpecGate(window=10, threshold=0.3, pause=5, pause_max=80)
    for _ in range(9):
        assert g.open()
        g.record(3, 0)
    assert g.open()
    g.record(3, 0)  # the 10th failing attempt: pause of 5
    assert [g.open() for _ in range(5)] == [False] * 5
    assert g.open()
    g.record(3, 0)  # the window is still below 30 %: the next pause is 10
    assert [g.open() for _ in range(10)] == [False] * 10
    lengths = []
    for _ in range(4):
        assert g.open()
        g.record(3, 0)
        n = 0
        while not g.open():
            n += 1
        lengths.append(n)
    assert lengths == [20, 40, 80, 80]  # doubling, capped at 80


def test_gate_length_resets_once_the_window_recovers():
    g = mie.SpecGate(window=2, threshold=0.5, pause=1, pause_max=8)
    assert g.open()
    g.record(1, 0)  # one attempt: no full window yet
    assert g.open()
    g.record(1, 0)  # window 0 / 2: pause 1, next 2
    assert not g.open() and g.open()
    g.record(1, 1)  # window 1 / 2 = threshold: length back to 1
    assert g.open()
    g.record(1, 0)  # window 1 / 2: no pause
    assert g.open()
    g.record(1, 0)  # window 0 / 2: pause of the reset length 1
    assert not g.open() and g.open()
    g.record(1, 0)  # still 0 / 2: the consecutive pause doubles to 2
    assert [g.open(), g.open(), g.open()] == [False, False, True]
