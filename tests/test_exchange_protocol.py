"""CPU checks of the on-chip combine's exchange protocol through its model (tests/exchange_model.py).

Both forms as built (pulled, the default; pushed, opt-in) must be clean for cluster sizes 2..16,
with and without unwinding CTAs and with bounded waits that run out at random; each planted
reordering must be caught in some interleaving.
"""

import itertools

import pytest

from tests import exchange_model as em

SIZES = (2, 3, 5, 8, 16)


@pytest.mark.parametrize("push", [False, True])
def test_exchange_as_built_is_clean(push):
    for n, seed in itertools.product(SIZES, range(25)):
        em.ExchangeSim(n, push, seed).run()
        em.ExchangeSim(n, push, seed, unwound={seed % n}).run()
        em.ExchangeSim(n, push, seed, unwound=set(range(n))).run()
        em.ExchangeSim(n, push, seed, abort_rate=0.05).run()


def test_pushed_bytes_may_land_before_their_arrival():
    # A store's bytes can be counted before its sender's expect-tx arrival (the transaction count
    # dips below zero): the phase still completes only once every arrival and byte is in.
    for n, seed in itertools.product(SIZES, range(25)):
        em.ExchangeSim(n, True, seed, mutations=("stores_before_arrival",)).run()


def caught(mutation, push, **kw):
    for n, seed in itertools.product(SIZES, range(60)):
        try:
            em.ExchangeSim(n, push, seed, mutations=(mutation,), **kw).run()
        except em.ProtocolError as e:
            return str(e)
    return None


def test_pushed_closing_barrier_is_for_the_unwinding_path():
    # The stores leave from registers and every owner waits for its own rows before it tears
    # down, so an owner that arrives at the closing barrier before its rows have landed harms
    # nothing in a clean run; the barrier matters once an owner gives up (see below).
    assert caught("arrive_before_recv_wait", True) is None


@pytest.mark.parametrize("mutation,push,kw,expect", [
    # pushed: the owner reads its receive area without waiting for the bytes
    ("combine_without_wait", True, {}, "before it landed"),
    # pushed: an owner that gave up (unwinding, or a wait that ran out) passes the closing barrier
    # with stores still on their way into it
    ("no_drain_on_abort", True, {"unwound": {1}}, "after it tore down"),
    ("no_drain_on_abort", True, {"abort_rate": 0.05}, "after it tore down"),
    # pushed: an unwinding rank that does not arrive leaves every owner waiting
    ("no_zero_arrival", True, {"unwound": {0}}, "deadlock"),
    # pulled: without the closing barrier a CTA tears down while others still read its staging
    ("no_closing_barrier", False, {}, "after it tore down"),
    # pulled: without the first barrier an owner reads staging not yet written
    ("no_first_barrier", False, {}, "before it was staged"),
])
def test_planted_exchange_hazards_are_caught(mutation, push, kw, expect):
    msg = caught(mutation, push, **kw)
    assert msg is not None and expect in msg, msg
