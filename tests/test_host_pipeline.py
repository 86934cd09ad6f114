"""CPU checks of the launch protocol of the library's calls on one stream through its model
(tests/stream_model.py): back-to-back host-buffer and device calls, in-place chains, mixed
sequences, and planted orderings that break them."""

import itertools

import pytest

from tests import stream_model as sm

CHAINS = {
    "distinct": [("x0", "o0"), ("x1", "o1"), ("x2", "o2"), ("x3", "o3")],
    "same_buffers": [("x", "o")] * 4,
    "in_place": [("h", "h")] * 4,
    "chained": [("x", "a"), ("a", "b"), ("b", "c"), ("c", "d")],
    # device calls (mg_attn_run): the fused kernel loads its inputs early
    "device_distinct": [("x0", "o0", "device"), ("x1", "o1", "device"), ("x2", "o2", "device")],
    "device_chained": [("x", "a", "device"), ("a", "b", "device"), ("b", "c", "device"), ("c", "d", "device")],
    "device_in_place": [("h", "h", "device")] * 4,
    "mixed_chained": [("x", "a"), ("a", "b", "device"), ("b", "c"), ("c", "d", "device"), ("d", "e", "device")],
    # level 2 (dependents released at the start): a call reading the output of a call further back
    "device_skip": [("x0", "a", "device"), ("x1", "b", "device"), ("x2", "c", "device"), ("a", "d", "device"),
                    ("x3", "e", "device"), ("b", "f", "device")],
    "small_skip": [("x0", "a", "device_small"), ("x1", "b", "device_small"), ("a", "c", "device_small")],
    # partials through the workspace and a combine kernel, which releases the next call early too
    "split_chain": [("x0", "a", "device_split"), ("x1", "b", "device_split"), ("a", "c", "device_split"),
                    ("x2", "d", "device"), ("c", "e", "device_split")],
}


@pytest.mark.parametrize("chain", list(CHAINS))
def test_launch_protocol_as_built_is_clean(chain):
    for seed in range(300):
        sm.StreamSim(CHAINS[chain], seed).run()


def caught(chain, mutation, tries=600):
    for seed in range(tries):
        try:
            sm.StreamSim(CHAINS[chain], seed, mutations=(mutation,)).run()
        except sm.ProtocolError as e:
            return str(e)
    return None


def test_early_loads_need_the_alias_rule():
    # The next call's copy kernel loads its inputs before the previous call's attention kernel has
    # finished: an input that is that call's output (O fed back in place) would be read stale.
    # The entry point therefore keeps the loads after the wait when O shares bytes with an input.
    msg = caught("in_place", "early_despite_alias")
    assert msg is not None and "loaded an input" in msg


def test_chains_need_the_previous_output_in_the_rule():
    # A call whose input is the previous call's output (O of call k as Q of call k + 1, in other
    # buffers than its own O) is read stale if only the call's own O is compared with its inputs;
    # the entry point also compares them with the previous call's output on the stream.
    msg = caught("chained", "alias_own_only")
    assert msg is not None and "loaded an input" in msg
    assert caught("chained", "early_despite_alias") is not None


@pytest.mark.parametrize("mutation,expect", [
    ("attn_no_wait", "reads staging"),            # attention before its copy completed
    ("store_before_wait", "staging"),   # staging rewritten under (or before) the previous call's read
])
def test_planted_orderings_are_caught(mutation, expect):
    msg = caught("distinct", mutation)
    assert msg is not None and expect in msg, msg


@pytest.mark.parametrize("chain", ["device_chained", "device_in_place", "mixed_chained"])
def test_device_calls_need_the_alias_rule(chain):
    # The fused kernel of a device call loads Q, K and V before the previous kernel on the stream
    # has completed; a call that reads the previous call's output (or its own, in place) would
    # read it stale without the rule.
    msg = caught(chain, "early_despite_alias")
    assert msg is not None and "loaded an input" in msg, msg


def test_device_chains_need_the_previous_output_in_the_rule():
    msg = caught("device_chained", "alias_own_only")
    assert msg is not None and "loaded an input" in msg


def test_first_call_is_not_early():
    sim = sm.StreamSim(CHAINS["device_distinct"], 0)
    assert [k["early"] for k in sim.kernels] == [False, True, True]


def test_level2_needs_the_window():
    # With dependents released at the start, a call may run while calls further back than the
    # previous one still write; comparing the inputs with the previous call's output alone reads
    # stale data, the window of recent outputs does not.
    for seed in range(300):
        sm.StreamSim(CHAINS["device_skip"], seed).run()
    msg = caught("device_skip", "window_1")
    assert msg is not None and "loaded an input" in msg, msg


def test_level1_needs_only_the_previous_output():
    # Kernels that release their dependents after their own wait: the previous call's output is
    # the only one that can still be written, so the narrower comparison suffices there.
    for seed in range(300):
        sm.StreamSim(CHAINS["small_skip"], seed, mutations=("window_1",)).run()


def test_levels_as_chosen():
    sim = sm.StreamSim([("x0", "a", "device"), ("x1", "b", "device_small"), ("a", "c", "device")], 0)
    assert [k["level"] for k in sim.kernels] == [0, 1, 0]


def test_combine_kernel_released_early():
    # After a fused kernel that started early, the combine kernel releases the next call at its
    # start as well: the next fused kernel then runs beside this call's combine, and its writes
    # of the shared workspace still wait for the combine to complete.
    for seed in range(300):
        sm.StreamSim(CHAINS["split_chain"], seed).run()
    msg = caught("split_chain", "combine_no_wait")
    assert msg is not None and "workspace" in msg, msg
    msg = caught("split_chain", "window_1")
    assert msg is not None and "loaded an input" in msg, msg
