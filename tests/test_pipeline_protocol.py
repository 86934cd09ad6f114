"""CPU checks of the fused kernel's mbarrier protocol through its model (tests/pipeline_model.py).

The model restates, role by role, every barrier wait, arrival, commit and copy of
mg_attn_fwd_partial, and explores random interleavings of the roles with asynchronous copy and
tensor-pipe completion. The protocol as built must pass for every variant and for the ring
depths and P-buffer counts the plans use; each planted reordering must be caught in some
interleaving. One of them is the ordering that faulted a GPU when an A/B copy of the kernel
tried it: the P.V warp waiting for V before P in the two-pass variants.
"""

import itertools

import pytest

from tests import pipeline_model as pm

VARIANTS = {"plain": pm.PLAIN, "max-subtracted": pm.SAFE, "qk-norm": pm.QKNORM}
# (stages, P buffers): d = 64 plans use 2..6 stages and 3 P buffers, d = 128 plans 2..3 and 2.
RINGS = [(6, 3), (5, 3), (4, 3), (3, 3), (2, 3), (3, 2), (2, 2)]


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("stages,pbufs", RINGS)
def test_protocol_as_built_is_clean(variant, stages, pbufs):
    for T, seed in itertools.product((1, 2, 3, 4, 7, 12), range(12)):
        pm.Sim(T, stages, pbufs, VARIANTS[variant], seed).run()


def caught(mutation, variant, tries=40):
    for T, (stages, pbufs), seed in itertools.product((1, 2, 3, 5, 8), [(6, 3), (3, 2)], range(tries)):
        try:
            pm.Sim(T, stages, pbufs, variant, seed, mutations=(mutation,)).run()
        except pm.ProtocolError as e:
            return str(e)
    return None


@pytest.mark.parametrize("variant", ["max-subtracted", "qk-norm"])
def test_pv_warp_waiting_for_v_first_passes_a_parity_wait_early(variant):
    msg = caught("pv_waits_v_first", VARIANTS[variant])
    assert msg is not None and "VFull" in msg and "passed with" in msg


def test_pv_warp_waits_for_v_first_only_without_the_row_maximum_pass():
    # As built, the graph as written waits for V first (every V phase completes on a copy the
    # P.V warp has waited for in order); the clean runs above cover it. The two-pass variants
    # wait for P first, and forcing V first there is caught (the test above).
    assert caught("pv_waits_v_first", pm.PLAIN, tries=20) is None


@pytest.mark.parametrize("mutation,variant", [
    ("s_no_sempty_wait", pm.PLAIN),             # S written while the softmax group reads it
    ("producer_no_kvempty_wait", pm.PLAIN),     # K/V stage refilled while an MMA reads it
    ("qk_kvempty_before_barrier", pm.QKNORM),   # K stage released before every warp summed it
    # Key scales read before the other group wrote them. With several tiles per split the
    # in-order S issue orders this hand-off as well; with one tile per split (a row-maximum
    # step for group 0, the main-pass step for group 1) only the maximum exchange's barriers do.
    ("no_max_exchange", pm.QKNORM),
])
def test_planted_hazards_are_caught(mutation, variant):
    assert caught(mutation, variant) is not None


@pytest.mark.parametrize("variant", list(VARIANTS))
def test_unwinding_from_any_wait_is_clean(variant):
    # A bounded wait may run out anywhere (here: a random blocked wait at a random moment).
    # Every role must then unwind without waiting on a peer that left, and nothing the CTA
    # issued (copies, MMAs, commits) may still be in flight when it tears down.
    for T, (stages, pbufs), seed in itertools.product((1, 2, 3, 5, 8), [(6, 3), (3, 2), (2, 2)], range(12)):
        pm.Sim(T, stages, pbufs, VARIANTS[variant], seed, abort_rate=0.02).run()


def test_draining_only_after_a_failed_loop_leaves_mmas_in_flight():
    # The S warp once drained its MMAs only when its own loop failed, and the P.V warp not when
    # its tail waits failed: an abort raised elsewhere after those loops could free tensor
    # memory under a running MMA.
    hit = None
    for T, (stages, pbufs), seed in itertools.product((2, 3, 5, 8), [(6, 3), (3, 2)], range(60)):
        try:
            pm.Sim(T, stages, pbufs, pm.PLAIN, seed, mutations=("drain_only_on_failure",), abort_rate=0.01).run()
        except pm.ProtocolError as e:
            hit = str(e)
            break
    assert hit is not None and "in flight" in hit


def test_barrier_parity_semantics():
    # The model's parity test is the hardware's: phase k is seen as complete when the open
    # phase's parity differs from k's, which is also true while phase k - 1 is still open.
    b = pm.Barrier("x", 1)
    assert not b.test(0)          # phase 0 open
    b.arrive()
    assert b.test(0) and not b.test(1)
    b.arrive()
    assert b.test(1) and not b.test(0)
    with pytest.raises(pm.ProtocolError):
        c = pm.Barrier("y", 1)
        c.arrive(expect_tx=4)
        c.complete_tx(8)


# ------------------------------------------------------------------ two-Q-tile kernel

@pytest.mark.parametrize("stages", [2, 3, 4, 5, 6])
def test_pair_protocol_as_built_is_clean(stages):
    for T, seed in itertools.product((1, 2, 3, 4, 7, 12), range(12)):
        pm.PairSim(T, stages, seed).run()


def caught_pair(mutation, tries=40):
    for T, stages, seed in itertools.product((1, 2, 3, 5, 8), (6, 3, 2), range(tries)):
        try:
            pm.PairSim(T, stages, seed, mutations=(mutation,)).run()
        except pm.ProtocolError as e:
            return str(e)
    return None


@pytest.mark.parametrize("mutation,expect", [
    ("pair_s_no_sempty_wait", "writes S buffer"),       # S of the next tile over the one being read
    ("pair_no_pempty_wait", "overwritten"),             # P rewritten before the previous P.V read it
    ("pair_kvempty_after_pv0", "overwritten"),          # stage released while the second P.V reads V
    ("producer_no_kvempty_wait", "stage"),
])
def test_pair_planted_hazards_are_caught(mutation, expect):
    msg = caught_pair(mutation)
    assert msg is not None and expect in msg, msg


def test_pair_unwinding_from_any_wait_is_clean():
    for T, stages, seed in itertools.product((1, 2, 3, 5, 8), (6, 3, 2), range(12)):
        pm.PairSim(T, stages, seed, abort_rate=0.02).run()


def test_pair_draining_only_after_a_failed_loop_leaves_mmas_in_flight():
    hit = None
    for T, stages, seed in itertools.product((1, 2, 3, 5, 8), (6, 3, 2), range(60)):
        try:
            pm.PairSim(T, stages, seed, mutations=("drain_only_on_failure",), abort_rate=0.1).run()
        except pm.ProtocolError as e:
            hit = str(e)
            break
    assert hit is not None and "in flight" in hit


# ------------------------------------------------------------------ stream-K segments

SEGMENTS = [[1], [3], [1, 1], [2, 1], [1, 2], [5, 4], [7, 9], [1, 12], [13, 1], [3, 3]]


@pytest.mark.parametrize("stages,pbufs", [(6, 3), (3, 3), (3, 2), (2, 2)])
def test_segment_protocol_as_built_is_clean(stages, pbufs):
    for segs, seed in itertools.product(SEGMENTS, range(10)):
        pm.SegmentSim(segs, stages, pbufs, seed).run()


def test_segment_protocol_is_clean_when_any_role_lags():
    # Adversarial schedules: one role is seldom picked, so the others run far ahead of it.
    for segs, seed in itertools.product(([1, 1], [2, 2], [3, 1], [5, 4]), range(12)):
        for slow in ("softmax0", "softmax1", "pv_warp", "s_warp", "producer"):
            sim = pm.SegmentSim(segs, 3, 2, seed)
            sim.slow = (slow,)
            sim.run()


def test_segment_epilogue_needs_its_read_barrier():
    # Without the barrier that ends a segment's epilogue, the group that takes the next segment's
    # first tile can write its P, and that tile's P.V overwrite O, while the other group still
    # reads O: caught once that other group lags.
    hit = None
    for segs, seed in itertools.product(([1, 1], [2, 2], [3, 1]), range(10)):
        for slow in ("softmax0", "softmax1"):
            sim = pm.SegmentSim(segs, 3, 2, seed, mutations=("seg_no_read_barrier",))
            sim.slow = (slow,)
            try:
                sim.run()
            except pm.ProtocolError as e:
                hit = str(e)
                break
        if hit:
            break
    assert hit is not None and "overwrites O" in hit


def test_segment_needs_ofull_per_segment():
    with pytest.raises(pm.ProtocolError, match="deadlock"):
        pm.SegmentSim([2, 2], 3, 2, 0, mutations=("seg_no_ofull_per_segment",)).run()


def test_segment_unwinding_from_any_wait_is_clean():
    for segs, (stages, pbufs), seed in itertools.product(([2, 1], [1, 2], [3, 4], [1, 1], [4]), [(6, 3), (3, 2)],
                                                         range(12)):
        pm.SegmentSim(segs, stages, pbufs, seed, abort_rate=0.02).run()


# ------------------------------------------------------------------ few-row kernel
# The few-row kernel releases a stage's K and V halves on barriers of their own and issues K tile
# t + 2 before V tile t. Its QK-norm form also reads each K tile in the softmax warps (the key
# scales): there the K half is released once the S product has completed and every warp of the
# tile's group has read it.
SWAP_LEAD = 2
SWAP_FORMS = {
    "plain": dict(variant=pm.PLAIN, k_lead=SWAP_LEAD),
    "max-subtracted": dict(variant=pm.ONLINE, k_lead=SWAP_LEAD),
    "qk-norm": dict(variant=pm.ONLINE, k_lead=SWAP_LEAD, softmax_reads_k=True, k_softmax_release=True),
}


def swap_sim(form, T, stages, pbufs, seed, **kw):
    args = dict(SWAP_FORMS[form])
    args.update(kw)
    variant = args.pop("variant")
    return pm.Sim(T, stages, pbufs, variant, seed, **args)


@pytest.mark.parametrize("form", list(SWAP_FORMS))
@pytest.mark.parametrize("stages,pbufs", [(3, 3), (2, 3)])
def test_swap_protocol_as_built_is_clean(form, stages, pbufs):
    # The max-subtracted form adds, per tile, the group's rescale of its own O after the P.V
    # product of its previous tile (a wait on that tile's P-buffer barrier).
    for T, seed in itertools.product((1, 2, 3, 4, 7, 12), range(12)):
        swap_sim(form, T, stages, pbufs, seed).run()


@pytest.mark.parametrize("lead", [0, 1, 3, 4])
def test_swap_protocol_is_clean_for_other_k_leads(lead):
    # K released after S: any lead is free of deadlock (a K tile waits only for S products, which
    # need no V tile the producer has still to issue).
    for T, (stages, pbufs), seed in itertools.product((1, 3, 7, 12), [(3, 3), (2, 3)], range(6)):
        swap_sim("plain", T, stages, pbufs, seed, k_lead=lead).run()
        swap_sim("max-subtracted", T, stages, pbufs, seed, k_lead=lead).run()


def swap_caught(form, tries=40, **kw):
    for T, (stages, pbufs), seed in itertools.product((3, 5, 8), [(3, 3), (2, 3)], range(tries)):
        try:
            swap_sim(form, T, stages, pbufs, seed, **kw).run()
        except pm.ProtocolError as e:
            return str(e)
    return None


def test_swap_k_stage_refilled_without_its_wait_is_caught():
    msg = swap_caught("plain", mutations=("producer_no_kempty_wait",))
    assert msg is not None and "K stage" in msg


def test_swap_qk_norm_k_released_after_s_alone_is_caught():
    # The softmax warps read the K tile for the key scales: a release after S alone lets the
    # producer overwrite it under them.
    msg = swap_caught("qk-norm", k_softmax_release=False)
    assert msg is not None and "K stage" in msg


def test_swap_k_released_after_pv_with_a_lead_of_the_ring_depth_deadlocks():
    # Both halves released after P.V (an earlier form of the QK-norm kernel): a K tile issued
    # ring-depth tiles ahead waits for the P.V product of a tile whose V tile is queued behind it.
    msg = swap_caught("qk-norm", k_softmax_release=False, k_at_pv=True, k_lead=3)
    assert msg is not None and "deadlock" in msg
    for T, seed in itertools.product((3, 7), range(6)):
        swap_sim("qk-norm", T, 3, 3, seed, k_softmax_release=False, k_at_pv=True, k_lead=0).run()


def test_online_rescale_needs_its_wait():
    hit = None
    for T, (stages, pbufs), seed in itertools.product((3, 5, 8), [(3, 3), (2, 3)], range(60)):
        try:
            swap_sim("max-subtracted", T, stages, pbufs, seed, mutations=("online_no_rescale_wait",)).run()
        except pm.ProtocolError as e:
            hit = str(e)
            break
    assert hit is not None and "rescales its O" in hit


@pytest.mark.parametrize("form", list(SWAP_FORMS))
def test_swap_unwinding_from_any_wait_is_clean(form):
    for T, (stages, pbufs), seed in itertools.product((1, 2, 3, 5, 8), [(3, 3), (2, 3)], range(12)):
        swap_sim(form, T, stages, pbufs, seed, abort_rate=0.02).run()
