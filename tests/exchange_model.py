"""Protocol model of the on-chip combine's exchange between the CTAs of a thread-block cluster.

The fused kernels (mg_attn_fwd_partial, mg_attn_fwd_swap) combine the n split partials of a row
tile inside one cluster. Each CTA stages its partial in its own shared memory; rank o owns a
slice of the rows (or columns) and writes that slice of O. Two forms are restated here, with
every cluster barrier, mbarrier operation and store they perform, as coroutines per CTA role:

* pulled (the default): a cluster barrier (release/acquire) after staging, the owners' loads
  from every CTA's staging, a closing cluster barrier before any CTA exits;
* pushed (opt-in): the first half of a cluster barrier at the start (receive barriers
  initialised), its wait before the first store; asynchronous stores (st.async, from registers)
  of each row into its owner's receive slot, each completing its bytes on the owner's receive
  mbarrier at any later moment, and per warp and owner one arrival with the bytes sent (the
  model lumps a rank's warps into one arrival per owner: the barrier's count differs, its
  protocol does not); the
  owner's bounded wait on its receive barrier, its combine from the receive area, and a closing
  cluster barrier that each owner reaches only once its rows have landed (or, unwinding, after a
  bounded drain of the stores still on their way).

A CTA may be unwinding (its output was never complete: it stages nothing and sends only its
arrivals), and a bounded wait may run out at any moment once `abort_rate` is set. The scheduler
runs the roles of all CTAs under random interleavings and checks:

* a store writes its destination only while that CTA is alive (it has not passed the closing
  barrier and torn down); its data leaves from the sender's registers, so the sender may be gone;
* an owner reads a sender's slot (pushed) or staging (pulled) only once those bytes are there,
  and, when no CTA is unwinding and no wait ran out, every owner combines;
* nothing deadlocks: every role finishes.

The transaction count of an mbarrier may go below zero for a while (a store's bytes can land
before its sender's expect-tx arrival is counted); the phase completes when both the pending
arrivals and the count are zero. The mutations in tests/test_exchange_protocol.py show that the
model catches the hazards it is meant to.
"""

from __future__ import annotations

import random


class ProtocolError(AssertionError):
    pass


class TxBarrier:
    """One phase of an mbarrier with arrivals and transaction bytes (the receive barrier)."""

    def __init__(self, name: str, count: int):
        self.name, self.pending, self.tx, self.done = name, count, 0, False

    def arrive(self, expect_tx: int):
        if self.done:
            raise ProtocolError(f"{self.name}: arrival after its phase completed")
        self.pending -= 1
        self.tx += expect_tx
        if self.pending < 0:
            raise ProtocolError(f"{self.name}: more arrivals than its count")
        self._check()

    def complete_tx(self, nbytes: int):
        if self.done:
            raise ProtocolError(f"{self.name}: bytes landed after its phase completed")
        self.tx -= nbytes
        self._check()

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.done = True


class ClusterBarrier:
    """barrier.cluster: a phase completes once every thread (here: every role) has arrived."""

    def __init__(self, roles: int):
        self.roles, self.arrived, self.phase = roles, 0, 0

    def arrive(self):
        self.arrived += 1
        if self.arrived == self.roles:
            self.arrived = 0
            self.phase += 1


class ExchangeSim:
    ROLES_PER_CTA = 2  # the softmax warps (stage, send, combine) and the other warps

    def __init__(self, n: int, push: bool, seed: int, unwound=(), mutations=(), abort_rate: float = 0.0):
        self.n, self.push = n, push
        self.rng = random.Random(seed)
        self.unwound = set(unwound)   # CTAs whose output was never complete
        self.mut = set(mutations)
        self.abort_rate = abort_rate
        self.cbar = ClusterBarrier(n * self.ROLES_PER_CTA)
        self.recv = [TxBarrier(f"recv{o}", n) for o in range(n)]
        self.staged = [False] * n      # staging written (sender side)
        self.alive = [True] * n        # not yet torn down
        self.landed = [[False] * n for _ in range(n)]  # landed[o][r]: r's rows in o's receive slot
        self.stores = []               # in flight: (src, dst)
        self.combined = [False] * n
        self.timed_out = [False] * n
        self.bytes = lambda r, o: 3 + (r + o) % 2  # a sender's bytes for an owner (varies)

    # -------------------------------------------------------------- helpers for the roles
    def _barrier(self, k):
        # This role's k-th cluster barrier (k = 1, 2, ...): arrive, then wait for its phase.
        self.cbar.arrive()
        while self.cbar.phase < k:
            yield "cbar"

    def _store_lands(self, src, dst):
        if not self.alive[dst]:
            raise ProtocolError(f"store {src}->{dst} lands in CTA {dst} after it tore down")
        self.landed[dst][src] = True
        self.recv[dst].complete_tx(self.bytes(src, dst))

    def _wait_recv(self, o):
        # The bounded wait: passes once the phase completed; returns at once when the CTA is
        # unwinding, and may run out at any moment with abort_rate.
        if o in self.unwound:
            return False
        while not self.recv[o].done:
            if self.abort_rate and self.rng.random() < self.abort_rate:
                self.timed_out[o] = True
                return False
            yield "recv"
        return True

    def _send(self, r):
        for o in range(self.n):  # one sender thread per owner; their order does not matter
            if r in self.unwound:
                if "no_zero_arrival" not in self.mut:
                    self.recv[o].arrive(0)
            elif "stores_before_arrival" in self.mut:
                self.stores.append((r, o))
                yield "send"
                self.recv[o].arrive(self.bytes(r, o))
            else:
                self.recv[o].arrive(self.bytes(r, o))
                self.stores.append((r, o))
            yield "send"

    # -------------------------------------------------------------- roles
    def softmax(self, r):
        n = self.n
        if r not in self.unwound:
            self.staged[r] = True
        yield "staged"
        if self.push:
            # The prologue's arrival (receive barriers initialised) was made at the start; its
            # wait comes before the first store.
            while self.cbar.phase < 1:
                yield "cbar"
            yield from self._send(r)
            if "arrive_before_recv_wait" in self.mut:
                self.cbar.arrive()  # the closing barrier's arrival before the rows have landed
            got = True if "combine_without_wait" in self.mut else (yield from self._wait_recv(r))
            if got:
                for s in range(n):
                    # (an unwinding rank sends nothing: its slot is undefined, as is O then)
                    if not self.landed[r][s] and s not in self.unwound:
                        raise ProtocolError(f"owner {r} reads rank {s}'s slot before it landed")
                    yield "combine"
                self.combined[r] = True
            elif "no_drain_on_abort" not in self.mut:
                # the bounded drain of the stores still on their way in: every rank has issued
                # its stores and arrivals before any wait of its own
                while not self.recv[r].done:
                    yield "drain"
            if "arrive_before_recv_wait" in self.mut:
                while self.cbar.phase < 2:
                    yield "cbar"
            else:
                yield from self._barrier(2)
        else:
            k = 0
            if "no_first_barrier" not in self.mut:
                k += 1
                yield from self._barrier(k)
            for s in range(n):
                if not self.alive[s]:
                    raise ProtocolError(f"owner {r} reads the staging of CTA {s} after it tore down")
                if not self.staged[s] and s not in self.unwound:
                    raise ProtocolError(f"owner {r} reads the staging of CTA {s} before it was staged")
                yield "combine"
            self.combined[r] = True
            if "no_closing_barrier" not in self.mut:
                k += 1
                yield from self._barrier(k)
        self.alive[r] = False  # teardown (the CTA's other warps passed the same barriers)

    def others(self, r):
        # Warps 0, 1 and the P.V warp: the cluster barriers, nothing else.
        if self.push:
            while self.cbar.phase < 1:
                yield "cbar"
            yield from self._barrier(2)
        else:
            k = 0
            if "no_first_barrier" not in self.mut:
                k += 1
                yield from self._barrier(k)
            if "no_closing_barrier" not in self.mut:
                k += 1
                yield from self._barrier(k)

    # -------------------------------------------------------------- scheduler
    def run(self, max_steps: int = 200000):
        if self.push:
            for _ in range(self.n * self.ROLES_PER_CTA):  # the prologue's arrivals
                self.cbar.arrive()
        actors = {f"softmax{r}": self.softmax(r) for r in range(self.n)}
        actors.update({f"others{r}": self.others(r) for r in range(self.n)})
        for _ in range(max_steps):
            if not actors and not self.stores:
                break
            choices = list(actors) + (["store"] if self.stores else [])
            pick = self.rng.choice(choices)
            if pick == "store":
                src, dst = self.stores.pop(self.rng.randrange(len(self.stores)))
                self._store_lands(src, dst)
                continue
            try:
                next(actors[pick])
            except StopIteration:
                del actors[pick]
        else:
            raise ProtocolError(f"deadlock: {sorted(actors)} still waiting, {len(self.stores)} stores in flight")
        if not self.unwound and not any(self.timed_out) and not all(self.combined):
            raise ProtocolError("an owner did not combine although no CTA unwound")
        return self
