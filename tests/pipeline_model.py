"""Protocol model of the fused kernel's mbarrier pipeline (mg_attn_fwd_partial), for CPU tests.

The kernel's roles and every barrier operation they perform are restated here as Python
coroutines, in the kernel's order: the TMA producer, the S-issuing warp, the P.V-issuing warp
and the two groups of four softmax warps, for the graph as written, the max-subtracted variant
(a row-maximum pass over K first) and the QK-norm variant (whose softmax warps also read the K
tiles in that pass). Copies and tensor-core work complete asynchronously: a TMA copy at any
later moment, the tensor pipe's operations in issue order, a commit once every operation issued
before it has completed.

A scheduler runs the roles under random interleavings and checks, at every step:

* parity waits: an mbarrier wait passes only when the phase its caller means has just
  completed. The hardware test compares the barrier's current phase bit with the parity, so a
  wait on phase k while phase k-1 is still open passes early; a wait that falls two phases
  behind never passes (reported as a deadlock);
* unwinding: with `abort_rate`, a blocked wait may run out at any moment; every later wait
  whose phase has not completed then fails, as the kernel's bounded waits do once the CTA's
  abort flag is up, and the roles unwind as the kernel's do. No role may deadlock, and no copy
  or tensor-core operation may still be in flight when the CTA tears down;
* data hazards (when no abort): a copy lands in a K or V stage only when no operation still reads it; an MMA
  reads K, V and P only once the step's data is there and writes an S buffer only when its
  softmax group has finished reading it; the softmax warps read S only after its MMA and write
  a P buffer only after the P.V product of three (d = 64) or two (d = 128) tiles earlier;
  the epilogue reads O only after the last P.V product, and stages its output in the K/V
  ring only when no copy into it or MMA reading it is still in flight.

The model is a restatement, not the kernel: a change to the kernel's barrier protocol has to
be made here too. The mutations in tests/test_pipeline_protocol.py show that it catches the
hazards it is meant to (for example, the P.V warp waiting for V before P in the two-pass
variants).
"""

from __future__ import annotations

import random

PLAIN, SAFE, QKNORM, ONLINE = 0, 1, 2, 3
# ONLINE: the few-row kernel's max-subtracted form, in one pass. The protocol is the graph as
# written's, plus per tile t a rescale of the group's own O accumulator (O_g, g = t % 2) by the
# change of its running maxima, after the P.V product of the group's previous tile (t - 2) has
# completed and before P of tile t is announced.
GROUP_WARPS = 4
# Split release (`k_lead` set; the few-row kernel): a stage's K half and V half are released by
# barriers of their own, KEmpty (committed after the stage's S product, or with `k_at_pv` after
# its P.V product) and KvEmpty (after P.V); the producer issues K tile t + k_lead before V tile t.
# Where the softmax warps read the K tile too (`softmax_reads_k`, the QK-norm form), KEmpty also
# counts one arrival from each warp of the tile's group once it has read it (`k_softmax_release`).


class ProtocolError(AssertionError):
    pass


class Barrier:
    """An mbarrier: arrival count, transaction bytes and the number of completed phases."""

    def __init__(self, name: str, count: int):
        self.name = name
        self.count = count
        self.pending = count
        self.tx = 0
        self.completed = 0  # completed phases; the open phase has index `completed`

    def arrive(self, expect_tx: int = 0):
        self.tx += expect_tx
        self.pending -= 1
        if self.pending < 0:
            raise ProtocolError(f"{self.name}: more arrivals than its count in phase {self.completed}")
        self._maybe_complete()

    def complete_tx(self, nbytes: int):
        self.tx -= nbytes
        if self.tx < 0:
            raise ProtocolError(f"{self.name}: transaction bytes below zero in phase {self.completed}")
        self._maybe_complete()

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.completed += 1
            self.pending = self.count

    def test(self, parity: int) -> bool:
        # What the hardware's parity test sees: the open phase's parity differs from `parity`.
        return (self.completed & 1) != parity


class Sim:
    def __init__(self, T: int, stages: int, pbufs: int, variant: int, seed: int, mutations=(),
                 abort_rate: float = 0.0, k_lead=None, k_at_pv: bool = False, softmax_reads_k: bool = False,
                 k_softmax_release: bool = False):
        if T < 1 or stages < 2 or pbufs < 2:
            raise ValueError("T >= 1, stages >= 2, pbufs >= 2")
        if k_lead is not None and variant not in (PLAIN, ONLINE):
            raise ValueError("the split release is modelled for the one-pass forms")
        self.k_lead, self.k_at_pv, self.sm_reads_k = k_lead, k_at_pv, softmax_reads_k
        self.k_sm_release = k_softmax_release
        self.T, self.S, self.P, self.var = T, stages, pbufs, variant
        self.safe = variant in (SAFE, QKNORM)
        self.qk = variant == QKNORM
        self.online = variant == ONLINE
        self.T1 = T if self.safe else 0
        self.U = self.T1 + T
        self.mut = set(mutations)
        self.rng = random.Random(seed)
        self.abort_rate = abort_rate  # chance per step that a blocked wait runs out (0: never)
        self.slow = ()                # prefixes of actors the scheduler seldom picks (see run)
        self.abort = False
        self.bars = {}

        def mk(name, count):
            self.bars[name] = Barrier(name, count)

        mk("QFull", 1)
        for s in range(stages):
            mk(f"KFull{s}", 1)
            mk(f"VFull{s}", 1)
            mk(f"KvEmpty{s}", 1)
            if k_lead is not None:
                mk(f"KEmpty{s}", 1 + (GROUP_WARPS if k_softmax_release else 0))
        for g in range(2):
            mk(f"SFull{g}", 1)
            mk(f"SEmpty{g}", GROUP_WARPS)
        for p in range(pbufs):
            mk(f"PFull{p}", GROUP_WARPS)
            mk(f"PEmpty{p}", 1)
        mk("OFull", 1)
        # Buffer contents (the step or tile held, None while undefined) and their live readers.
        self.q_loaded = False
        self.kst = [None] * stages
        self.vst = [None] * stages
        self.k_readers = [0] * stages
        self.v_readers = [0] * stages
        self.sbuf = [None, None]
        self.s_readers = [0, 0]
        self.s_pending_write = [False, False]
        self.pbuf = [None] * pbufs          # tile whose P is complete in the buffer
        self.pieces = [set() for _ in range(pbufs)]
        self.p_tile_writing = [None] * pbufs
        self.p_readers = [0] * pbufs
        self.pv_done = 0
        self.pv_completed = set()           # tiles whose P.V product has completed
        self.o_rescaled = {0: set(), 1: set()}  # group -> tiles at which its O was rescaled
        self.pv_issued = 0
        self.scale_parts = {}               # QK-norm: tile -> softmax warps that wrote its key scales
        self.tma = []                       # in-flight copies: (barrier, bytes, effect)
        self.pipe = []                      # tensor pipe FIFO: ("mma", effect) or ("commit", barrier)
        self.gbar = {}                      # named barriers: id -> {"gen": n, "arrived": set()}
        self.gbar_wait = {}                 # actor -> (barrier id, generation it waits to end)
        self.actors = {}
        self._make_actors()

    # ------------------------------------------------------------------ checks
    def fail(self, msg):
        raise ProtocolError(msg)

    def wait(self, bar, parity, k, who):
        return ("wait", bar, parity, k, who)

    # ------------------------------------------------------------------ roles
    # A role yields ("wait", ...) and receives True, or False once the CTA is aborting and the
    # phase has not completed (the kernel's bounded wait); ("gbar", id, n, pred) receives the AND
    # of the participants' predicates; ("drain", kind) waits, ignoring the abort, until the
    # role's copies ("tma") or tensor-core operations ("pipe") have completed.
    def _producer(self):
        if self.k_lead is not None:
            yield from self._producer_split()
            return
        S = self.S
        ok = True
        yield ("do", lambda: self._tma_q())
        t = 0
        while ok and t < self.U:
            s = t % S
            rnd = t // S
            if t >= S and "producer_no_kvempty_wait" not in self.mut:
                if not (yield self.wait(f"KvEmpty{s}", (rnd & 1) ^ 1, rnd - 1, f"producer step {t}")):
                    ok = False
                    break
            yield ("do", lambda t=t, s=s: self._issue_step(t, s))
            t += 1
        if ok:
            for u in range(max(self.U - S, 0), self.U):
                ok = yield self.wait(f"KvEmpty{u % S}", (u // S) & 1, u // S, f"producer tail {u}")
                if not ok:
                    break
        if self.abort:
            yield ("drain", "tma")

    def _producer_split(self):
        S, U = self.S, self.U
        ok = True
        yield ("do", lambda: self._tma_q())
        tk = tv = 0
        while ok and tv < U:
            if tk < U and tk <= tv + self.k_lead:
                s, rnd = tk % S, tk // S
                if tk >= S and "producer_no_kempty_wait" not in self.mut:
                    if not (yield self.wait(f"KEmpty{s}", (rnd & 1) ^ 1, rnd - 1, f"producer K {tk}")):
                        ok = False
                        break
                yield ("do", lambda t=tk, s=s: self._issue_k(t, s))
                tk += 1
            else:
                s, rnd = tv % S, tv // S
                if tv >= S:
                    if not (yield self.wait(f"KvEmpty{s}", (rnd & 1) ^ 1, rnd - 1, f"producer V {tv}")):
                        ok = False
                        break
                yield ("do", lambda t=tv, s=s: self._issue_v(t, s))
                tv += 1
        if ok:
            for u in range(max(U - S, 0), U):
                ok = (yield self.wait(f"KEmpty{u % S}", (u // S) & 1, u // S, f"producer tail K {u}")) and \
                     (yield self.wait(f"KvEmpty{u % S}", (u // S) & 1, u // S, f"producer tail V {u}"))
                if not ok:
                    break
        if self.abort:
            yield ("drain", "tma")

    def _issue_k(self, t, s):
        if self.k_readers[s] and not self.abort:
            self.fail(f"K stage {s} overwritten for tile {t} while still read")
        self.kst[s] = None
        self.bars[f"KFull{s}"].arrive(expect_tx=1)
        self.tma.append((f"KFull{s}", 1, lambda: self.kst.__setitem__(s, t)))

    def _issue_v(self, t, s):
        if self.v_readers[s] and not self.abort:
            self.fail(f"V stage {s} overwritten for tile {t} while still read")
        self.vst[s] = None
        self.bars[f"VFull{s}"].arrive(expect_tx=1)
        self.tma.append((f"VFull{s}", 1, lambda: self.vst.__setitem__(s, t)))

    def _tma_q(self):
        self.bars["QFull"].arrive(expect_tx=1)
        self.tma.append(("QFull", 1, lambda: setattr(self, "q_loaded", True)))

    def _issue_step(self, t, s):
        if self.k_readers[s] and not self.abort:
            self.fail(f"K stage {s} overwritten for step {t} while still read")
        self.kst[s] = None
        kb = self.bars[f"KFull{s}"]
        kb.arrive(expect_tx=1)
        self.tma.append((f"KFull{s}", 1, lambda: self.kst.__setitem__(s, t)))
        vb = self.bars[f"VFull{s}"]
        if t < self.T1:
            vb.arrive()  # a row-maximum step loads no V
        else:
            if self.v_readers[s] and not self.abort:
                self.fail(f"V stage {s} overwritten for step {t} while still read")
            self.vst[s] = None
            vb.arrive(expect_tx=1)
            self.tma.append((f"VFull{s}", 1, lambda: self.vst.__setitem__(s, t)))

    def _s_warp(self):
        S = self.S
        ok = yield self.wait("QFull", 0, 0, "S warp Q")
        u = 0
        while ok and u < self.U:
            s, sb = u % S, u & 1
            if not (yield self.wait(f"KFull{s}", (u // S) & 1, u // S, f"S warp K {u}")):
                ok = False
                break
            if u >= 2 and "s_no_sempty_wait" not in self.mut:
                if not (yield self.wait(f"SEmpty{sb}", ((u >> 1) & 1) ^ 1, (u >> 1) - 1, f"S warp S buffer {u}")):
                    ok = False
                    break
            yield ("do", lambda u=u, s=s, sb=sb: self._issue_s(u, s, sb))
            u += 1
        if not ok or "drain_only_on_failure" not in self.mut:
            yield ("drain", "pipe")

    def _issue_s(self, u, s, sb):
        if not self.abort:
            if not self.q_loaded:
                self.fail(f"S MMA {u} issued before Q landed")
            if self.kst[s] != u:
                self.fail(f"S MMA {u} reads K stage {s} holding step {self.kst[s]}")
            if self.s_readers[sb]:
                self.fail(f"S MMA {u} writes S buffer {sb} while softmax warps read it")
        self.k_readers[s] += 1
        self.s_pending_write[sb] = True

        def done():
            self.k_readers[s] -= 1
            self.sbuf[sb] = u
            self.s_pending_write[sb] = False

        self.pipe.append(("mma", done))
        self.pipe.append(("commit", f"SFull{sb}"))
        if self.k_lead is not None and not self.k_at_pv:
            self.pipe.append(("commit", f"KEmpty{s}"))
        if not self.qk and u < self.T1:
            self.pipe.append(("commit", f"KvEmpty{s}"))

    def _pv_warp(self):
        S, P = self.S, self.P
        ok = True
        v = 0
        while ok and v < self.T:
            u = self.T1 + v
            pb, s = v % P, u % S
            w_p = self.wait(f"PFull{pb}", (v // P) & 1, v // P, f"PV warp P {v}")
            w_v = self.wait(f"VFull{s}", (u // S) & 1, u // S, f"PV warp V {v}")
            # As built: V first for the graph as written, P first in the two-pass variants.
            v_first = (not self.safe) or "pv_waits_v_first" in self.mut
            for w in ((w_v, w_p) if v_first else (w_p, w_v)):
                if not (yield w):
                    ok = False
                    break
            if not ok:
                break
            yield ("do", lambda v=v, u=u, pb=pb, s=s: self._issue_pv(v, u, pb, s))
            v += 1
        if ok:
            for t in range(max(self.T - P, 0), self.T):
                ok = yield self.wait(f"PEmpty{t % P}", (t // P) & 1, t // P, f"PV warp tail {t}")
                if not ok:
                    break
            if not ok and "drain_only_on_failure" not in self.mut:
                yield ("drain", "pipe")
        else:
            yield ("drain", "pipe")

    def _issue_pv(self, v, u, pb, s):
        if not self.abort:
            if self.pbuf[pb] != v:
                self.fail(f"P.V MMA {v} reads P buffer {pb} holding tile {self.pbuf[pb]}")
            if self.vst[s] != u:
                self.fail(f"P.V MMA {v} reads V stage {s} holding step {self.vst[s]}")
        self.p_readers[pb] += 1
        self.v_readers[s] += 1
        self.pv_issued += 1

        def done():
            self.p_readers[pb] -= 1
            self.v_readers[s] -= 1
            self.pv_done += 1
            self.pv_completed.add(v)

        self.pipe.append(("mma", done))
        self.pipe.append(("commit", f"KvEmpty{s}"))
        if self.k_lead is not None and self.k_at_pv:
            self.pipe.append(("commit", f"KEmpty{s}"))
        self.pipe.append(("commit", f"PEmpty{pb}"))
        if v == self.T - 1:
            self.pipe.append(("commit", "OFull"))

    def _softmax_warp(self, g, gw):
        S, P = self.S, self.P
        who = f"softmax g{g}w{gw}"
        ok = True
        if self.qk:
            ok = yield self.wait("QFull", 0, 0, who + " Q")
        # Row-maximum pass.
        if self.qk:
            # All four warps of the group run every iteration and vote at the first barrier.
            for u in range(g, self.T1, 2):
                s = u % S
                w_ok = ok and (yield self.wait(f"KFull{s}", (u // S) & 1, u // S, f"{who} K {u}"))
                if w_ok:
                    yield ("do", lambda s=s, u=u: self._read_k(s, u, +1))
                    yield ("do", lambda s=s: self._read_k(s, None, -1))
                    yield ("do", lambda u=u: self.scale_parts.setdefault(u, set()).add(gw))
                    if gw == 0 and "qk_kvempty_before_barrier" in self.mut:
                        # Mutation: the stage is released before the other warps have read K.
                        yield ("do", lambda s=s: self.bars[f"KvEmpty{s}"].arrive())
                w_ok = w_ok and (yield self.wait(f"SFull{g}", (u >> 1) & 1, u >> 1, f"{who} S {u}"))
                w_ok = yield ("gbar", f"group{g}", GROUP_WARPS, w_ok)
                if not w_ok:
                    ok = False
                    break
                if gw == 0 and "qk_kvempty_before_barrier" not in self.mut:
                    yield ("do", lambda s=s: self.bars[f"KvEmpty{s}"].arrive())
                yield ("do", lambda u=u: self._read_s(g, u, +1))
                yield ("do", lambda u=u: self._read_s(g, u, -1))
                yield ("do", lambda: self.bars[f"SEmpty{g}"].arrive())
                yield ("gbar", f"group{g}", GROUP_WARPS, True)
        else:
            u = g
            while ok and u < self.T1:
                if not (yield self.wait(f"SFull{g}", (u >> 1) & 1, u >> 1, f"{who} S {u}")):
                    ok = False
                    break
                yield ("do", lambda u=u: self._read_s(g, u, +1))
                yield ("do", lambda u=u: self._read_s(g, u, -1))
                yield ("do", lambda: self.bars[f"SEmpty{g}"].arrive())
                u += 2
        if self.safe and "no_max_exchange" not in self.mut:
            yield ("gbar", "softmax", 2 * GROUP_WARPS, True)
            yield ("gbar", "softmax", 2 * GROUP_WARPS, True)
        # Main pass.
        u = self.T1 if (self.T1 % 2 == g) else self.T1 + 1
        while ok and u < self.U:
            t = u - self.T1
            pb = t % P
            if self.sm_reads_k:
                # The few-row QK-norm form: the key scales from the K tile, before S is read.
                s = u % S
                if not (yield self.wait(f"KFull{s}", (u // S) & 1, u // S, f"{who} K {u}")):
                    ok = False
                    break
                yield ("do", lambda s=s, u=u: self._read_k(s, u, +1))
                yield ("do", lambda s=s: self._read_k(s, None, -1))
                if self.k_sm_release:
                    yield ("do", lambda s=s: self.bars[f"KEmpty{s}"].arrive())
            if not (yield self.wait(f"SFull{g}", (u >> 1) & 1, u >> 1, f"{who} S {u}")):
                ok = False
                break
            yield ("do", lambda u=u: self._read_s(g, u, +1))            # half 0 loaded
            if t >= P:
                if not (yield self.wait(f"PEmpty{pb}", ((t // P) & 1) ^ 1, t // P - 1, f"{who} P buffer {t}")):
                    ok = False
                    break
            if self.qk:
                yield ("do", lambda t=t: self._read_scales(t))
            yield ("do", lambda t=t, pb=pb: self._write_p(pb, t, (gw, 0)))
            yield ("do", lambda u=u: self._read_s(g, u, -1))            # half 1 loaded: S released
            yield ("do", lambda: self.bars[f"SEmpty{g}"].arrive())
            yield ("do", lambda t=t, pb=pb: self._write_p(pb, t, (gw, 1)))
            if self.online and t >= 2:
                # Rescale O_g once P.V of this group's previous tile has completed.
                q = t - 2
                if "online_no_rescale_wait" not in self.mut:
                    if not (yield self.wait(f"PEmpty{q % P}", (q // P) & 1, q // P, f"{who} O rescale {t}")):
                        ok = False
                        break
                yield ("do", lambda g=g, t=t: self._rescale_o(g, t))
            yield ("do", lambda pb=pb: self.bars[f"PFull{pb}"].arrive())
            u += 2
        # Epilogue: a vote on "O is ready" that every softmax warp takes part in.
        o_ok = ok and (yield self.wait("OFull", 0, 0, f"{who} O"))
        o_ready = yield ("gbar", "softmax", 2 * GROUP_WARPS, o_ok)
        if o_ready:
            yield ("do", lambda: self._read_o())

    def _rescale_o(self, g, t):
        if self.abort:
            return
        missing = [q for q in range(g, t, 2) if q not in self.pv_completed]
        if missing:
            self.fail(f"group {g} rescales its O at tile {t} while P.V of tile {missing[0]} is in flight")
        self.o_rescaled[g].add(t)

    def _read_k(self, s, u, delta):
        if delta > 0 and self.kst[s] != u and not self.abort:
            self.fail(f"QK-norm softmax reads K stage {s} holding step {self.kst[s]}, expected {u}")
        self.k_readers[s] += delta

    def _read_s(self, g, u, delta):
        if delta > 0 and (self.sbuf[g] != u or self.s_pending_write[g]) and not self.abort:
            self.fail(f"softmax group {g} reads S buffer holding step {self.sbuf[g]}, expected {u}")
        self.s_readers[g] += delta

    def _write_p(self, pb, t, piece):
        if self.abort:
            return
        if self.p_readers[pb]:
            self.fail(f"P buffer {pb} written for tile {t} while a P.V MMA reads it")
        if self.p_tile_writing[pb] != t:
            if self.pbuf[pb] is not None and self.pv_done <= self.pbuf[pb]:
                self.fail(f"P buffer {pb} overwritten for tile {t} before P.V of tile {self.pbuf[pb]}")
            self.p_tile_writing[pb] = t
            self.pieces[pb] = set()
            self.pbuf[pb] = None
        self.pieces[pb].add(piece)
        if len(self.pieces[pb]) == 2 * GROUP_WARPS:
            self.pbuf[pb] = t

    def _read_scales(self, t):
        # QK-norm main pass: tile t's key-vector scales were written to global memory in the
        # row-maximum pass (step t), by the four warps of whichever group took that step.
        if not self.abort and len(self.scale_parts.get(t, ())) != GROUP_WARPS:
            self.fail(f"main pass reads tile {t}'s key scales before all four warps wrote them")

    def _read_o(self):
        if self.pv_done != self.T:
            self.fail(f"O read after {self.pv_done} of {self.T} P.V products")
        # The epilogue stages its output in the K/V ring: no copy may still be landing there and
        # no MMA may still read it.
        if any(bar.startswith(("KFull", "VFull")) for bar, _, _ in self.tma):
            self.fail("output staged in the K/V ring while a copy into it is in flight")
        if any(self.k_readers) or any(self.v_readers):
            self.fail("output staged in the K/V ring while an MMA reads it")

    def _make_actors(self):
        self.actors["producer"] = self._producer()
        self.actors["s_warp"] = self._s_warp()
        self.actors["pv_warp"] = self._pv_warp()
        for g in range(2):
            for gw in range(GROUP_WARPS):
                self.actors[f"softmax{g}.{gw}"] = self._softmax_warp(g, gw)

    # ------------------------------------------------------------------ scheduler
    def _runnable(self, name, op):
        """(runnable, value sent back) for an actor's pending operation."""
        kind = op[0]
        if kind == "do":
            return True, None
        if kind == "wait":
            _, bar, parity, k, who = op
            if self.bars[bar].test(parity):
                return True, True
            return (True, False) if self.abort else (False, None)
        if kind == "gbar":
            _, gid, n, pred = op
            g = self.gbar.setdefault(gid, {"gen": 0, "arrived": {}, "result": {}})
            if name not in self.gbar_wait:
                return True, None
            gen = self.gbar_wait[name][1]
            return (g["gen"] > gen), g["result"].get(gen)
        if kind == "drain":
            return (not self.tma) if op[1] == "tma" else (not self.pipe), None
        raise ValueError(kind)

    def run(self, max_steps: int = 400000):
        gens = dict(self.actors)
        nxt = {name: next(gen) for name, gen in gens.items()}
        steps = 0
        while nxt or self.tma or self.pipe:
            steps += 1
            if steps > max_steps:
                self.fail("step limit")
            if not nxt:
                # Every role has finished: the CTA tears down (tensor memory freed, shared
                # memory released). Nothing may still be in flight.
                self.fail(f"teardown with {len(self.tma)} copies and {len(self.pipe)} tensor-pipe "
                          "operations in flight")
            # A bounded wait that runs out: some blocked wait times out and the CTA aborts.
            if self.abort_rate and not self.abort and self.rng.random() < self.abort_rate:
                blocked = [n for n, op in nxt.items() if op[0] == "wait" and not self._runnable(n, op)[0]]
                if blocked:
                    self.abort = True
            options = []
            for name, op in nxt.items():
                ready, _ = self._runnable(name, op)
                if ready:
                    options.append(("actor", name))
            options += [("tma", i) for i in range(len(self.tma))]
            if self.pipe:
                options.append(("pipe", 0))
            if not options:
                self.fail("deadlock: " + ", ".join(f"{n} at {op[0]} {op[1:3] if op[0] != 'do' else ''}"
                                                    for n, op in nxt.items()))
            if self.slow:
                # Actors named with a prefix in `slow` are picked rarely: an adversarial schedule in
                # which those roles lag far behind the others.
                w = [0.02 if k == "actor" and any(n.startswith(p) for p in self.slow) else 1.0 for k, n in options]
                kind, key = self.rng.choices(options, weights=w)[0]
            else:
                kind, key = self.rng.choice(options)
            if kind == "tma":
                bar, nbytes, effect = self.tma.pop(key)
                effect()
                self.bars[bar].complete_tx(nbytes)
                continue
            if kind == "pipe":
                op = self.pipe.pop(0)
                if op[0] == "mma":
                    op[1]()
                else:
                    self.bars[op[1]].arrive()
                continue
            name = key
            op = nxt[name]
            _, value = self._runnable(name, op)
            if op[0] == "do":
                op[1]()
            elif op[0] == "wait" and value:
                _, bar, parity, k, who = op
                b = self.bars[bar]
                if b.completed != k + 1:
                    self.fail(f"{who}: wait on {bar} for phase {k} passed with {b.completed} phases complete")
            elif op[0] == "gbar":
                _, gid, n, pred = op
                g = self.gbar[gid]
                if name not in self.gbar_wait:
                    # Arrive with a predicate; the last arrival ends this generation of the
                    # barrier and fixes the AND of the predicates.
                    gen = g["gen"]
                    self.gbar_wait[name] = (gid, gen)
                    g["arrived"][name] = bool(pred)
                    if len(g["arrived"]) == n:
                        g["result"][gen] = all(g["arrived"].values())
                        g["gen"] += 1
                        g["arrived"] = {}
                    if g["gen"] == gen:
                        continue  # stays at the barrier until the others arrive
                    value = g["result"][gen]
                else:
                    value = g["result"][self.gbar_wait[name][1]]
                del self.gbar_wait[name]
            try:
                nxt[name] = gens[name].send(value)
            except StopIteration:
                del nxt[name]
        return steps


class PairSim(Sim):
    """The two-Q-tile kernel (mg_attn_fwd_pair): each CTA holds two 128-row Q tiles of one batch
    and streams every K/V tile once for both. Softmax group g owns Q tile g, its S buffer g, its
    single P buffer g and its accumulator O_g; no row data passes between the groups. Per step t:
    the S warp issues S_0 and S_1 (each once its group has read the previous S out of its buffer),
    the P.V warp issues O_0 += P_0 V_t and O_1 += P_1 V_t (each once its group has written P), and
    the commit after the second one releases the K/V stage. Graph as written only (no row-maximum
    pass).

    Mutations: "pair_s_no_sempty_wait", "pair_no_pempty_wait" (P written before the previous P.V
    read it), "pair_kvempty_after_pv0" (the stage released after the first P.V), plus the base
    class's "producer_no_kvempty_wait" and "drain_only_on_failure"."""

    def __init__(self, T: int, stages: int, seed: int, mutations=(), abort_rate: float = 0.0):
        super().__init__(T, stages, 2, PLAIN, seed, mutations, abort_rate)
        self.pv_done_g = [0, 0]

    def _s_warp(self):
        S = self.S
        ok = yield self.wait("QFull", 0, 0, "S warp Q")
        t = 0
        while ok and t < self.T:
            s = t % S
            if not (yield self.wait(f"KFull{s}", (t // S) & 1, t // S, f"S warp K {t}")):
                ok = False
                break
            for g in range(2):
                if t >= 1 and "pair_s_no_sempty_wait" not in self.mut:
                    if not (yield self.wait(f"SEmpty{g}", (t - 1) & 1, t - 1, f"S warp S{g} buffer {t}")):
                        ok = False
                        break
                yield ("do", lambda t=t, s=s, g=g: self._issue_s_pair(t, s, g))
            t += 1
        if not ok or "drain_only_on_failure" not in self.mut:
            yield ("drain", "pipe")

    def _issue_s_pair(self, t, s, g):
        if not self.abort:
            if not self.q_loaded:
                self.fail(f"S MMA {t} issued before Q landed")
            if self.kst[s] != t:
                self.fail(f"S{g} MMA {t} reads K stage {s} holding step {self.kst[s]}")
            if self.s_readers[g]:
                self.fail(f"S{g} MMA {t} writes S buffer {g} while softmax warps read it")
        self.k_readers[s] += 1
        self.s_pending_write[g] = True

        def done():
            self.k_readers[s] -= 1
            self.sbuf[g] = t
            self.s_pending_write[g] = False

        self.pipe.append(("mma", done))
        self.pipe.append(("commit", f"SFull{g}"))

    def _pv_warp(self):
        S = self.S
        ok = True
        t = 0
        while ok and t < self.T:
            s = t % S
            if not (yield self.wait(f"VFull{s}", (t // S) & 1, t // S, f"PV warp V {t}")):
                ok = False
                break
            for g in range(2):
                if not (yield self.wait(f"PFull{g}", t & 1, t, f"PV warp P{g} {t}")):
                    ok = False
                    break
                yield ("do", lambda t=t, s=s, g=g: self._issue_pv_pair(t, s, g))
            t += 1
        if ok:
            for g in range(2):
                ok = yield self.wait(f"PEmpty{g}", (self.T - 1) & 1, self.T - 1, f"PV warp tail P{g}")
                if not ok:
                    break
            if not ok and "drain_only_on_failure" not in self.mut:
                yield ("drain", "pipe")
        else:
            yield ("drain", "pipe")

    def _issue_pv_pair(self, t, s, g):
        if not self.abort:
            if self.pbuf[g] != t:
                self.fail(f"P.V{g} MMA {t} reads P buffer {g} holding tile {self.pbuf[g]}")
            if self.vst[s] != t:
                self.fail(f"P.V{g} MMA {t} reads V stage {s} holding step {self.vst[s]}")
        self.p_readers[g] += 1
        self.v_readers[s] += 1
        self.pv_issued += 1

        def done():
            self.p_readers[g] -= 1
            self.v_readers[s] -= 1
            self.pv_done += 1
            self.pv_done_g[g] += 1

        self.pipe.append(("mma", done))
        self.pipe.append(("commit", f"PEmpty{g}"))
        if g == 1 or "pair_kvempty_after_pv0" in self.mut:
            if g == 0 or "pair_kvempty_after_pv0" not in self.mut:
                self.pipe.append(("commit", f"KvEmpty{s}"))
        if g == 1 and t == self.T - 1:
            self.pipe.append(("commit", "OFull"))

    def _softmax_warp(self, g, gw):
        who = f"softmax g{g}w{gw}"
        ok = True
        t = 0
        while ok and t < self.T:
            if not (yield self.wait(f"SFull{g}", t & 1, t, f"{who} S {t}")):
                ok = False
                break
            yield ("do", lambda t=t: self._read_s(g, t, +1))             # half 0 loaded
            if t >= 1 and "pair_no_pempty_wait" not in self.mut:
                if not (yield self.wait(f"PEmpty{g}", (t - 1) & 1, t - 1, f"{who} P buffer {t}")):
                    ok = False
                    break
            yield ("do", lambda t=t: self._write_p_pair(g, t, (gw, 0)))
            yield ("do", lambda t=t: self._read_s(g, t, -1))             # half 1 loaded: S released
            yield ("do", lambda: self.bars[f"SEmpty{g}"].arrive())
            yield ("do", lambda t=t: self._write_p_pair(g, t, (gw, 1)))
            yield ("do", lambda: self.bars[f"PFull{g}"].arrive())
            t += 1
        o_ok = ok and (yield self.wait("OFull", 0, 0, f"{who} O"))
        o_ready = yield ("gbar", "softmax", 2 * GROUP_WARPS, o_ok)
        if o_ready:
            yield ("do", lambda: self._read_o())

    def _write_p_pair(self, g, t, piece):
        if self.abort:
            return
        if self.p_readers[g]:
            self.fail(f"P buffer {g} written for tile {t} while a P.V MMA reads it")
        if self.p_tile_writing[g] != t:
            if self.pbuf[g] is not None and self.pv_done_g[g] <= self.pbuf[g]:
                self.fail(f"P buffer {g} overwritten for tile {t} before P.V of tile {self.pbuf[g]}")
            self.p_tile_writing[g] = t
            self.pieces[g] = set()
            self.pbuf[g] = None
        self.pieces[g].add(piece)
        if len(self.pieces[g]) == 2 * GROUP_WARPS:
            self.pbuf[g] = t

    def _read_o(self):
        if self.pv_done != 2 * self.T:
            self.fail(f"O read after {self.pv_done} of {2 * self.T} P.V products")
        if any(bar.startswith(("KFull", "VFull")) for bar, _, _ in self.tma):
            self.fail("output staged in the K/V ring while a copy into it is in flight")
        if any(self.k_readers) or any(self.v_readers):
            self.fail("output staged in the K/V ring while an MMA reads it")


class SegmentSim(Sim):
    """The one-tile kernel under a stream-K schedule (the graph as written): the CTA's steps form
    consecutive segments, each a run of column tiles of one row tile with its own Q tile (all loaded
    at the start, one barrier), its own row sums and its own partial. The two softmax groups still
    take alternate steps; after its last step of a segment each group joins that segment's epilogue,
    which waits for OFull's phase k (committed after the segment's last P.V), reads O, and ends with
    a barrier of all eight softmax warps. The first P.V of segment k+1 overwrites O (no accumulate):
    it needs P of that tile, which its group writes only after that barrier, so it cannot overtake
    the epilogue's reads and needs no barrier of its own.

    Mutations: "seg_no_read_barrier" (no barrier after the epilogue's reads), "seg_no_ofull_per_segment"
    (OFull committed only after the last segment), plus the base class's."""

    def __init__(self, seg_lengths, stages: int, pbufs: int, seed: int, mutations=(), abort_rate: float = 0.0):
        if not seg_lengths or min(seg_lengths) < 1:
            raise ValueError("segments of at least one step")
        self.segs = list(seg_lengths)
        super().__init__(sum(seg_lengths), stages, pbufs, PLAIN, seed, mutations, abort_rate)
        self.seg_of = []
        for k, n in enumerate(self.segs):
            self.seg_of += [k] * n
        self.seg_start = [sum(self.segs[:k]) for k in range(len(self.segs))]
        self.seg_last = [self.seg_start[k] + self.segs[k] - 1 for k in range(len(self.segs))]
        self.pv_done_seg = [0] * len(self.segs)
        self.o_reads = [0] * len(self.segs)   # softmax warps that finished reading segment k's O
        self.o_readers = 0                   # softmax warps reading O right now

    def _pv_warp(self):
        S, P = self.S, self.P
        ok = True
        v = 0
        while ok and v < self.T:
            k = self.seg_of[v]
            pb, s = v % P, v % S
            if not (yield self.wait(f"VFull{s}", (v // S) & 1, v // S, f"PV warp V {v}")):
                ok = False
                break
            if not (yield self.wait(f"PFull{pb}", (v // P) & 1, v // P, f"PV warp P {v}")):
                ok = False
                break
            yield ("do", lambda v=v, pb=pb, s=s, k=k: self._issue_pv_seg(v, pb, s, k))
            v += 1
        if ok:
            for t in range(max(self.T - P, 0), self.T):
                ok = yield self.wait(f"PEmpty{t % P}", (t // P) & 1, t // P, f"PV warp tail {t}")
                if not ok:
                    break
            if not ok and "drain_only_on_failure" not in self.mut:
                yield ("drain", "pipe")
        else:
            yield ("drain", "pipe")

    def _issue_pv_seg(self, v, pb, s, k):
        if not self.abort:
            if self.pbuf[pb] != v:
                self.fail(f"P.V MMA {v} reads P buffer {pb} holding tile {self.pbuf[pb]}")
            if self.vst[s] != v:
                self.fail(f"P.V MMA {v} reads V stage {s} holding step {self.vst[s]}")
            if v == self.seg_start[k] and k >= 1 and (self.o_readers or self.o_reads[k - 1] != 2 * GROUP_WARPS):
                self.fail(f"segment {k}'s first P.V overwrites O while segment {k - 1}'s epilogue reads it")
        self.p_readers[pb] += 1
        self.v_readers[s] += 1
        self.pv_issued += 1

        def done():
            self.p_readers[pb] -= 1
            self.v_readers[s] -= 1
            self.pv_done += 1
            self.pv_done_seg[k] += 1

        self.pipe.append(("mma", done))
        self.pipe.append(("commit", f"KvEmpty{s}"))
        self.pipe.append(("commit", f"PEmpty{pb}"))
        if v == self.seg_last[k] and ("seg_no_ofull_per_segment" not in self.mut or v == self.T - 1):
            n = 1 if "seg_no_ofull_per_segment" not in self.mut else len(self.segs)
            for _ in range(n):
                self.pipe.append(("commit", "OFull"))

    def _softmax_warp(self, g, gw):
        P = self.P
        who = f"softmax g{g}w{gw}"
        ok = True
        for k in range(len(self.segs)):
            for u in range(self.seg_start[k], self.seg_last[k] + 1):
                if u % 2 != g or not ok:
                    continue
                t = u
                pb = t % P
                if not (yield self.wait(f"SFull{g}", (u >> 1) & 1, u >> 1, f"{who} S {u}")):
                    ok = False
                    continue
                yield ("do", lambda u=u: self._read_s(g, u, +1))
                if t >= P:
                    if not (yield self.wait(f"PEmpty{pb}", ((t // P) & 1) ^ 1, t // P - 1, f"{who} P buffer {t}")):
                        ok = False
                        continue
                yield ("do", lambda t=t, pb=pb: self._write_p(pb, t, (gw, 0)))
                yield ("do", lambda u=u: self._read_s(g, u, -1))
                yield ("do", lambda: self.bars[f"SEmpty{g}"].arrive())
                yield ("do", lambda t=t, pb=pb: self._write_p(pb, t, (gw, 1)))
                yield ("do", lambda pb=pb: self.bars[f"PFull{pb}"].arrive())
            # Segment k's epilogue: every softmax warp votes (an unwound warp votes no).
            o_ok = ok and (yield self.wait("OFull", k & 1, k, f"{who} O of segment {k}"))
            o_ready = yield ("gbar", "softmax", 2 * GROUP_WARPS, o_ok)
            if o_ready:
                yield ("do", lambda k=k: self._read_o_seg(k, +1))
                yield ("do", lambda k=k: self._read_o_seg(k, -1))
                if "seg_no_read_barrier" not in self.mut:
                    yield ("gbar", "softmax", 2 * GROUP_WARPS, True)
            else:
                ok = False

    def _read_o_seg(self, k, delta):
        if self.abort:
            return
        if delta > 0 and self.pv_done_seg[k] != self.segs[k]:
            self.fail(f"segment {k}'s O read after {self.pv_done_seg[k]} of {self.segs[k]} P.V products")
        self.o_readers += delta
        if delta < 0:
            self.o_reads[k] += 1

    def _read_o(self):  # not used: each segment has its own epilogue
        pass
