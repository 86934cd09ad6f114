"""Protocol model of the launches of the library's calls on one stream, for CPU tests.

A host-buffer call (mg_attn_run_host) enqueues a copy kernel (pinned host inputs -> the plan's
device staging) and the attention kernel (staging -> O, written straight into the pinned
output). A device call (mg_attn_run) enqueues the attention kernel alone, reading its inputs
where the caller keeps them. Every kernel is launched with programmatic dependent launch: a
kernel may start once every CTA of the kernel before it has released its dependents
(griddepcontrol.launch_dependents), and it passes its own griddepcontrol.wait only once that
kernel has completed, with its memory visible; every thread releases the dependents only after
its own wait, so a kernel completes only after its wait and the completions stay in stream order.

    copy kernel, early form:    load the inputs; wait; release dependents; store them into staging
    copy kernel, late form:     wait; release dependents; load the inputs; store them into staging
    attention kernel (host):    wait; release dependents; read staging; write O
    attention kernel (device),
      level 2:                  release dependents; load the inputs; wait; write O
      level 1:                  load the inputs; wait; release dependents; write O
      level 0:                  wait; release dependents; load the inputs; write O

A kernel at level 2 releases its dependents at its start, so the kernels after it may start (and
load) while kernels before it still run; the device holds fewer than W = 16 of them at once
(grids of more than SMs / 16 CTAs, one per SM), which the model, without resources, takes as a bound on
the calls it runs. The early forms (copy early, device levels 1 and 2) are used unless an input
shares bytes with the call's own O or with the O of one of the last W calls on the stream, or
the call is the first on the stream (its previous kernel unknown); level 2 only for calls of
kind "device" (large grids), level 1 for "device_small". A call of kind "device_split" is a
level-2-capable device call whose split partials go through the plan's workspace: its fused
kernel writes them (after its wait) and a second kernel sums them into O:

    combine kernel:             (after a level-2 fused kernel) release dependents; wait; read the
                                workspace; write O.  Otherwise: wait; release dependents; ... The caller writes a call's inputs before it
enqueues the call. The scheduler interleaves the kernels' steps at random within those rules and
checks every read: staging is read only after the copy that filled it for this call has
completed, staging is not overwritten while an earlier call still reads it, and every input read
sees the value written for that call (an input that is an earlier call's O must be read after
that call's attention kernel wrote it).
"""

from __future__ import annotations

import random


class ProtocolError(AssertionError):
    pass


class StreamSim:
    def __init__(self, calls, seed: int, mutations=()):
        """calls: list of (inputs, output) or (inputs, output, kind) buffer names, kind "host"
        (the default), "device" or "device_small", e.g. [("x0", "o0"), ("o0", "o1", "device")]
        (the second call reads the first call's output)."""
        calls = [c if len(c) == 3 else (c[0], c[1], "host") for c in calls]
        self.calls = calls
        self.rng = random.Random(seed)
        self.mut = set(mutations)
        self.version = {}        # buffer -> which call's value it holds ("host" for host-written inputs)
        self.staging = None      # (call, complete) of the staged inputs
        self.staging_readers = set()
        self.ws_readers = set()       # combine kernels reading the plan's workspace
        self.kernels = []        # in stream order: dicts with name, state
        W = 16
        for k, (inp, out, kind) in enumerate(calls):
            # The entry points' rule: load early unless the input is this call's output or the
            # output of one of the last W calls on the stream, or the call is the stream's first
            # (mutations: no rule, the own output only, the previous call's output only).
            recent = [c[1] for c in calls[max(0, k - W):k]]
            if "early_despite_alias" in self.mut:
                early = True
            elif "alias_own_only" in self.mut:
                early = inp != out
            elif "window_1" in self.mut:
                early = k > 0 and inp != out and inp != calls[k - 1][1]
            else:
                early = k > 0 and inp != out and inp not in recent
            if kind == "host":
                self.kernels.append({"name": f"copy{k}", "call": k, "kind": "copy", "early": early,
                                     "inp": inp, "out": out})
                self.kernels.append({"name": f"attn{k}", "call": k, "kind": "attn", "inp": inp, "out": out})
            else:
                level = (2 if kind in ("device", "device_split") else 1) if early else 0
                split = kind == "device_split"
                self.kernels.append({"name": f"dattn{k}", "call": k, "kind": "dattn", "early": early,
                                     "level": level, "inp": inp, "out": "ws" if split else out})
                if split:
                    self.kernels.append({"name": f"comb{k}", "call": k, "kind": "comb",
                                         "level": level, "inp": "ws", "out": out})
        for kern in self.kernels:
            kern.update(started=False, triggered=False, waited=False, done=False)
        # the host wrote every call's inputs before enqueueing it; an input that is an earlier call's
        # output is expected to hold that call's value
        self.expect = {}
        writer = {}
        for k, (inp, out, _) in enumerate(calls):
            self.expect[k] = writer.get(inp, "host")
            writer[out] = k
        for inp, _, _ in calls:
            self.version.setdefault(inp, "host")

    # ---------------------------------------------------------------- kernel bodies
    def _prev(self, i):
        return self.kernels[i - 1] if i > 0 else None

    def _may_start(self, i):
        prev = self._prev(i)
        return prev is None or prev["triggered"] or prev["done"]

    def _may_pass_wait(self, i):
        prev = self._prev(i)
        return prev is None or prev["done"]

    def _store(self, k, loaded):
        if loaded != self.expect[k]:
            raise ProtocolError(f"copy{k} loaded an input holding {loaded!r}, not {self.expect[k]!r}")
        if self.staging_readers:
            raise ProtocolError(f"copy{k} overwrites staging while {sorted(self.staging_readers)} read it")
        self.staging = (k, False)

    def body(self, i):
        kern = self.kernels[i]
        while not self._may_start(i):
            yield
        kern["started"] = True
        k = kern["call"]
        if kern["kind"] == "dattn":
            loaded = None
            if kern["level"] == 2:
                kern["triggered"] = True  # the dependents released at the start
                yield
            if kern["early"]:
                loaded = self.version.get(kern["inp"])
                yield
            while not self._may_pass_wait(i):
                yield
            kern["waited"] = True
            kern["triggered"] = True
            yield
            if loaded is None:
                loaded = self.version.get(kern["inp"])
                yield
            if loaded != self.expect[k]:
                raise ProtocolError(f"dattn{k} loaded an input holding {loaded!r}, not {self.expect[k]!r}")
            if kern["out"] == "ws" and self.ws_readers:
                raise ProtocolError(f"dattn{k} writes the workspace while {sorted(self.ws_readers)} read it")
            self.version[kern["out"]] = k
        elif kern["kind"] == "comb":
            if kern["level"] == 2:
                kern["triggered"] = True
                yield
            if "combine_no_wait" not in self.mut:
                while not self._may_pass_wait(i):
                    yield
            kern["waited"] = True
            kern["triggered"] = True
            yield
            if self.version.get("ws") != k:
                raise ProtocolError(f"comb{k} reads the workspace holding {self.version.get('ws')!r}")
            self.ws_readers.add(k)
            yield
            self.ws_readers.discard(k)
            self.version[kern["out"]] = k
            if "combine_no_wait" in self.mut:
                while not self._may_pass_wait(i):  # completion still in stream order
                    yield
        elif kern["kind"] == "copy":
            loaded = None
            if kern["early"]:
                loaded = self.version.get(kern["inp"])
                yield
            if "store_before_wait" in self.mut and loaded is not None:
                self._store(k, loaded)
                yield
            while not self._may_pass_wait(i):
                yield
            kern["waited"] = True
            kern["triggered"] = True
            yield
            if loaded is None:
                loaded = self.version.get(kern["inp"])
                yield
            if "store_before_wait" not in self.mut or not kern["early"]:
                self._store(k, loaded)
                yield
            self.staging = (k, True)
        else:
            if "attn_no_wait" in self.mut:
                kern["triggered"] = True
            else:
                while not self._may_pass_wait(i):
                    yield
                kern["waited"] = True
                kern["triggered"] = True
            yield
            if self.staging != (k, True):
                raise ProtocolError(f"attn{k} reads staging holding {self.staging!r}")
            self.staging_readers.add(k)
            yield
            self.staging_readers.discard(k)
            self.version[kern["out"]] = k
        if "attn_no_wait" in self.mut and kern["kind"] == "attn":
            while not self._may_pass_wait(i):  # completion still in stream order
                yield
        kern["done"] = True

    # ---------------------------------------------------------------- scheduler
    def run(self, max_steps: int = 100000):
        actors = {i: self.body(i) for i in range(len(self.kernels))}
        for _ in range(max_steps):
            if not actors:
                return self
            i = self.rng.choice(list(actors))
            try:
                next(actors[i])
            except StopIteration:
                del actors[i]
        raise ProtocolError(f"deadlock: {sorted(self.kernels[i]['name'] for i in actors)}")
