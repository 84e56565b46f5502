"""The synchronisation of the persistent tensor-core attention, checked on a
model (no GPU).

attn_tcp_kernel (csrc/attn.cu) runs eleven warps per CTA that meet only at
mbarriers: warp 0 takes units from the queue, publishes them in a two-slot
ring, loads Q and gathers K; warp 10 gathers V; one thread of warp 1 issues
the MMAs; eight softmax warps in two groups of four take the tiles of even and
odd (CTA-wide) index. Every wait polls one barrier for the completion of a
phase of given parity. Two ways to get this wrong do not show as wrong
numbers but as a wait that never ends (the kernel's bounded waits then give up
and flag an error):

  * a cycle of waits (a deadlock), and
  * a parity wait that polls its barrier only after it has completed two more
    phases: the parity then matches again and the wait misses its phase.

The model restates each role's sequence of arrivals, commits and waits, with
the kernel's barrier names, arrival counts and parities; copies (TMA) and MMA
commits complete asynchronously, commits in issue order as the tensor pipe
runs them. A random scheduler interleaves the roles over random unit lists
(empty units, one to eight tiles; one or two Q slots). The test asserts that
every run ends, and that every wait finds its barrier exactly one phase past
the phase it waits for. It also removes the MMA thread's one scheduling rule
that is not plain pipelining (issue the previous unit's last P V at once when
the queue yields an empty unit) and checks that the model then deadlocks: it
does on the GPU too.
"""
import random

import pytest

STAGES = 3  # K and V ring slots


class Barrier:
    def __init__(self, count: int, world) -> None:
        self.count, self.phases, self.arrivals, self.tx, self.world = count, 0, 0, 0, world

    def arrive(self) -> None:
        self.arrivals += 1
        self.world.version += 1
        self._complete()

    def _complete(self) -> None:
        if self.arrivals == self.count and self.tx == 0:
            self.phases += 1
            self.arrivals = 0


class Model:
    """One CTA of attn_tcp_kernel over the unit list ``units`` (tiles per unit)."""

    def __init__(self, units, q_slots: int, seed: int, flush_on_empty: bool = True) -> None:
        self.rng = random.Random(seed)
        self.units, self.nq, self.flush = units, q_slots, flush_on_empty
        self.version = 0
        b = {}
        for i in range(STAGES):
            for name in ("k_full", "k_empty", "v_full", "v_empty"):
                b[f"{name}{i}"] = Barrier(1, self)
        for i in range(2):
            b[f"s_full{i}"] = Barrier(1, self)
            b[f"p_full{i}"] = Barrier(4, self)   # the four warps of a softmax group
            b[f"pv_done{i}"] = Barrier(1, self)
            b[f"q_full{i}"] = Barrier(1, self)
            b[f"q_free{i}"] = Barrier(1, self)
            b[f"u_full{i}"] = Barrier(1, self)
            b[f"u_empty{i}"] = Barrier(10, self)  # MMA thread, eight softmax warps, V gather
        b["o_free"] = Barrier(4, self)    # the even group
        b["xm_full"] = Barrier(4, self)   # the odd group
        b["xm_empty"] = Barrier(4, self)  # the even group
        b["fin"] = Barrier(1, self)
        self.bars = b
        self.unit_slot = [None, None]
        self.copies = []    # barriers with a copy in flight
        self.commits = []   # MMA commits, completed in order
        self.ticket = 0
        self.faults = []

    # -- primitives --
    def wait(self, name: str, phase: int):
        """Wait for the completion of phase ``phase`` (0-based) by its parity."""
        bar = self.bars[name]
        while True:
            if bar.phases >= phase + 2:
                self.faults.append(f"{name}: waits for phase {phase}, barrier already {bar.phases} phases on")
                return
            if (bar.phases & 1) != (phase & 1):
                return
            yield name

    def copy(self, name: str) -> None:  # mbarrier.arrive.expect_tx + the TMA copies
        bar = self.bars[name]
        bar.tx += 1
        bar.arrive()
        self.copies.append(name)

    def commit(self, name: str) -> None:  # tcgen05.commit
        self.commits.append(name)

    def take_unit(self, k: int):
        yield from self.wait(f"u_full{k & 1}", k >> 1)
        u = self.unit_slot[k & 1]
        self.bars[f"u_empty{k & 1}"].arrive()
        return u

    # -- roles --
    def k_gather(self):
        J = qi = k = 0
        while True:
            if k >= 2:
                yield from self.wait(f"u_empty{k & 1}", (k >> 1) - 1)
            u = self.ticket if self.ticket < len(self.units) else -1
            self.ticket += 1
            self.unit_slot[k & 1] = u
            self.bars[f"u_full{k & 1}"].arrive()
            k += 1
            if u < 0:
                return
            if self.units[u] == 0:
                continue
            qs = qi % self.nq
            if qi >= self.nq:
                yield from self.wait(f"q_free{qs}", qi // self.nq - 1)
            self.copy(f"q_full{qs}")
            qi += 1
            for _ in range(self.units[u]):
                if J >= STAGES:
                    yield from self.wait(f"k_empty{J % STAGES}", (J - STAGES) // STAGES)
                self.copy(f"k_full{J % STAGES}")
                J += 1

    def v_gather(self):
        J = k = 0
        while True:
            u = yield from self.take_unit(k)
            k += 1
            if u < 0:
                return
            for _ in range(self.units[u]):
                if J >= STAGES:
                    yield from self.wait(f"v_empty{J % STAGES}", (J - STAGES) // STAGES)
                self.copy(f"v_full{J % STAGES}")
                J += 1

    def mma(self):
        J = qi = k = o_waits = 0
        pend, pend_wait = -1, False

        def pv(Jp, wait_o):
            nonlocal o_waits
            if wait_o:  # the first P V of a unit: the even group has read both accumulators
                yield from self.wait("o_free", o_waits)
                o_waits += 1
            yield from self.wait(f"p_full{Jp & 1}", Jp >> 1)
            yield from self.wait(f"v_full{Jp % STAGES}", Jp // STAGES)
            self.commit(f"v_empty{Jp % STAGES}")
            self.commit(f"pv_done{Jp & 1}")

        while True:
            u = yield from self.take_unit(k)
            k += 1
            if u < 0:
                break
            nt = self.units[u]
            if nt == 0:
                if self.flush and pend >= 0:
                    yield from pv(pend, pend_wait)
                    pend = -1
                continue
            qs = qi % self.nq
            yield from self.wait(f"q_full{qs}", qi // self.nq)
            for j in range(nt):
                yield from self.wait(f"k_full{J % STAGES}", J // STAGES)
                self.commit(f"k_empty{J % STAGES}")  # S of tile J
                self.commit(f"s_full{J & 1}")
                if j == nt - 1:
                    self.commit(f"q_free{qs}")
                if pend >= 0:
                    yield from pv(pend, pend_wait)
                pend, pend_wait = J, j == 0 and qi > 0
                J += 1
            qi += 1
        if pend >= 0:
            yield from pv(pend, pend_wait)
        self.commit("fin")
        yield from self.wait("fin", 0)

    def softmax_warp(self, grp: int):
        J = qi = k = 0
        while True:
            u = yield from self.take_unit(k)
            k += 1
            if u < 0:
                return
            nt = self.units[u]
            if nt == 0:
                continue
            J0, J = J, J + nt
            last = -1
            for Jt in range(J0 + ((J0 ^ grp) & 1), J, 2):
                yield from self.wait(f"s_full{grp}", Jt >> 1)
                if self.rng.random() < 0.3:  # a tile past the context: its V rows are zeroed
                    yield from self.wait(f"v_full{Jt % STAGES}", Jt // STAGES)
                if last >= 0:  # O of the group's previous tile before a rescale
                    yield from self.wait(f"pv_done{grp}", last >> 1)
                self.bars[f"p_full{grp}"].arrive()
                last = Jt
            if last >= 0:
                yield from self.wait(f"pv_done{grp}", last >> 1)
            if grp == 1:
                if qi >= 1:
                    yield from self.wait("xm_empty", qi - 1)
                self.bars["xm_full"].arrive()
            else:
                yield from self.wait("xm_full", qi)
                self.bars["xm_empty"].arrive()
                self.bars["o_free"].arrive()
            qi += 1

    def run(self) -> str:
        roles = {"k_gather": self.k_gather(), "v_gather": self.v_gather(), "mma": self.mma()}
        for w in range(8):
            roles[f"softmax{w}"] = self.softmax_warp(w // 4)
        blocked = {}  # role -> (barrier, model version when it blocked)
        while roles:
            pending = (["copy"] if self.copies else []) + (["commit"] if self.commits else [])
            if not pending and all(blocked.get(r, ("", -1))[1] == self.version for r in roles):
                return "deadlock: " + ", ".join(f"{r} waits {blocked[r][0]}" for r in sorted(roles))
            pick = self.rng.choice(list(roles) + pending * 3)
            if pick == "copy":
                bar = self.bars[self.copies.pop(self.rng.randrange(len(self.copies)))]
                bar.tx -= 1
                self.version += 1
                bar._complete()
            elif pick == "commit":
                self.bars[self.commits.pop(0)].arrive()
            else:
                try:
                    blocked[pick] = (next(roles[pick]), self.version)
                except StopIteration:
                    del roles[pick]
                    blocked.pop(pick, None)
                    self.version += 1
        return "ok"


def random_case(seed: int):
    rng = random.Random(seed)
    mix = rng.choice([[0, 1], [0, 0, 0, 1, 2], [1, 2, 3, 5, 8], [0, 1, 1, 2, 3, 5], [1], [0, 7]])
    return [rng.choice(mix) for _ in range(rng.randint(1, 24))], rng.choice([1, 2])


@pytest.mark.parametrize("block", range(6))
def test_every_schedule_ends_and_every_wait_meets_its_phase(block):
    for seed in range(block * 250, (block + 1) * 250):
        units, nq = random_case(seed)
        m = Model(units, nq, seed)
        result = m.run()
        assert result == "ok", f"units {units}, {nq} Q slot(s), seed {seed}: {result}"
        assert not m.faults, f"units {units}, {nq} Q slot(s), seed {seed}: {m.faults[:3]}"


def test_holding_the_last_pv_past_an_empty_unit_deadlocks():
    """Without the MMA thread's rule for empty units: a unit with tiles and
    then two empty ones deadlock on every schedule (the softmax warps wait in
    the first unit's epilogue for its last P V, the MMA thread for the next
    unit, and the queue for the softmax warps to take the second empty one)."""
    for seed in range(20):
        assert Model([1, 0, 0, 1], 2, seed, flush_on_empty=False).run().startswith("deadlock")
        assert Model([1, 0, 0, 1], 2, seed).run() == "ok"
