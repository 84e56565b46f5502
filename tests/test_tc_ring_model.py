"""A randomised model of the tcgen05 dq_gemm kernel's ring protocol, run on
the host: a weight-copy producer and an activation-copy producer fill the A
and activation rings slab after slab (each waits on a slot's "empty" barrier
before refilling it), two MMA issuers take alternate slabs (each waits on the
slot's "full" barriers, then commits the slot's "empty" barriers), and copies
land in random order. Barrier waits test only the parity of the phase they
wait for, as mbarrier.try_wait.parity does.

The kernel sizes both rings with an even number of slots so that each slot is
used by one issuer only; this model shows why: with an odd ring the issuer
running ahead waits on a slot two phases behind its barrier, and the parity
test lets it through on a copy that has not landed."""
import heapq
import random

import pytest


def _run(nas, nbs, nl, seed):
    rnd = random.Random(seed)
    done = {}  # completed phases per barrier
    for s in range(nas):
        done[("a_full", s)] = done[("a_empty", s)] = 0
    for s in range(nbs):
        done[("b_full", s)] = done[("b_empty", s)] = 0
    wrong = []

    def passes(bar, use):  # try_wait.parity(use & 1): true iff the completed-phase count's parity differs
        return (done[bar] & 1) != (use & 1)

    def complete(bar, use):
        if done[bar] != use:
            wrong.append(("phase completed out of order", bar, use, done[bar]))
        done[bar] += 1

    events, seq, now = [], 0, 0.0

    def later(dt, fn):
        nonlocal seq
        heapq.heappush(events, (now + dt, seq, fn))
        seq += 1

    nxt_w = nxt_b = 0
    nxt_issue = [0, 1]
    while True:
        moved = False
        if nxt_w < nl:  # weight producer
            s, u = nxt_w % nas, nxt_w // nas
            if u == 0 or passes(("a_empty", s), u - 1):
                later(rnd.expovariate(1.0) * (6.0 if rnd.random() < 0.1 else 1.0),
                      lambda s=s, u=u: complete(("a_full", s), u))
                nxt_w += 1
                moved = True
        if nxt_b < nl:  # activation producer
            s, u = nxt_b % nbs, nxt_b // nbs
            if u == 0 or passes(("b_empty", s), u - 1):
                later(rnd.expovariate(1.0) * (6.0 if rnd.random() < 0.1 else 1.0),
                      lambda s=s, u=u: complete(("b_full", s), u))
                nxt_b += 1
                moved = True
        for e in range(2):  # the two MMA issuers
            i = nxt_issue[e]
            if i < nl:
                sa, ua, sb, ub = i % nas, i // nas, i % nbs, i // nbs
                if passes(("a_full", sa), ua) and passes(("b_full", sb), ub):
                    if done[("a_full", sa)] != ua + 1 or done[("b_full", sb)] != ub + 1:
                        wrong.append(("wait passed on an earlier phase", e, i))
                    d = rnd.expovariate(2.0)
                    later(d, lambda sa=sa, ua=ua: complete(("a_empty", sa), ua))
                    later(d, lambda sb=sb, ub=ub: complete(("b_empty", sb), ub))
                    nxt_issue[e] += 2
                    moved = True
        if not moved:
            if not events:
                break
            now, _, fn = heapq.heappop(events)
            fn()
    finished = nxt_w == nl and nxt_b == nl and min(nxt_issue) >= nl
    return wrong, finished


@pytest.mark.parametrize("nas,nbs", [(4, 4), (6, 6), (8, 16), (10, 10), (12, 2), (4, 2)])
def test_even_rings_never_pass_a_wait_early(nas, nbs):
    for seed in range(150):
        wrong, finished = _run(nas, nbs, 96, seed)
        assert finished and not wrong, (seed, wrong[:3])


@pytest.mark.parametrize("nas,nbs", [(9, 16), (8, 3), (11, 11), (6, 5)])
def test_odd_rings_let_a_wait_pass_on_an_earlier_phase(nas, nbs):
    hits = sum(bool(_run(nas, nbs, 96, seed)[0]) for seed in range(150))
    assert hits > 0
