"""Pins for the oracle's speculative verify step.

Greedy verify (Algorithm 1 of the speculative-decoding energy notes): hand
cases for every first-mismatch position, ties, and out-of-range drafts; and
the notes' argument that greedy verification reproduces plain greedy
decoding, checked by running verify rounds against a synthetic deterministic
target with drafts that are sometimes right and comparing with token-by-token
greedy decoding of the same target.

Speculative sampling (CS336 notes §6): the worked exercise p = (0.2, 0.2, 0.6),
q = (0.5, 0.3, 0.2) (acceptance 0.6, residual (0.75, 0.25, 0), output
distribution q) and the two-token example, checked exactly by sweeping the
draft draw and both uniforms over stratified grids."""
from fractions import Fraction

import numpy as np
import pytest

from memory_bound_decode_dq_gb300 import synth


def _onehot_logits(tokens, V, base=None):
    """bf16 logits [len(tokens), V] whose argmax at row i is tokens[i]."""
    rng = np.random.default_rng(len(tokens) * 7 + V)
    lg = rng.standard_normal((len(tokens), V)).astype(np.float32) if base is None else base
    for i, t in enumerate(tokens):
        lg[i, t] = 10.0 + i
    return synth.f32_to_bf16_bits(lg)


@pytest.mark.parametrize("first_bad", [0, 1, 2, 3, None])
def test_greedy_accepts_the_matching_prefix(oracle_lib, first_bad):
    V, k = 50, 4
    target = [7, 3, 3, 41, 9]                       # t_0 .. t_4
    draft = list(target[:k])
    if first_bad is not None:
        draft[first_bad] = (draft[first_bad] + 1) % V
    lg = _onehot_logits(target, V)[None]
    out, cnt, ctx = oracle_lib.spec_verify_greedy(lg, np.array([draft]), np.array([100]))
    a = k if first_bad is None else first_bad
    assert cnt[0] == a + 1
    assert list(out[0, :a + 1]) == target[:a + 1]   # accepted drafts, then the target's token
    assert ctx[0] == 100 - (k - a)


def test_greedy_ties_and_bad_ids(oracle_lib):
    V = 8
    lg = np.zeros((1, 3, V), np.float32)
    lg[0, 0, [2, 5]] = 1.0                          # tie between 2 and 5: the smaller id
    lg[0, 1, 6] = 1.0
    lg[0, 2, 0] = 1.0
    out, cnt, _ = oracle_lib.spec_verify_greedy(synth.f32_to_bf16_bits(lg), np.array([[2, 6]]))
    assert cnt[0] == 3 and list(out[0]) == [2, 6, 0]
    out, cnt, _ = oracle_lib.spec_verify_greedy(synth.f32_to_bf16_bits(lg), np.array([[2 + V, 6]]))
    assert cnt[0] == 1 and out[0, 0] == 2             # an id outside the vocabulary never matches


def test_greedy_verify_reproduces_plain_greedy_decoding(oracle_lib):
    """Rounds of draft + verify against a deterministic target emit exactly
    the tokens that plain greedy decoding of that target emits."""
    V, k, steps = 97, 5, 60

    def target_next(prefix):                        # the target's greedy choice after prefix
        h = 1469598103
        for t in prefix:
            h = (h * 16777619 + t + 1) % 1000003
        return h % V

    start = [11]
    plain = list(start)
    while len(plain) < len(start) + steps:
        plain.append(target_next(plain))

    rng = np.random.default_rng(0)
    seq = list(start)
    rounds = 0
    while len(seq) < len(start) + steps:
        # draft: right with probability 0.7 at each position, else a random token
        d, pref = [], list(seq)
        for _ in range(k):
            t = target_next(pref) if rng.random() < 0.7 else int(rng.integers(V))
            d.append(t)
            pref.append(t)
        # the verify forward: position i sees the round's input and d_1..d_i (causal)
        block = [target_next(seq + d[:i]) for i in range(k + 1)]
        out, cnt, _ = oracle_lib.spec_verify_greedy(_onehot_logits(block, V)[None], np.array([d]))
        seq.extend(int(t) for t in out[0, :cnt[0]])
        rounds += 1
    assert seq[:len(plain)] == plain
    assert rounds < steps                               # some rounds emitted several tokens


def _stratified_outputs(oracle_lib, p, q, n_x, n_u):
    """Sweep the draft draw x ~ p (inverse CDF on an n_x grid of midpoints)
    and both uniforms (n_u midpoints each; grids chosen so that every
    probability of the example is a whole number of grid cells and no
    midpoint sits on a boundary); return the exact output distribution over
    the sweep as Fractions."""
    V = len(p)
    cp = np.cumsum(p)
    xs = [int(np.searchsorted(cp, (i + 0.5) / n_x, side="right")) for i in range(n_x)]
    us = [(i + 0.5) / n_u for i in range(n_u)]
    P = np.array(p, np.float32)[None, None, :]
    Q = np.array([q, q], np.float32)[None, :, :]      # position 1 (extra token) also q
    counts = np.zeros(V, np.int64)
    xx, ua, us_ = np.meshgrid(np.array(xs), np.array(us), np.array(us), indexing="ij")
    n = xx.size
    out, cnt, _ = oracle_lib.spec_verify_sample(np.broadcast_to(P, (n, 1, V)), np.broadcast_to(Q, (n, 2, V)),
                                                xx.reshape(n, 1), ua.reshape(n, 1).astype(np.float32),
                                                us_.reshape(n).astype(np.float32))
    first = out[:, 0]
    for t in range(V):
        counts[t] = int(np.sum(first == t))
    accepted = int(np.sum(cnt == 2))
    return [Fraction(int(c), n) for c in counts], Fraction(accepted, n)


def test_exercise_three_tokens(oracle_lib):
    p, q = [0.2, 0.2, 0.6], [0.5, 0.3, 0.2]
    dist, acc = _stratified_outputs(oracle_lib, p, q, 50, 24)
    assert acc == Fraction(3, 5)                                    # sum min(p, q) = 0.6
    assert dist == [Fraction(1, 2), Fraction(3, 10), Fraction(1, 5)]  # the output is distributed as q


def test_residual_of_the_exercise(oracle_lib):
    """A rejected draft resamples from norm(max(q - p, 0)) = (0.75, 0.25, 0)."""
    p, q = [0.2, 0.2, 0.6], [0.5, 0.3, 0.2]
    n = 400
    us = (np.arange(n) + 0.5) / n
    P = np.broadcast_to(np.array(p, np.float32), (n, 1, 3))
    Q = np.broadcast_to(np.array([q, q], np.float32), (n, 2, 3))
    # draft token 2 with u_accept 0.999: rejected (0.999 * 0.6 >= 0.2)
    out, cnt, _ = oracle_lib.spec_verify_sample(P, Q, np.full((n, 1), 2), np.full((n, 1), 0.999, np.float32),
                                                us.astype(np.float32))
    assert np.all(cnt == 1)
    assert np.mean(out[:, 0] == 0) == 0.75 and np.mean(out[:, 0] == 1) == 0.25


def test_two_token_example(oracle_lib):
    """Vocabulary {A, B}, the draft overestimates A: the residual is [0, 1]."""
    p, q = [0.8, 0.2], [0.6, 0.4]
    n = 200
    us = ((np.arange(n) + 0.5) / n).astype(np.float32)
    P = np.broadcast_to(np.array(p, np.float32), (n, 1, 2))
    Q = np.broadcast_to(np.array([q, q], np.float32), (n, 2, 2))
    out, cnt, _ = oracle_lib.spec_verify_sample(P, Q, np.zeros((n, 1)), np.full((n, 1), 0.9, np.float32), us)
    assert np.all(cnt == 1) and np.all(out[:, 0] == 1)      # rejected A always resamples B
    dist, acc = _stratified_outputs(oracle_lib, p, q, 50, 24)
    assert dist == [Fraction(3, 5), Fraction(2, 5)]


def test_all_accepted_adds_the_targets_next_token(oracle_lib):
    V, k = 6, 3
    p = np.full((1, k, V), 1.0 / V, np.float32)
    q = np.zeros((1, k + 1, V), np.float32)
    q[0, :, 4] = 1.0                                   # the target is sure of token 4
    out, cnt, ctx = oracle_lib.spec_verify_sample(p, q, np.full((1, k), 4), np.zeros((1, k), np.float32),
                                                  np.array([0.3], np.float32), np.array([50]))
    assert cnt[0] == k + 1 and list(out[0]) == [4, 4, 4, 4] and ctx[0] == 50
