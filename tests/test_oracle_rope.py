"""Pins for the oracle's rotary embedding and KV append.

RoPE is a rotation of each (2i, 2i+1) pair: lengths are kept, position 0 is
the identity, one pair at position 1 with theta = 1 turns (1, 0) into
(cos 1, sin 1), pairs do not mix, and the score of a rotated query and key
depends only on their distance (the property the rotary form is built for),
which also fixes the sign convention up to a common flip. The append places
token i of sequence b at global position ctx - W + i of the block table."""
import math

import numpy as np
import pytest

from memory_bound_decode_dq_gb300 import synth


def test_identity_at_zero_and_norms(oracle_lib):
    rng = np.random.default_rng(0)
    x = rng.standard_normal((20, 128))
    assert np.array_equal(oracle_lib.rope(x, np.zeros(20)), x)
    y = oracle_lib.rope(x, rng.integers(0, 200000, 20).astype(np.float64))
    pairs = lambda a: np.hypot(a[:, 0::2], a[:, 1::2])
    np.testing.assert_allclose(pairs(y), pairs(x), rtol=1e-13)


def test_first_pair_turns_by_the_position(oracle_lib):
    x = np.zeros((1, 2))
    x[0, 0] = 1.0
    y = oracle_lib.rope(x, np.array([1.0]))              # d = 2: theta_0 = base^0 = 1
    np.testing.assert_allclose(y[0], [math.cos(1.0), math.sin(1.0)], rtol=0, atol=1e-15)
    x = np.zeros((1, 8))
    x[0, 6] = 1.0                                         # pair i = 3 of d = 8: theta = base^(-3/4)
    y = oracle_lib.rope(x, np.array([5.0]), base=10000.0)
    a = 5.0 * 10000.0 ** (-0.75)
    expect = np.zeros(8)
    expect[6], expect[7] = math.cos(a), math.sin(a)
    np.testing.assert_allclose(y[0], expect, rtol=0, atol=1e-15)


def test_scores_depend_only_on_distance(oracle_lib):
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal((1, 128)), rng.standard_normal((1, 128))
    base = []
    for shift in (0, 17, 4096, 131000):
        qr = oracle_lib.rope(q, np.array([shift + 40.0]))
        kr = oracle_lib.rope(k, np.array([shift + 3.0]))
        base.append(float(qr[0] @ kr[0]))
    np.testing.assert_allclose(base, base[0], rtol=1e-9)
    # and it does depend on the distance
    qr = oracle_lib.rope(q, np.array([41.0]))
    assert abs(float(qr[0] @ oracle_lib.rope(k, np.array([3.0]))[0]) - base[0]) > 1e-3


def test_append_positions_and_heads(oracle_lib):
    B, W, hq, hkv, d = 2, 3, 4, 2, 16
    ctx = np.array([20, 3], np.int32)
    table, nblk = synth.block_table(0, "t", ctx)
    qkv = synth.normal_bf16(0, "qkv", (B * W, (hq + 2 * hkv) * d))
    q, k, v, slot = oracle_lib.rope_kv_append(qkv, B, W, hq, hkv, 10000.0, ctx, table, nblk)
    f = (qkv.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(B, W, hq + 2 * hkv, d)
    np.testing.assert_array_equal(v, f[:, :, hq + hkv:])            # V is appended as is
    for b in range(B):
        for i in range(W):
            pos = ctx[b] - W + i
            assert slot[b, i] == table[b, pos // 16] * hkv * 16 + pos % 16
            np.testing.assert_allclose(q[b, i], oracle_lib.rope(f[b, i, :hq], np.full(hq, float(pos))), rtol=1e-15)
            np.testing.assert_allclose(k[b, i], oracle_lib.rope(f[b, i, hq:hq + hkv], np.full(hkv, float(pos))),
                                       rtol=1e-15)
