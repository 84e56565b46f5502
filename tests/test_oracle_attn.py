"""Pins for the oracle's paged GQA decode/verify attention.

Checked against properties that fix softmax attention independently of how
it is evaluated: a constant V comes back unchanged, one visible key returns
its V row, a dominant logit selects its V row, moving physical blocks (with
the table) changes nothing, the verify mask agrees with plain decode calls
at the corresponding context, and a single head over contiguous keys equals
scipy's softmax applied to q K^T."""
import math

import numpy as np
import pytest
from scipy.special import softmax

from memory_bound_decode_dq_gb300 import synth


def _f(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _setup(seed, B, W, hq, hkv, ctx, shuffle=True, d=128):
    kv = synth.paged_kv(seed, "kv", ctx, hkv, d, shuffle=shuffle)
    q = synth.normal_bf16(seed, "q", (B, W, hq, d))
    return q, kv


def _run(o, q, kv, hkv, scale=None, rows=None, ctx=None, table=None):
    d = q.shape[-1]
    return o.gqa_decode_attn(q, kv.k_pool, kv.v_pool,
                             kv.block_table if table is None else table,
                             kv.context_lens if ctx is None else ctx, hkv,
                             1 / math.sqrt(d) if scale is None else scale, rows=rows)


def test_uniform_v_returns_v(oracle_lib):
    q, kv = _setup(0, 2, 3, 8, 2, (40, 77))
    v = synth.normal_bf16(0, "vrow", (2, 128))
    kv.v_pool[:] = v[None, :, None, :]                  # every V row of head g equals v[g]
    out = _run(oracle_lib, q, kv, 2)
    want = np.broadcast_to(_f(v)[None, None, [0, 0, 0, 0, 1, 1, 1, 1], :], out.shape)
    np.testing.assert_allclose(out, want, rtol=1e-13, atol=1e-13)


def test_single_key_returns_its_value(oracle_lib):
    q, kv = _setup(1, 1, 1, 4, 4, (1,))
    out = _run(oracle_lib, q, kv, 4)
    blk = kv.block_table[0, 0]
    assert np.array_equal(out[0, 0], _f(kv.v_pool[blk, :, 0, :]))


def test_dominant_logit_selects_its_row(oracle_lib):
    d = 128
    q, kv = _setup(2, 1, 1, 2, 1, (50,), shuffle=False)
    kv.k_pool[:] = 0
    q[:] = 0
    q[0, 0, :, 0] = 0x3F80                              # q = e_0 for both heads
    kv.k_pool[2, 0, 3, 0] = 0x41F0                      # key 35 (block 2, slot 3): logit 30
    out = _run(oracle_lib, q, kv, 1, scale=1.0)
    target = _f(kv.v_pool[2, 0, 3])
    others = _f(kv.v_pool[:, 0].reshape(-1, d)[:50])
    bound = 49 * math.exp(-30) * np.abs(others).max() * 2
    assert np.abs(out[0, 0, 0] - target).max() < bound
    assert np.abs(out[0, 0, 1] - target).max() < bound


def test_mha_single_head_matches_scipy_softmax(oracle_lib):
    ctx = (70,)
    q, kv = _setup(3, 1, 1, 1, 1, ctx, shuffle=False)
    keys = _f(kv.k_pool[:, 0].reshape(-1, 128)[:70])
    vals = _f(kv.v_pool[:, 0].reshape(-1, 128)[:70])
    p = softmax(_f(q[0, 0, 0]) @ keys.T * 0.0883883476)
    out = _run(oracle_lib, q, kv, 1, scale=0.0883883476)
    np.testing.assert_allclose(out[0, 0, 0], p @ vals, rtol=1e-12, atol=1e-13)


def test_gqa_equals_mha_with_repeated_kv(oracle_lib):
    """Hq=8 over Hkv=2 equals Hq=8 over Hkv=8 where KV head h holds a copy of
    group h // 4's data (contiguous grouping)."""
    ctx = (33, 64)
    q, kv = _setup(4, 2, 2, 8, 2, ctx)
    a = _run(oracle_lib, q, kv, 2)
    rep = synth.PagedKV(k_pool=np.repeat(kv.k_pool, 4, axis=1), v_pool=np.repeat(kv.v_pool, 4, axis=1),
                        block_table=kv.block_table, context_lens=kv.context_lens, num_blocks=kv.num_blocks)
    b = _run(oracle_lib, q, rep, 8)
    assert np.array_equal(a, b)


def test_block_permutation_invariance(oracle_lib):
    ctx = (100, 37, 16)
    q, kv = _setup(5, 3, 2, 4, 2, ctx)
    a = _run(oracle_lib, q, kv, 2)
    perm = np.random.default_rng(9).permutation(kv.num_blocks)   # new slot of old block i
    kp = np.empty_like(kv.k_pool)
    vp = np.empty_like(kv.v_pool)
    kp[perm] = kv.k_pool
    vp[perm] = kv.v_pool
    table = perm[kv.block_table].astype(np.int32)
    moved = synth.PagedKV(kp, vp, table, kv.context_lens, kv.num_blocks)
    assert np.array_equal(_run(oracle_lib, q, moved, 2), a)


def test_verify_rows_equal_plain_decode_at_shorter_context(oracle_lib):
    W, ctx = 5, (61, 200)
    q, kv = _setup(6, 2, W, 4, 1, ctx)
    out = _run(oracle_lib, q, kv, 1)
    for i in range(W):
        short = np.asarray(ctx, np.int32) - W + i + 1
        one = _run(oracle_lib, q[:, i:i + 1].copy(), kv, 1, ctx=short)
        assert np.array_equal(out[:, i], one[:, 0])
    # the last verify row is the plain decode call at the full context
    last = _run(oracle_lib, q[:, W - 1:].copy(), kv, 1)
    assert np.array_equal(out[:, W - 1], last[:, 0])


def test_row_subset_equals_full(oracle_lib):
    q, kv = _setup(7, 2, 3, 4, 2, (20, 48))
    full = _run(oracle_lib, q, kv, 2).reshape(-1, 128)
    rows = np.array([0, 23, 5, 5, 17])
    assert np.array_equal(_run(oracle_lib, q, kv, 2, rows=rows), full[rows])


def test_rejects_context_shorter_than_width(oracle_lib):
    q, kv = _setup(8, 1, 4, 2, 1, (8,))
    with pytest.raises(ValueError):
        _run(oracle_lib, q, kv, 1, ctx=np.array([3], np.int32))
