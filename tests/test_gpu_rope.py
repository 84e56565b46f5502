"""GPU parity of rope_kv_append against the oracle: rotated q and k within the
floating-point tolerance, v copied bit for bit (bf16 cache) or encoded as the
oracle's E4M3 codes (FP8 cache), every other cache slot untouched, and the
step followed by the attention equal to the oracle's attention over the
appended cache."""
import math

import numpy as np
import pytest
import torch

import oracle
from memory_bound_decode_dq_gb300 import synth
from gpu_util import assert_close, bf, bits, f64, i32, require_cuda, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_cuda()


@pytest.fixture(scope="module")
def dqd():
    from memory_bound_decode_dq_gb300 import dqd as m
    return m


def _f(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _case(seed, B, W, hq, hkv, d, ctx):
    ctx = np.asarray(ctx, np.int32)
    table, nblk = synth.block_table(seed, "tbl", ctx, spare_blocks=2)
    qkv = synth.normal_bf16(seed, "qkv", (B * W, (hq + 2 * hkv) * d))
    return qkv, table, nblk, ctx


CASES = [
    # B, W, hq, hkv, d, contexts, base
    (1, 1, 32, 8, 128, (8192,), 500000.0),
    (2, 6, 32, 8, 128, (6, 700), 10000.0),
    (3, 16, 64, 2, 128, (16, 131072, 40), 500000.0),  # positions up to 2^17
    (4, 3, 12, 4, 64, (5, 16, 31, 47), 10000.0),
]


@pytest.mark.parametrize("B,W,hq,hkv,d,ctx,base", CASES)
def test_bf16_cache_against_oracle(dev, dqd, B, W, hq, hkv, d, ctx, base):
    qkv, table, nblk, ctx = _case(B * 10 + W, B, W, hq, hkv, d, ctx)
    kp0 = synth.normal_bf16(1, "kp", (nblk, hkv, 16, d))
    vp0 = synth.normal_bf16(2, "vp", (nblk, hkv, 16, d))
    kp, vp = bf(kp0, dev), bf(vp0, dev)
    q = dqd.rope_kv_append(bf(qkv, dev), B, W, hq, hkv, kp, vp, i32(table, dev), i32(ctx, dev), rope_base=base)
    rq, rk, rv, slot = oracle.rope_kv_append(qkv, B, W, hq, hkv, base, ctx, table, nblk)
    assert_close(f64(q), rq, what="rotated q")
    kb, vb = bits(kp), bits(vp)
    rows_k = kb.reshape(-1, d)
    rows_v = vb.reshape(-1, d)
    touched = np.zeros(rows_k.shape[0], bool)
    for r in range(B):
        for i in range(W):
            s = slot[r, i]
            if s < 0:
                continue
            for g in range(hkv):
                touched[s + 16 * g] = True
                assert_close(_f(rows_k[s + 16 * g]), rk[r, i, g], what=f"k r={r} i={i} g={g}")
                assert np.array_equal(rows_v[s + 16 * g], qkv[r * W + i, (hq + hkv + g) * d:(hq + hkv + g + 1) * d])
    # every other slot keeps its old contents
    assert np.array_equal(rows_k[~touched], kp0.reshape(-1, d)[~touched])
    assert np.array_equal(rows_v[~touched], vp0.reshape(-1, d)[~touched])


def test_fp8_cache_codes(dev, dqd):
    B, W, hq, hkv, d = 2, 4, 16, 4, 128
    qkv, table, nblk, ctx = _case(7, B, W, hq, hkv, d, (9, 300))
    ks, vs = 1 / 64, 1 / 128
    kp = torch.zeros((nblk, hkv, 16, d), dtype=torch.uint8, device=dev)
    vp = torch.zeros_like(kp)
    dqd.rope_kv_append(bf(qkv, dev), B, W, hq, hkv, kp, vp, i32(table, dev), i32(ctx, dev), k_scale=ks,
                       v_scale=vs)
    _, rk, rv, slot = oracle.rope_kv_append(qkv, B, W, hq, hkv, 10000.0, ctx, table, nblk)
    kc, vc = kp.cpu().numpy().reshape(-1, d), vp.cpu().numpy().reshape(-1, d)
    for r in range(B):
        for i in range(W):
            for g in range(hkv):
                row = slot[r, i] + 16 * g
                # v: the oracle's own E4M3 encoding of fp32(v / scale), bit for bit
                want = oracle.e4m3_encode((rv[r, i, g] / vs).astype(np.float32))
                assert np.array_equal(vc[row], want)
                # k: rotated in binary32, so within one E4M3 step of the oracle's value
                dec = oracle.e4m3_decode(kc[row]) * ks
                step = np.maximum(np.abs(rk[r, i, g]) * 2.0 ** -3, 2.0 ** -9 * ks)
                assert np.all(np.abs(dec - np.clip(rk[r, i, g], -448 * ks, 448 * ks)) <= step)


def test_append_then_attend(dev, dqd):
    """rope_kv_append followed by gqa_decode_attn equals the oracle's
    attention with the oracle's rotated q over the oracle-appended cache."""
    B, W, hq, hkv, d = 2, 5, 32, 8, 128
    qkv, table, nblk, ctx = _case(11, B, W, hq, hkv, d, (77, 400))
    kp0 = synth.normal_bf16(3, "kp", (nblk, hkv, 16, d))
    vp0 = synth.normal_bf16(4, "vp", (nblk, hkv, 16, d))
    kp, vp = bf(kp0, dev), bf(vp0, dev)
    t, c = i32(table, dev), i32(ctx, dev)
    q = dqd.rope_kv_append(bf(qkv, dev), B, W, hq, hkv, kp, vp, t, c)
    out = dqd.gqa_decode_attn(q, kp, vp, t, c, int(ctx.max()))
    rq, rk, rv, slot = oracle.rope_kv_append(qkv, B, W, hq, hkv, 10000.0, ctx, table, nblk)
    kref, vref = kp0.reshape(-1, d).copy(), vp0.reshape(-1, d).copy()
    for r in range(B):
        for i in range(W):
            for g in range(hkv):
                kref[slot[r, i] + 16 * g] = oracle.bf16_round(rk[r, i, g])
                vref[slot[r, i] + 16 * g] = oracle.bf16_round(rv[r, i, g])
    ref = oracle.gqa_decode_attn(oracle.bf16_round(rq), kref.reshape(kp0.shape), vref.reshape(vp0.shape),
                                 table, ctx, hkv, 1 / math.sqrt(d))
    assert_close(f64(out), ref, what="append then attend")


def test_rejects_bad_arguments(dev, dqd):
    qkv = torch.zeros((2, 48 * 128), dtype=torch.bfloat16, device=dev)
    kp = torch.zeros((4, 8, 16, 128), dtype=torch.bfloat16, device=dev)
    t, c = i32(np.zeros((2, 4), np.int32), dev), i32(np.array([5, 5], np.int32), dev)
    with pytest.raises(ValueError):
        dqd.rope_kv_append(qkv, 2, 2, 32, 8, kp, kp, t, c)           # 2 rows for b*w = 4
    with pytest.raises(dqd.DqdError):
        dqd.rope_kv_append(qkv, 2, 1, 32, 8, kp, kp, t, c, rope_base=0.5)


def test_out_of_range_table_entry_is_clamped_and_reported(dev, dqd):
    """A table entry past the pool appends into the pool's last block (no
    write outside the pool) and raises the bad-input flag once."""
    assert dqd.device_errors() == 0
    B, W, hq, hkv, d = 1, 2, 8, 2, 128
    qkv, table, nblk, ctx = _case(12, B, W, hq, hkv, d, (40,))
    kp = bf(np.zeros((nblk, hkv, 16, d), np.uint16), dev)
    vp = bf(np.zeros((nblk, hkv, 16, d), np.uint16), dev)
    bad = table.copy()
    bad[0, (int(ctx[0]) - 1) // 16] = nblk + 7
    dqd.rope_kv_append(bf(qkv, dev), B, W, hq, hkv, kp, vp, i32(bad, dev), i32(ctx, dev))
    assert dqd.device_errors() == dqd.DQD_DEVICE_ERR_BAD_INPUT
    assert np.any(bits(vp)[nblk - 1] != 0)     # the clamped append landed in the last block
    assert dqd.device_errors() == 0


def test_no_device_error_flags(dev, dqd):
    assert dqd.device_errors() == 0
