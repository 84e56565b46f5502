"""Pins for the oracle's attention over an FP8-E4M3 KV cache.

The FP8 cache holds one E4M3 code per element and one scale per pool, so
attention over it must equal attention over a bf16 cache that holds the
decoded values: every E4M3 value times a power of two is a bf16 number, and
the bf16 oracle is pinned on its own (closed forms, scipy's softmax). The
codes are decoded here by torch's float8_e4m3fn type, not by the oracle.
Closed forms and invariants pin the two scales: a constant V code returns
decode(code) * v_scale, k_scale = 0 gives uniform weights (the mean of the
visible V rows), the output is linear in v_scale, and k_scale multiplies the
logits exactly as the softmax scale does."""
import math

import numpy as np
import pytest
import torch

from memory_bound_decode_dq_gb300 import synth


def _torch_decode(codes) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _exact_bf16_bits(values: np.ndarray) -> np.ndarray:
    f = values.astype(np.float32)
    assert np.array_equal(f.astype(np.float64), values)
    u = f.view(np.uint32)
    assert not np.any(u & 0xFFFF), "value not representable in bf16"
    return (u >> 16).astype(np.uint16)


def _setup(seed, B, W, hq, hkv, ctx, shuffle=True, exp_lo=0, exp_hi=15):
    kv = synth.paged_kv_fp8(seed, "kv8", ctx, hkv, shuffle=shuffle, exp_lo=exp_lo, exp_hi=exp_hi)
    q = synth.normal_bf16(seed, "q", (B, W, hq, 128))
    return q, kv


def _run(o, q, kv, hkv, ks, vs, scale=None, ctx=None):
    return o.gqa_decode_attn_fp8kv(q, kv.k_codes, kv.v_codes, kv.block_table,
                                   kv.context_lens if ctx is None else ctx, hkv,
                                   1 / math.sqrt(128) if scale is None else scale, ks, vs)


def test_decoded_codes_cover_every_finite_value():
    codes = synth.e4m3_codes(0, "all", (20000,))
    assert not np.any((codes & 0x7F) == 0x7F)
    assert len(np.unique(codes)) == 254          # 256 codes minus the two NaNs


@pytest.mark.parametrize("ks,vs", [(1.0, 1.0), (2.0 ** -4, 2.0 ** -3), (4.0, 0.5)])
def test_equals_bf16_attention_on_decoded_values(oracle_lib, ks, vs):
    ctx = (1, 45, 130)
    q, kv = _setup(11, 3, 2, 8, 2, ctx)
    q8 = q.copy()
    kbits = _exact_bf16_bits(_torch_decode(kv.k_codes) * ks)
    vbits = _exact_bf16_bits(_torch_decode(kv.v_codes) * vs)
    want = oracle_lib.gqa_decode_attn(q, kbits, vbits, kv.block_table, np.maximum(kv.context_lens, 2),
                                      2, 0.07)
    got = oracle_lib.gqa_decode_attn_fp8kv(q8, kv.k_codes, kv.v_codes, kv.block_table,
                                           np.maximum(kv.context_lens, 2), 2, 0.07, ks, vs)
    assert np.array_equal(got, want)


def test_constant_v_code_returns_its_value(oracle_lib):
    q, kv = _setup(12, 2, 3, 4, 2, (40, 77))
    kv.v_codes[:] = 0xB5                          # -(1 + 5/8) * 2^(6-7) = -0.8125
    out = _run(oracle_lib, q, kv, 2, 0.01, 3.0)
    np.testing.assert_allclose(out, -0.8125 * 3.0, rtol=1e-13, atol=0)


def test_zero_k_scale_averages_visible_rows(oracle_lib):
    W, ctx = 3, (40, 77)
    q, kv = _setup(13, 2, W, 4, 2, ctx)
    out = _run(oracle_lib, q, kv, 2, 0.0, 0.25)
    vals = _torch_decode(kv.v_codes)
    for b, c in enumerate(ctx):
        rows = np.concatenate([vals[kv.block_table[b, j // 16], :, j % 16][None] for j in range(c)])
        for i in range(W):
            mean = rows[: c - W + i + 1].mean(axis=0) * 0.25           # [hkv, 128]
            for h in range(4):
                np.testing.assert_allclose(out[b, i, h], mean[h // 2], rtol=1e-12, atol=1e-14)


def test_linear_in_v_scale(oracle_lib):
    q, kv = _setup(14, 2, 2, 8, 8, (33, 90), exp_lo=4, exp_hi=12)
    a = _run(oracle_lib, q, kv, 8, 0.02, 1.0)
    b = _run(oracle_lib, q, kv, 8, 0.02, 0.3)
    # each output is a sum of signed terms: compare against the size of the terms
    np.testing.assert_allclose(b, 0.3 * a, rtol=1e-13, atol=1e-13 * np.abs(b).max())


def test_k_scale_acts_like_softmax_scale(oracle_lib):
    q, kv = _setup(15, 1, 4, 4, 1, (60,), exp_lo=4, exp_hi=12)
    a = _run(oracle_lib, q, kv, 1, 0.05, 1.0, scale=0.125)
    b = _run(oracle_lib, q, kv, 1, 1.0, 1.0, scale=0.125 * 0.05)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_single_key_returns_its_scaled_value(oracle_lib):
    q, kv = _setup(16, 1, 1, 2, 2, (1,))
    out = _run(oracle_lib, q, kv, 2, 0.5, 0.125)
    blk = kv.block_table[0, 0]
    assert np.array_equal(out[0, 0], _torch_decode(kv.v_codes[blk, :, 0, :]) * 0.125)
