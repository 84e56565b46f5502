"""GPU parity of gqa_decode_attn_fp8kv (paged GQA attention over an FP8-E4M3
KV cache) against the float64 oracle, plus properties that hold whatever the
evaluation order: a constant V code comes back as its value times v_scale,
one visible key returns its row, moving blocks changes no bit, and stale
codes past the context are never seen."""
import math

import numpy as np
import pytest
import torch

import oracle
from memory_bound_decode_dq_gb300 import synth
from gpu_util import assert_close, bf, bits, f64, i32, require_cuda, u8

pytestmark = pytest.mark.gpu

KS, VS = 1 / 64, 1 / 128   # cached K = code / 64, V = code / 128


@pytest.fixture(scope="module")
def dev():
    return require_cuda()


@pytest.fixture(scope="module")
def dqd():
    from memory_bound_decode_dq_gb300 import dqd as m
    return m


@pytest.fixture
def chunk(monkeypatch):
    def set_chunk(v):
        monkeypatch.setenv("DQD_ATTN_CHUNK_BLOCKS", str(v))
    yield set_chunk
    monkeypatch.delenv("DQD_ATTN_CHUNK_BLOCKS", raising=False)


def run(dqd, dev, q, kv, ctx=None, scale=None, ks=KS, vs=VS, max_context=None, table=None,
        as_float8=False):
    ctx = kv.context_lens if ctx is None else np.asarray(ctx, np.int32)
    table = kv.block_table if table is None else table
    kp, vp = u8(kv.k_codes, dev), u8(kv.v_codes, dev)
    if as_float8:
        kp, vp = kp.view(torch.float8_e4m3fn), vp.view(torch.float8_e4m3fn)
    return dqd.gqa_decode_attn_fp8kv(bf(q, dev), kp, vp, i32(table, dev), i32(ctx, dev),
                                     int(max_context or max(int(ctx.max()), 1)), ks, vs,
                                     softmax_scale=scale)


def ref(q, kv, hkv, ctx=None, scale=None, ks=KS, vs=VS, rows=None):
    return oracle.gqa_decode_attn_fp8kv(q, kv.k_codes, kv.v_codes, kv.block_table,
                                        kv.context_lens if ctx is None else ctx, hkv,
                                        1 / math.sqrt(128) if scale is None else scale, ks, vs,
                                        rows=rows)


CASES = [
    # B, W, Hq, Hkv, contexts
    (1, 1, 8, 2, (256,)),
    (1, 1, 64, 8, (1000,)),
    (3, 1, 8, 2, (1, 17, 300)),
    (2, 1, 4, 4, (33, 64)),          # MHA
    (2, 1, 64, 8, (129, 2048)),      # 8 heads per group
    (2, 6, 32, 8, (6, 700)),         # verify, 24 rows per kv head
    (2, 16, 32, 8, (16, 513)),       # verify, 64 rows per kv head
    (1, 16, 64, 8, (900,)),          # 128 rows per kv head: two query groups
    (4, 3, 12, 4, (5, 16, 31, 47)),
]


@pytest.mark.parametrize("B,W,hq,hkv,ctx", CASES)
def test_against_oracle(dev, dqd, B, W, hq, hkv, ctx):
    kv = synth.paged_kv_fp8(B * 100 + W, "kv8", ctx, hkv, spare_blocks=3)
    q = synth.normal_bf16(B + W, "q", (B, W, hq, 128))
    out = run(dqd, dev, q, kv)
    assert_close(f64(out), ref(q, kv, hkv), what=f"fp8kv B={B} W={W} {hq}/{hkv} ctx={ctx}")


@pytest.mark.parametrize("cb", [1, 2, 3, 4, 7, 16, 1000])
@pytest.mark.parametrize("W", [1, 16])
def test_every_chunk_size(dev, dqd, chunk, cb, W):
    chunk(cb)
    kv = synth.paged_kv_fp8(cb, "kv8", (W + 40, 333), 2)
    q = synth.normal_bf16(cb, "q", (2, W, 8, 128))
    assert_close(f64(run(dqd, dev, q, kv)), ref(q, kv, 2), what=f"chunk_blocks={cb} W={W}")


@pytest.mark.parametrize("ks,vs", [(1.0, 1.0), (0.003, 0.5), (0.0, 0.01)])
def test_scales(dev, dqd, ks, vs):
    """k_scale 0 gives uniform weights over the visible keys."""
    kv = synth.paged_kv_fp8(21, "kv8", (90, 260), 2, exp_lo=2, exp_hi=12)
    q = synth.normal_bf16(21, "q", (2, 3, 8, 128))
    assert_close(f64(run(dqd, dev, q, kv, ks=ks, vs=vs)), ref(q, kv, 2, ks=ks, vs=vs),
                 what=f"k_scale={ks} v_scale={vs}")


def test_constant_v_code_returns_its_value(dev, dqd):
    kv = synth.paged_kv_fp8(22, "kv8", (77, 500), 2)
    kv.v_codes[:] = 0xB5                          # -0.8125
    q = synth.normal_bf16(22, "q", (2, 4, 8, 128))
    out = f64(run(dqd, dev, q, kv, vs=3.0))
    # a normalised sum of identical rows: exact up to the final bf16 rounding
    assert np.all(np.abs(out + 0.8125 * 3.0) <= 0.8125 * 3.0 * 2 ** -8)


def test_single_key_returns_its_scaled_value(dev, dqd):
    kv = synth.paged_kv_fp8(23, "kv8", (1, 1), 4)
    q = synth.normal_bf16(23, "q", (2, 1, 4, 128))
    out = bits(run(dqd, dev, q, kv, vs=0.125))
    dec = torch.from_numpy(kv.v_codes).view(torch.float8_e4m3fn).to(torch.float32) * 0.125
    want = dec.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    # p * V accumulates onto +0, which turns a -0 value (code 0x80) into +0
    # (IEEE: +0 + -0 = +0), so zeros are compared by value
    want = np.where(want == 0x8000, 0, want).astype(np.uint16)
    for b in range(2):
        blk = kv.block_table[b, 0]
        assert np.array_equal(out[b, 0], want[blk, :, 0, :])


def test_block_permutation_is_bit_identical(dev, dqd):
    ctx = (100, 37, 16, 200)
    kv = synth.paged_kv_fp8(24, "kv8", ctx, 2)
    q = synth.normal_bf16(24, "q", (4, 2, 8, 128))
    a = bits(run(dqd, dev, q, kv))
    perm = np.random.default_rng(9).permutation(kv.num_blocks)
    kp = np.empty_like(kv.k_codes)
    vp = np.empty_like(kv.v_codes)
    kp[perm] = kv.k_codes
    vp[perm] = kv.v_codes
    moved = synth.PagedKVFp8(kp, vp, perm[kv.block_table].astype(np.int32), kv.context_lens,
                             kv.num_blocks)
    assert np.array_equal(bits(run(dqd, dev, q, moved)), a)


def test_stale_codes_do_not_leak(dev, dqd):
    """Slots past the context inside the last block hold the largest code
    (+448) in K and V; the output must not see them."""
    ctx = (21, 5)
    kv = synth.paged_kv_fp8(25, "kv8", ctx, 2)
    clean = synth.PagedKVFp8(kv.k_codes.copy(), kv.v_codes.copy(), kv.block_table, kv.context_lens,
                             kv.num_blocks)
    for b, c in enumerate(ctx):
        last = kv.block_table[b, (c - 1) // 16]
        kv.k_codes[last, :, c % 16:, :] = 0x7E
        kv.v_codes[last, :, c % 16:, :] = 0x7E
    q = synth.normal_bf16(25, "q", (2, 1, 8, 128))
    assert np.array_equal(bits(run(dqd, dev, q, kv)), bits(run(dqd, dev, q, clean)))


def test_float8_tensors_are_accepted(dev, dqd):
    kv = synth.paged_kv_fp8(26, "kv8", (70,), 2)
    q = synth.normal_bf16(26, "q", (1, 1, 8, 128))
    assert np.array_equal(bits(run(dqd, dev, q, kv)), bits(run(dqd, dev, q, kv, as_float8=True)))


def test_rejects_bad_arguments(dev, dqd):
    kv = synth.paged_kv_fp8(27, "kv8", (16,), 2)
    q = synth.normal_bf16(27, "q", (1, 1, 4, 128))
    with pytest.raises(dqd.DqdError):
        run(dqd, dev, q, kv, ks=float("inf"))
    with pytest.raises(dqd.DqdError):
        run(dqd, dev, q, kv, vs=float("nan"))
    with pytest.raises(TypeError):
        dqd.gqa_decode_attn_fp8kv(bf(q, dev), bf(np.zeros((1, 2, 16, 128), np.uint16), dev),
                                  bf(np.zeros((1, 2, 16, 128), np.uint16), dev),
                                  i32(kv.block_table, dev), i32(kv.context_lens, dev), 16, 1.0, 1.0)


def test_no_device_error_flags_after_the_suite(dev, dqd):
    """No bounded wait on an asynchronous copy gave up during this module."""
    assert dqd.device_errors() == 0
