"""GPU parity of gqa_decode_attn against the float64 oracle, plus the
properties that fix attention independently of its evaluation order."""
import math

import numpy as np
import pytest
import torch

import oracle
from memory_bound_decode_dq_gb300 import synth
from gpu_util import assert_close, bf, bits, f64, i32, require_cuda

pytestmark = pytest.mark.gpu


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
        if v is None:
            monkeypatch.delenv("DQD_ATTN_CHUNK_BLOCKS", raising=False)
        else:
            monkeypatch.setenv("DQD_ATTN_CHUNK_BLOCKS", str(v))
    yield set_chunk
    monkeypatch.delenv("DQD_ATTN_CHUNK_BLOCKS", raising=False)


def run(dqd, dev, q, kv, hkv, ctx=None, scale=None, max_context=None, table=None):
    ctx = kv.context_lens if ctx is None else np.asarray(ctx, np.int32)
    table = kv.block_table if table is None else table
    out = dqd.gqa_decode_attn(bf(q, dev), bf(kv.k_pool, dev), bf(kv.v_pool, dev), i32(table, dev),
                              i32(ctx, dev), int(max_context or max(int(ctx.max()), 1)),
                              softmax_scale=scale)
    return out


def ref(q, kv, hkv, ctx=None, scale=None, table=None):
    d = q.shape[-1]
    return oracle.gqa_decode_attn(q, kv.k_pool, kv.v_pool, kv.block_table if table is None else table,
                                  kv.context_lens if ctx is None else ctx, hkv,
                                  1 / math.sqrt(d) if scale is None else scale)


CASES = [
    # B, W, Hq, Hkv, contexts
    (1, 1, 8, 2, (256,)),
    (1, 1, 32, 8, (1000,)),
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
    kv = synth.paged_kv(B * 100 + W, "kv", ctx, hkv, spare_blocks=3)
    q = synth.normal_bf16(B + W, "q", (B, W, hq, 128))
    out = run(dqd, dev, q, kv, hkv)
    assert_close(f64(out), ref(q, kv, hkv), what=f"attn B={B} W={W} {hq}/{hkv} ctx={ctx}")


@pytest.mark.parametrize("cb", [1, 2, 3, 4, 7, 16, 1000])
@pytest.mark.parametrize("W", [1, 16])
def test_every_chunk_size(dev, dqd, chunk, cb, W):
    chunk(cb)
    kv = synth.paged_kv(cb, "kv", (W + 40, 333), 2)
    q = synth.normal_bf16(cb, "q", (2, W, 8, 128))
    assert_close(f64(run(dqd, dev, q, kv, 2)), ref(q, kv, 2), what=f"chunk_blocks={cb} W={W}")


def test_uniform_v_returns_v(dev, dqd):
    kv = synth.paged_kv(1, "kv", (77, 500), 2)
    v = synth.normal_bf16(1, "v", (2, 128))
    kv.v_pool[:] = v[None, :, None, :]
    q = synth.normal_bf16(1, "q", (2, 4, 8, 128))
    out = bits(run(dqd, dev, q, kv, 2))
    want = np.broadcast_to(v[None, None, [0, 0, 0, 0, 1, 1, 1, 1], :], out.shape)
    # normalised sum of identical rows: exact up to the final rounding
    diff = np.abs(((out.astype(np.uint32) << 16).view(np.float32)) - ((want.astype(np.uint32) << 16).view(np.float32)))
    assert np.all(diff <= np.abs((want.astype(np.uint32) << 16).view(np.float32)) * 2 ** -7)
    assert np.mean(out == want) > 0.99


def test_single_key_returns_its_value(dev, dqd):
    kv = synth.paged_kv(2, "kv", (1, 1), 4)
    q = synth.normal_bf16(2, "q", (2, 1, 4, 128))
    out = bits(run(dqd, dev, q, kv, 4))
    for b in range(2):
        blk = kv.block_table[b, 0]
        assert np.array_equal(out[b, 0], kv.v_pool[blk, :, 0, :])


def test_dominant_logit(dev, dqd):
    kv = synth.paged_kv(3, "kv", (50,), 1, shuffle=False)
    kv.k_pool[:] = 0
    q = np.zeros((1, 1, 2, 128), np.uint16)
    q[0, 0, :, 0] = 0x3F80
    kv.k_pool[2, 0, 3, 0] = 0x41F0  # logit 30 at key 35
    out = f64(run(dqd, dev, q, kv, 1, scale=1.0))
    target = (kv.v_pool[2, 0, 3].astype(np.uint32) << 16).view(np.float32)
    assert np.abs(out[0, 0, 0] - target).max() <= np.abs(target).max() * 2 ** -7
    assert np.abs(out[0, 0, 1] - target).max() <= np.abs(target).max() * 2 ** -7


def test_block_permutation_is_bit_identical(dev, dqd):
    ctx = (100, 37, 16, 200)
    kv = synth.paged_kv(5, "kv", ctx, 2)
    q = synth.normal_bf16(5, "q", (4, 2, 8, 128))
    a = bits(run(dqd, dev, q, kv, 2))
    perm = np.random.default_rng(9).permutation(kv.num_blocks)
    kp = np.empty_like(kv.k_pool)
    vp = np.empty_like(kv.v_pool)
    kp[perm] = kv.k_pool
    vp[perm] = kv.v_pool
    moved = synth.PagedKV(kp, vp, perm[kv.block_table].astype(np.int32), kv.context_lens, kv.num_blocks)
    assert np.array_equal(bits(run(dqd, dev, q, moved, 2)), a)


def test_verify_rows_match_plain_decode(dev, dqd):
    W, ctx = 6, (61, 250)
    kv = synth.paged_kv(6, "kv", ctx, 2)
    q = synth.normal_bf16(6, "q", (2, W, 8, 128))
    out = f64(run(dqd, dev, q, kv, 2))
    for i in range(W):
        short = np.asarray(ctx, np.int32) - W + i + 1
        one = f64(run(dqd, dev, q[:, i:i + 1].copy(), kv, 2, ctx=short, max_context=max(ctx)))
        assert_close(out[:, i], one[:, 0], what=f"verify row {i}")


def test_stale_pool_contents_do_not_leak(dev, dqd):
    """Slots past the context inside the last block hold NaN; the output must
    not see them."""
    ctx = (21, 5)
    kv = synth.paged_kv(7, "kv", ctx, 2)
    for b, c in enumerate(ctx):
        last = kv.block_table[b, (c - 1) // 16]
        kv.k_pool[last, :, c % 16:, :] = 0x7FC0
        kv.v_pool[last, :, c % 16:, :] = 0x7FC0
    q = synth.normal_bf16(7, "q", (2, 1, 8, 128))
    out = f64(run(dqd, dev, q, kv, 2))
    assert np.all(np.isfinite(out))
    assert_close(out, ref(q, kv, 2), what="NaN padding")


def test_context_shorter_than_width_gives_zero_rows(dev, dqd):
    assert dqd.device_errors() == 0
    kv = synth.paged_kv(8, "kv", (10,), 1)
    q = synth.normal_bf16(8, "q", (1, 4, 2, 128))
    out = f64(run(dqd, dev, q, kv, 1, ctx=np.array([2], np.int32), max_context=10))
    # rows 0 and 1 sit at positions -2 and -1: they see no key
    assert np.all(out[0, :2] == 0)
    ref_rows = oracle.gqa_decode_attn(q[:, 2:], kv.k_pool, kv.v_pool, kv.block_table, np.array([2], np.int32),
                                      1, 1 / math.sqrt(128))
    assert_close(out[:, 2:], ref_rows, what="rows with keys")
    # a context below the width breaks the caller's precondition: reported once
    assert dqd.device_errors() == dqd.DQD_DEVICE_ERR_BAD_INPUT
    assert dqd.device_errors() == 0


def test_out_of_range_table_entry_is_clamped_and_reported(dev, dqd):
    """A corrupt block-table entry reads a block inside the pool (no fault),
    raises the bad-input flag, and leaves the context usable."""
    assert dqd.device_errors() == 0
    ctx = (40, 70)
    kv = synth.paged_kv(11, "kv", ctx, 2)
    q = synth.normal_bf16(11, "q", (2, 1, 8, 128))
    bad = kv.block_table.copy()
    bad[1, 2] = kv.num_blocks + 5          # past the pool: clamped to the last block
    out = f64(run(dqd, dev, q, kv, 2, table=bad))
    assert np.all(np.isfinite(out))
    assert_close(out[0], ref(q, kv, 2)[0], what="the sequence with a valid table")
    assert dqd.device_errors() == dqd.DQD_DEVICE_ERR_BAD_INPUT
    bad[1, 2] = -3                         # negative: clamped to block 0
    run(dqd, dev, q, kv, 2, table=bad)
    assert dqd.device_errors() == dqd.DQD_DEVICE_ERR_BAD_INPUT
    # the next, valid call is correct and raises nothing
    assert_close(f64(run(dqd, dev, q, kv, 2)), ref(q, kv, 2), what="after the clamped calls")
    assert dqd.device_errors() == 0


def test_context_above_max_context_is_taken_as_max_context(dev, dqd):
    """context_lens[b] > max_context breaks the caller's precondition: the
    kernel attends as if the context were max_context (bit-identical to that
    call) and raises the bad-input flag."""
    assert dqd.device_errors() == 0
    kv = synth.paged_kv(12, "kv", (300, 300), 2)
    q = synth.normal_bf16(12, "q", (2, 3, 8, 128))
    over = bits(run(dqd, dev, q, kv, 2, ctx=np.array([300, 260], np.int32), max_context=260))
    assert dqd.device_errors() == dqd.DQD_DEVICE_ERR_BAD_INPUT
    same = bits(run(dqd, dev, q, kv, 2, ctx=np.array([260, 260], np.int32), max_context=260))
    assert np.array_equal(over, same)
    assert dqd.device_errors() == 0


def test_rejects_bad_arguments(dev, dqd):
    kv = synth.paged_kv(9, "kv", (16,), 2)
    q = synth.normal_bf16(9, "q", (1, 17, 4, 128))
    with pytest.raises(dqd.DqdError):
        run(dqd, dev, q, kv, 2)          # width 17 > 16
    q = synth.normal_bf16(9, "q", (1, 1, 3, 128))
    with pytest.raises(dqd.DqdError):
        run(dqd, dev, q, kv, 2)          # 3 heads over 2 kv heads


def test_no_device_error_flags_after_the_suite(dev, dqd):
    """No bounded wait on an asynchronous copy gave up during this module."""
    assert dqd.device_errors() == 0


TC_CASES = [
    # B, W, Hq, Hkv, contexts: 17..128 query rows per kv head over a bf16 cache
    (2, 6, 32, 8, (6, 700)),          # 24 rows, one context shorter than a tile
    (2, 16, 32, 8, (16, 513)),        # 64 rows
    (1, 16, 64, 8, (900,)),           # 128 rows
    (3, 5, 16, 4, (5, 130, 2049)),    # 20 rows, ragged tiles
    (2, 9, 32, 4, (300, 4100)),       # 72 rows
]


@pytest.mark.parametrize("B,W,hq,hkv,ctx", TC_CASES)
@pytest.mark.parametrize("cb", [None, 1, 3, 8, 13])
def test_tensor_core_form(dev, dqd, monkeypatch, B, W, hq, hkv, ctx, cb):
    """The tcgen05 form (S and O in tensor memory, V as an MN-major operand)
    against the oracle, and against the mma.sync form within tolerance, for
    every chunking: chunks of whole tiles, of partial tiles, and of 1 block;
    bit-identical on a rerun and with one CTA per work unit instead of the
    persistent CTAs."""
    if cb is not None:
        monkeypatch.setenv("DQD_ATTN_CHUNK_BLOCKS", str(cb))
    kv = synth.paged_kv(B * 7 + W, "kv", ctx, hkv, spare_blocks=3)
    q = synth.normal_bf16(B + W + hq, "q", (B, W, hq, 128))
    a = run(dqd, dev, q, kv, hkv)
    assert np.array_equal(bits(a), bits(run(dqd, dev, q, kv, hkv)))
    for persist in ("0", "1"):  # one CTA per unit; persistent CTAs taking units from the queue
        monkeypatch.setenv("DQD_ATTN_PERSIST", persist)
        assert np.array_equal(bits(a), bits(run(dqd, dev, q, kv, hkv))), f"DQD_ATTN_PERSIST={persist}"
    monkeypatch.delenv("DQD_ATTN_PERSIST")
    r = ref(q, kv, hkv)
    assert_close(f64(a), r, what=f"tc attn B={B} W={W} {hq}/{hkv} ctx={ctx} cb={cb}")
    monkeypatch.setenv("DQD_ATTN_TC", "0")
    assert_close(f64(run(dqd, dev, q, kv, hkv)), r, what="mma.sync form")
    assert dqd.device_errors() == 0


@pytest.mark.parametrize("B,W,hq,hkv", [(20, 16, 32, 8), (24, 6, 32, 8), (21, 9, 32, 4)])
def test_tensor_core_balanced_tail(dev, dqd, monkeypatch, B, W, hq, hkv):
    """More work items than SMs: the items of the last partial wave are split
    into pieces of whole tiles (some empty, for short contexts) and merged by
    the tail merge. Within tolerance of the same items run whole (each piece
    rounds P to bf16 against its own reference maximum) and of the oracle
    (queries halved: with full ones, random contexts put rare elements of
    either attention form just past the 1% bound, an effect of the bf16 P that
    both forms share), bit-identical on a rerun."""
    rng = np.random.default_rng(B * 100 + W)
    # contexts of 256 .. 1499 tokens: with fewer keys per row the bf16 rounding
    # of P (either form) moves the output by a larger share of its rms (151
    # tokens: twice the rms error, the worst element at 1.0-1.15 of the bound);
    # items under 1024 tokens still leave pieces empty when split eight ways
    ctx = tuple(int(c) for c in rng.integers(256, 1500, size=B))
    kv = synth.paged_kv(B + W, "kv", ctx, hkv, spare_blocks=2)
    q = synth.normal_bf16(B * W, "q", (B, W, hq, 128), std=0.5)
    a = run(dqd, dev, q, kv, hkv)
    assert np.array_equal(bits(a), bits(run(dqd, dev, q, kv, hkv)))
    monkeypatch.setenv("DQD_ATTN_PERSIST", "0")
    assert np.array_equal(bits(a), bits(run(dqd, dev, q, kv, hkv))), "one CTA per unit"
    monkeypatch.delenv("DQD_ATTN_PERSIST")
    assert_close(f64(a), ref(q, kv, hkv), what=f"tc balanced tail B={B} W={W} {hq}/{hkv}")
    monkeypatch.setenv("DQD_ATTN_TAIL", "0")
    assert_close(f64(a), f64(run(dqd, dev, q, kv, hkv)), what="whole items")
    assert dqd.device_errors() == 0


@pytest.mark.parametrize("B,W,hq,hkv,lo,hi,cb", [
    (64, 16, 32, 8, 16, 700, None),   # 64 rows (two Q slots), 1-6 tiles per unit, odd and even counts
    (40, 16, 64, 8, 16, 900, None),   # 128 rows (one Q slot)
    (64, 6, 32, 8, 200, 2000, 8),     # 24 rows, 8-block chunks: many units per CTA, empty ones too
    (20, 16, 64, 8, 256, 1500, None), # 128 rows, a balanced tail of eight pieces per item
    (256, 6, 32, 8, 64, 400, None),   # the most sequences the longest-first order covers
    (300, 6, 32, 8, 64, 400, None),   # more sequences than the longest-first order covers: index order
])
def test_tensor_core_persistent_queue(dev, dqd, monkeypatch, B, W, hq, hkv, lo, hi, cb):
    """The persistent tcgen05 form with many units per CTA, taken from the
    queue in the workspace's counter region (longest contexts first, up to 256
    sequences): the same bits as one CTA per unit (the two softmax groups'
    accumulators are combined symmetrically, so the schedule cannot change the
    result), the same bits on reruns over one workspace, and the queue's
    counters back at zero after every call."""
    if cb is not None:
        monkeypatch.setenv("DQD_ATTN_CHUNK_BLOCKS", str(cb))
    rng = np.random.default_rng(B * 1000 + W * 10 + hq)
    ctx = tuple(int(c) for c in rng.integers(max(lo, W), hi + 1, size=B))
    kv = synth.paged_kv(B * 3 + W, "kv", ctx, hkv, spare_blocks=2)
    q = synth.normal_bf16(B * 5 + W, "q", (B, W, hq, 128), std=0.5)
    maxc = max(ctx)
    need = dqd.gqa_decode_attn_workspace_bytes(B, W, hq, hkv, 128, maxc)
    assert need >= 65536, "the persistent form needs the counter region"
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    args = (bf(q, dev), bf(kv.k_pool, dev), bf(kv.v_pool, dev), i32(kv.block_table, dev),
            i32(np.asarray(ctx, np.int32), dev), maxc)
    outs = []
    for _ in range(3):
        outs.append(dqd.gqa_decode_attn(*args, ws=ws))
        torch.cuda.synchronize()
        assert int(torch.count_nonzero(ws[:8]).item()) == 0, "queue counters left nonzero"
    for o in outs[1:]:
        assert np.array_equal(bits(o), bits(outs[0])), "rerun differs"
    monkeypatch.setenv("DQD_ATTN_PERSIST", "0")
    assert np.array_equal(bits(outs[0]), bits(dqd.gqa_decode_attn(*args))), "one CTA per unit differs"
    # parity is carried by the bit comparison above (the one-CTA-per-unit form
    # meets the oracle at 1% in the tests before); against the oracle directly
    # at 2%: with these many short contexts a rare element of either form sits
    # just past 1%, the bf16 rounding of P (1.13x the 1% bound at 20 x 16 x 64)
    assert_close(f64(outs[0]), ref(q, kv, hkv), tol=2e-2, what=f"persistent tc B={B} W={W} {hq}/{hkv}")
    assert dqd.device_errors() == 0
