"""GPU parity of dq_gemm_qkv_rope_append, the QKV projection fused with RoPE
and the paged KV append.

The fused call must reproduce the two-call chain dq_gemm -> rope_kv_append bit
for bit (q_out, K pool, V pool) on every epilogue the projection can take: the
warp-MMA kernels unsplit, split through a thread-block cluster and split
through global partials, and the tcgen05 kernel unsplit and split; for BF16,
FP8-E4M3 and INT4 g128 weights and for bf16 and FP8 caches. Against the
float64 oracle (its projection in float64, rotated in float64: the plain
definition, without the bf16 rounding of the projection's output that both
GPU forms take before rotating) q and k sit within the floating-point
tolerance (bounded per rotation pair, see assert_close_pairs) and v equals
the oracle's projection within the elementwise tolerance; attending over the
appended cache matches the oracle's attention."""
import math

import numpy as np
import pytest
import torch

import oracle
from memory_bound_decode_dq_gb300 import synth
from gpu_util import assert_close, bf, bits, f64, i32, require_cuda, u8

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def dev():
    return require_cuda()


@pytest.fixture(scope="module")
def dqd():
    from memory_bound_decode_dq_gb300 import dqd as m
    return m


class Weight:
    """A QKV weight in host (oracle) and device form."""

    def __init__(self, dqd, dev, wtype, n, k, seed):
        self.wtype = wtype
        if wtype == oracle.W_INT4_G128:
            wq = synth.int4_weight(seed, "wqkv", n, k)
            self.weight = dqd.Weight.int4(dqd.pack_int4_g128(u8(wq.codes, dev), bf(wq.scales, dev),
                                                             u8(wq.zeros, dev)))
            self.host = (wq.codes, wq.scales, wq.zeros)
        else:
            w = synth.bf16_weight(seed, "wqkv", n, k, std=0.02)
            if wtype == oracle.W_BF16:
                self.weight = dqd.Weight.bf16(bf(w, dev))
                self.host = (w, None, None)
            else:
                codes, scales = dqd.quant_fp8_rowwise(bf(w, dev))
                self.weight = dqd.Weight.fp8(codes, scales)
                self.host = oracle.quant_fp8_rowwise(w) + (None,)

    def ref(self, x):
        return oracle.dq_gemm(self.wtype, *self.host, x)


def pools(dev, nblk, hkv, fp8, seed):
    if fp8:
        k = synth.e4m3_codes(seed, "kp8", (nblk, hkv, 16, D))
        v = synth.e4m3_codes(seed, "vp8", (nblk, hkv, 16, D))
        return u8(k, dev), u8(v, dev)
    return bf(synth.normal_bf16(seed, "kp", (nblk, hkv, 16, D)), dev), \
        bf(synth.normal_bf16(seed, "vp", (nblk, hkv, 16, D)), dev)


def raw(t):
    return t.view(torch.uint8).cpu().numpy() if t.dtype == torch.uint8 else bits(t)


PATHS = {
    # name: environment of the planner's test hooks
    "warp_unsplit": {"DQD_GEMM_TC": "0", "DQD_GEMM_SPLITS": "1"},
    "warp_cluster": {"DQD_GEMM_TC": "0", "DQD_GEMM_SPLITS": "4", "DQD_GEMM_CLUSTER": "1"},
    "warp_global": {"DQD_GEMM_TC": "0", "DQD_GEMM_SPLITS": "3", "DQD_GEMM_CLUSTER": "0"},
    "tc_unsplit": {"DQD_GEMM_TC": "1", "DQD_GEMM_SPLITS": "1"},
    "tc_split": {"DQD_GEMM_TC": "1", "DQD_GEMM_SPLITS": "2"},
    "planned": {},
}

WT = [oracle.W_BF16, oracle.W_FP8_E4M3, oracle.W_INT4_G128]
WT_IDS = ["bf16", "fp8", "int4"]
KS, VS = 1.0 / 64, 1.0 / 128


def run_both(dqd, dev, wt, b, w, hq, hkv, k, ctx, fp8, base, seed, x_div=1):
    """The fused call and the two-call chain on identical inputs; returns
    their (q_out, K pool, V pool) and the host inputs. x ~ N(0, 1) / x_div
    (a power of two: exact in bf16)."""
    n = (hq + 2 * hkv) * D
    W_ = Weight(dqd, dev, wt, n, k, seed)
    x = synth.normal_bf16(seed, "x", (b * w, k))
    if x_div != 1:
        x = oracle.bf16_round(oracle.bf16_to_f64(x) / x_div)
    ctx = np.asarray(ctx, np.int32)
    table, nblk = synth.block_table(seed, "tbl", ctx, spare_blocks=2)
    t, c = i32(table, dev), i32(ctx, dev)
    kp1, vp1 = pools(dev, nblk, hkv, fp8, seed)
    kp2, vp2 = kp1.clone(), vp1.clone()
    q1 = dqd.dq_gemm_qkv_rope_append(W_.weight, bf(x, dev), b, w, hq, hkv, kp1, vp1, t, c, rope_base=base,
                                     k_scale=KS, v_scale=VS)
    qkv = dqd.dq_gemm(W_.weight, bf(x, dev))
    q2 = dqd.rope_kv_append(qkv, b, w, hq, hkv, kp2, vp2, t, c, rope_base=base, k_scale=KS, v_scale=VS)
    torch.cuda.synchronize()
    return (q1, kp1, vp1), (q2, kp2, vp2), (W_, x, ctx, table, nblk, qkv)


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("wt", WT, ids=WT_IDS)
@pytest.mark.parametrize("fp8", [False, True], ids=["bf16kv", "fp8kv"])
def test_fused_equals_two_calls_bit_for_bit(dev, dqd, monkeypatch, path, wt, fp8):
    for key in ("DQD_GEMM_TC", "DQD_GEMM_SPLITS", "DQD_GEMM_CLUSTER"):
        monkeypatch.delenv(key, raising=False)
    for key, val in PATHS[path].items():
        monkeypatch.setenv(key, val)
    # 3 sequences x 6 verify positions (m = 18: one 32-row tile of the tcgen05
    # kernel, three 8-token tiles of the warp-MMA ones), 8 / 2 heads
    b, w, hq, hkv, k = 3, 6, 8, 2, 1024
    fused, chain, _ = run_both(dqd, dev, wt, b, w, hq, hkv, k, (6, 300, 1000), fp8, 500000.0, 7 + wt)
    for name, a, c in zip(("q_out", "K pool", "V pool"), fused, chain):
        assert np.array_equal(raw(a), raw(c)), f"{path} {WT_IDS[wt]}: {name} differs from the two-call chain"
    assert dqd.device_errors() == 0


def assert_close_pairs(gpu, ref, what):
    """The tolerance rule for rotated outputs: |gpu - ref| <= 1e-2 (|pair| +
    rms(ref)) with |pair| the norm of the (2i, 2i+1) pair the element belongs
    to. The rotation is an isometry of each pair, so the projection's
    elementwise bound holds for the pair's norm, not for each rotated
    component: a component turned near zero still carries the rounding of its
    large partner."""
    gpu = np.asarray(gpu, np.float64).reshape(-1, 2)
    ref = np.asarray(ref, np.float64).reshape(-1, 2)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    bound = 1e-2 * (np.linalg.norm(ref, axis=1, keepdims=True) + rms)
    bad = np.abs(gpu - ref) > bound
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside the pair tolerance"


def oracle_rotated(W_, x, b, w, hq, hkv, ctx, table, nblk, base):
    """The oracle's projection (float64) with q and k rotated in float64 at
    each token's position, and the pool row of each token's append."""
    y = W_.ref(x).reshape(b * w, hq + 2 * hkv, D)
    pos = np.array([ctx[r] - w + i for r in range(b) for i in range(w)], np.float64)
    rq = oracle.rope(y[:, :hq].reshape(-1, D), np.repeat(pos, hq), base).reshape(b, w, hq, D)
    rk = oracle.rope(y[:, hq:hq + hkv].reshape(-1, D), np.repeat(pos, hkv), base).reshape(b, w, hkv, D)
    rv = y[:, hq + hkv:].reshape(b, w, hkv, D)
    slot = oracle.rope_kv_append(oracle.bf16_round(y.reshape(b * w, -1)), b, w, hq, hkv, base, ctx, table,
                                 nblk)[3]
    return rq, rk, rv, slot


@pytest.mark.parametrize("wt", WT, ids=WT_IDS)
@pytest.mark.parametrize("b,w,hq,hkv,k,ctx", [
    (1, 1, 32, 8, 4096, (8192,)),                # 8B decode, batch 1
    (2, 16, 32, 8, 4096, (16, 2000)),            # verify width 16
    (4, 1, 64, 8, 1024, (1, 17, 130, 3000)),     # 70B head counts
    (2, 2, 16, 2, 1024, (5, 131072)),            # positions up to 2^17
])
def test_against_oracle(dev, dqd, wt, b, w, hq, hkv, k, ctx):
    fused, _, (W_, x, ctx, table, nblk, _) = run_both(dqd, dev, wt, b, w, hq, hkv, k, ctx, False, 500000.0,
                                                      11 + b + wt)
    q, kp, vp = fused
    rq, rk, rv, slot = oracle_rotated(W_, x, b, w, hq, hkv, ctx, table, nblk, 500000.0)
    assert_close_pairs(f64(q), rq, what=f"{WT_IDS[wt]} rotated q")
    kb, vb = f64(kp).reshape(-1, D), f64(vp).reshape(-1, D)
    got_k = np.stack([kb[slot[r, i] + 16 * g] for r in range(b) for i in range(w) for g in range(hkv)])
    got_v = np.stack([vb[slot[r, i] + 16 * g] for r in range(b) for i in range(w) for g in range(hkv)])
    assert_close_pairs(got_k, rk.reshape(-1, D), what=f"{WT_IDS[wt]} appended k")
    assert_close(got_v, rv.reshape(-1, D), what=f"{WT_IDS[wt]} appended v")


def test_append_then_attend(dev, dqd):
    """The fused step followed by the attention equals the oracle's attention
    with the oracle's rotated q over the oracle-appended cache.

    Conditioning: the projection's outputs reach the GPU's rotation rounded to
    bf16 (as the two-call chain does), the oracle rotates them unrounded, and
    a softmax amplifies such differences by the spread of its logits. With x ~
    N(0, 1/16) the new tokens' q, k, v have about the pool's unit scale, and a
    softmax scale of 1/(4 sqrt(d)) keeps the logits' spread near one: the
    correct chain then stays within 0.4 of the tolerance (emulated on the CPU)
    while a k rotated one position off exceeds it 11-fold."""
    b, w, hq, hkv, k = 2, 5, 32, 8, 2048
    fused, _, (W_, x, ctx, table, nblk, _) = run_both(dqd, dev, oracle.W_INT4_G128, b, w, hq, hkv, k,
                                                      (77, 400), False, 10000.0, 21, x_div=4)
    q, kp, vp = fused
    scale = 1 / (4 * math.sqrt(D))
    out = dqd.gqa_decode_attn(q, kp, vp, i32(table, dev), i32(ctx, dev), int(ctx.max()), softmax_scale=scale)
    rq, rk, rv, slot = oracle_rotated(W_, x, b, w, hq, hkv, ctx, table, nblk, 10000.0)
    # the pools before the append, as run_both drew them; the cache and q hold bf16
    kref = synth.normal_bf16(21, "kp", (nblk, hkv, 16, D)).reshape(-1, D).copy()
    vref = synth.normal_bf16(21, "vp", (nblk, hkv, 16, D)).reshape(-1, D).copy()
    for r in range(b):
        for i in range(w):
            for g in range(hkv):
                kref[slot[r, i] + 16 * g] = oracle.bf16_round(rk[r, i, g])
                vref[slot[r, i] + 16 * g] = oracle.bf16_round(rv[r, i, g])
    ref = oracle.gqa_decode_attn(oracle.bf16_round(rq), kref.reshape(nblk, hkv, 16, D),
                                 vref.reshape(nblk, hkv, 16, D), table, ctx, hkv, scale)
    assert_close(f64(out), ref, what="fused append then attend")


def test_out_of_range_table_entry_is_clamped_and_reported(dev, dqd):
    assert dqd.device_errors() == 0
    b, w, hq, hkv, k = 1, 2, 8, 2, 512
    W_ = Weight(dqd, dev, oracle.W_BF16, (hq + 2 * hkv) * D, k, 3)
    x = synth.normal_bf16(3, "x", (b * w, k))
    ctx = np.array([40], np.int32)
    table, nblk = synth.block_table(3, "tbl", ctx)
    table[0, 2] = nblk + 9
    kp = torch.zeros((nblk, hkv, 16, D), dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    dqd.dq_gemm_qkv_rope_append(W_.weight, bf(x, dev), b, w, hq, hkv, kp, vp, i32(table, dev), i32(ctx, dev))
    assert dqd.device_errors() == dqd.DQD_DEVICE_ERR_BAD_INPUT
    assert torch.count_nonzero(vp[nblk - 1].float()).item() > 0
    assert dqd.device_errors() == 0


def test_rejects_bad_arguments(dev, dqd):
    W_ = Weight(dqd, dev, oracle.W_BF16, 12 * D, 256, 4)
    x = bf(synth.normal_bf16(4, "x", (2, 256)), dev)
    kp = torch.zeros((4, 2, 16, D), dtype=torch.bfloat16, device=dev)
    t, c = i32(np.zeros((2, 4), np.int32), dev), i32(np.array([5, 5], np.int32), dev)
    with pytest.raises(ValueError):
        dqd.dq_gemm_qkv_rope_append(W_.weight, x, 2, 1, 8, 3, kp, kp, t, c)     # n != (hq + 2 hkv) * 128
    with pytest.raises(dqd.DqdError):
        dqd.dq_gemm_qkv_rope_append(W_.weight, x, 2, 1, 8, 2, kp, kp, t, c, rope_base=0.5)


def test_no_device_error_flags(dev, dqd):
    assert dqd.device_errors() == 0
