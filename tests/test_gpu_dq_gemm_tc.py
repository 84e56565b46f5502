"""GPU parity of the tensor-core (tcgen05) dq_gemm path taken at wide m (from
17 rows for every weight type), against the float64 oracle and
against the warp-MMA kernels on the same inputs.

Shapes span several 128-row weight tiles and 128-token chunks with ragged n
(partial 16-row tiles and CTAs with fewer than eight tiles), ragged m and
k from one group to 32 groups."""
import numpy as np
import pytest

import oracle
from memory_bound_decode_dq_gb300 import synth
from gpu_util import assert_close, bf, bits, f64, require_cuda, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_cuda()


@pytest.fixture(scope="module")
def dqd():
    from memory_bound_decode_dq_gb300 import dqd as m
    return m


def _weight(dqd, dev, n, k, seed):
    wq = synth.int4_weight(seed, "w", n, k)
    p = dqd.pack_int4_g128(u8(wq.codes, dev), bf(wq.scales, dev), u8(wq.zeros, dev))
    return wq, dqd.Weight.int4(p)


SHAPES = [(128, 128, 128), (129, 1000, 256), (256, 2048, 1024), (300, 48, 4096), (1024, 130, 512),
          (500, 4112, 384), (200, 16, 128), (384, 6144, 4096), (33, 300, 1024), (40, 4096, 4096),
          (64, 28672, 4096), (17, 300, 1024), (32, 4096, 4096), (16, 300, 1024)]  # the last: the warp-MMA side of the boundary


@pytest.mark.parametrize("m,n,k", SHAPES)
def test_against_oracle(dev, dqd, m, n, k):
    wq, w = _weight(dqd, dev, n, k, seed=m + n + k)
    x = synth.normal_bf16(m * 7 + k, "x", (m, k))
    y = dqd.dq_gemm(w, bf(x, dev))
    assert y.shape == (m, n)
    rows = None if n * m * k <= 2 ** 28 else np.unique(np.r_[0, n - 1, np.arange(0, n, 97)])
    ref = oracle.dq_gemm(oracle.W_INT4_G128, wq.codes, wq.scales, wq.zeros, x, rows=rows)
    got = f64(y) if rows is None else f64(y)[:, rows]
    assert_close(got, ref, what=f"tc int4 m={m} n={n} k={k}")


@pytest.mark.parametrize("m,n,k", [(128, 256, 512), (777, 1040, 2048)])
def test_matches_warp_mma_path(dev, dqd, monkeypatch, m, n, k):
    wq, w = _weight(dqd, dev, n, k, seed=3)
    x = bf(synth.normal_bf16(3, "x", (m, k)), dev)
    a = f64(dqd.dq_gemm(w, x))
    monkeypatch.setenv("DQD_GEMM_TC", "0")
    b = f64(dqd.dq_gemm(w, x))
    assert_close(a, b, what="tcgen05 vs mma.sync")


def test_rerun_is_bit_identical(dev, dqd):
    _, w = _weight(dqd, dev, 3000, 1024, seed=11)
    x = bf(synth.normal_bf16(11, "x", (640, 1024)), dev)
    assert np.array_equal(bits(dqd.dq_gemm(w, x)), bits(dqd.dq_gemm(w, x)))


def test_one_hot_reads_back_dequantised_weights(dev, dqd):
    """128 one-hot tokens per call: y[t] = bf16((q - z) * s) of column t,
    bit for bit, over ragged n."""
    n, k = 200, 384
    wq, w = _weight(dqd, dev, n, k, seed=21)
    deq = oracle.int4_dequant(wq.codes, wq.scales, wq.zeros)
    for start in range(0, k, 128):
        x = np.zeros((128, k), np.uint16)
        x[np.arange(128), start + np.arange(128)] = 0x3F80
        y = bits(dqd.dq_gemm(w, bf(x, dev)))
        assert np.array_equal(y, deq[:, start:start + 128].T)


def test_no_device_error_flags(dev, dqd):
    assert dqd.device_errors() == 0


@pytest.mark.parametrize("split", [1, 2, 3, 5, 10])
def test_every_split_count(dev, dqd, monkeypatch, split):
    """k split on group boundaries (the last split shorter), partials summed
    by the last-arriving CTA in split order."""
    monkeypatch.setenv("DQD_GEMM_SPLITS", str(split))
    m, n, k = 300, 500, 1280
    wq, w = _weight(dqd, dev, n, k, seed=split)
    x = synth.normal_bf16(split, "x", (m, k))
    xd = bf(x, dev)
    y = dqd.dq_gemm(w, xd)
    ref = oracle.dq_gemm(oracle.W_INT4_G128, wq.codes, wq.scales, wq.zeros, x)
    assert_close(f64(y), ref, what=f"tc splits={split}")
    assert np.array_equal(bits(y), bits(dqd.dq_gemm(w, xd)))


def test_planner_splits_a_small_grid(dev, dqd):
    """384 tokens over a 4096 x 14336 weight is 64 CTAs unsplit: the planner
    splits k, which needs workspace."""
    _, w = _weight(dqd, dev, 4096, 14336, seed=1)
    assert dqd.dq_gemm_workspace_bytes(w, 384) > 0


def _dense(dqd, dev, wtype, n, k, seed):
    w = synth.bf16_weight(seed, "w", n, k, std=0.02, outlier_channels=6)
    if wtype == oracle.W_BF16:
        return dqd.Weight.bf16(bf(w, dev)), (w, None, None)
    codes, scales = dqd.quant_fp8_rowwise(bf(w, dev))
    rc, rs = oracle.quant_fp8_rowwise(w)
    return dqd.Weight.fp8(codes, scales), (rc, rs, None)


DENSE = [oracle.W_BF16, oracle.W_FP8_E4M3]


@pytest.mark.parametrize("wtype", DENSE, ids=["bf16", "fp8"])
@pytest.mark.parametrize("m,n,k", [(48, 130, 512), (49, 1000, 80), (64, 16, 4096), (100, 2050, 272),
                                   (300, 64, 1024), (48, 10240, 8192), (1024, 300, 128)])
def test_dense_against_oracle(dev, dqd, wtype, m, n, k):
    """Ragged k (a partial last slab), ragged n and m, one-slab k, big shapes
    (every weight type takes this path from 17 rows)."""
    w, host = _dense(dqd, dev, wtype, n, k, seed=m + n + k)
    x = synth.normal_bf16(m + 2 * k, "x", (m, k))
    y = dqd.dq_gemm(w, bf(x, dev))
    rows = None if n * m * k <= 2 ** 28 else np.unique(np.r_[0, n - 1, np.arange(0, n, 127)])
    ref = oracle.dq_gemm(wtype, *host, x, rows=rows)
    got = f64(y) if rows is None else f64(y)[:, rows]
    assert_close(got, ref, what=f"tc {wtype} m={m} n={n} k={k}")


@pytest.mark.parametrize("wtype", DENSE, ids=["bf16", "fp8"])
@pytest.mark.parametrize("split", [1, 2, 3, 7])
def test_dense_every_split(dev, dqd, monkeypatch, wtype, split):
    monkeypatch.setenv("DQD_GEMM_SPLITS", str(split))
    m, n, k = 56, 300, 1008
    w, host = _dense(dqd, dev, wtype, n, k, seed=split)
    x = synth.normal_bf16(split, "x", (m, k))
    xd = bf(x, dev)
    y = dqd.dq_gemm(w, xd)
    assert_close(f64(y), oracle.dq_gemm(wtype, *host, x), what=f"tc {wtype} splits={split}")
    assert np.array_equal(bits(y), bits(dqd.dq_gemm(w, xd)))


@pytest.mark.parametrize("wtype", DENSE, ids=["bf16", "fp8"])
def test_dense_matches_warp_mma_path(dev, dqd, monkeypatch, wtype):
    w, _ = _dense(dqd, dev, wtype, 2000, 2048, seed=4)
    x = bf(synth.normal_bf16(4, "x", (64, 2048)), dev)
    a = f64(dqd.dq_gemm(w, x))
    monkeypatch.setenv("DQD_GEMM_TC", "0")
    b = f64(dqd.dq_gemm(w, x))
    assert_close(a, b, what="tcgen05 vs mma.sync")


def test_dense_no_device_error_flags(dev, dqd):
    assert dqd.device_errors() == 0


@pytest.mark.parametrize("m,n,k", [(9, 300, 1024), (16, 6144, 4096), (12, 17, 72)])
def test_bf16_small_m_on_tensor_cores(dev, dqd, monkeypatch, m, n, k):
    """BF16 below its threshold, forced onto the tensor cores: N = 16 tokens
    per CTA, most of them zero padding."""
    monkeypatch.setenv("DQD_GEMM_TC", "1")
    w, host = _dense(dqd, dev, oracle.W_BF16, n, k, seed=m + n)
    x = synth.normal_bf16(m + k, "x", (m, k))
    rows = None if n <= 1024 else np.unique(np.r_[0, n - 1, np.arange(0, n, 97)])
    got = f64(dqd.dq_gemm(w, bf(x, dev)))
    ref = oracle.dq_gemm(oracle.W_BF16, *host, x, rows=rows)
    assert_close(got if rows is None else got[:, rows], ref, what=f"tc bf16 m={m}")


RING_N = [16, 32, 48, 96, 144, 192, 256]


@pytest.mark.parametrize("ntok", RING_N)
@pytest.mark.parametrize("wtype", [oracle.W_BF16, oracle.W_FP8_E4M3, oracle.W_INT4_G128], ids=["bf16", "fp8", "int4"])
def test_every_ring_layout(dev, dqd, monkeypatch, wtype, ntok):
    """Every ring layout the tokens per CTA select (N = 16 .. 256: weight, code
    and activation rings of different depths) over 128 slabs in one CTA, so
    that each slot is reused many times by the two MMA issuers: results agree
    with the oracle and no bounded wait gives up."""
    monkeypatch.setenv("DQD_GEMM_TC", "1")
    monkeypatch.setenv("DQD_GEMM_TC_N", str(ntok))
    monkeypatch.setenv("DQD_GEMM_SPLITS", "1")
    m, n, k = ntok - 5, 256, 8192
    x = synth.normal_bf16(ntok, "x", (m, k))
    if wtype == oracle.W_INT4_G128:
        wq, w = _weight(dqd, dev, n, k, seed=ntok)
        ref = oracle.dq_gemm(wtype, wq.codes, wq.scales, wq.zeros, x)
    else:
        w, host = _dense(dqd, dev, wtype, n, k, seed=ntok)
        ref = oracle.dq_gemm(wtype, *host, x)
    assert dqd.dq_gemm_workspace_bytes(w, m) == 0  # one split: the whole k in each CTA
    assert_close(f64(dqd.dq_gemm(w, bf(x, dev))), ref, what=f"tc {wtype} N={ntok}")
    assert dqd.device_errors() == 0


@pytest.mark.parametrize("ntok", [16, 32, 48, 64, 96, 128])
@pytest.mark.parametrize("k,split", [(64, 1), (1008, 1), (8192, 1), (8192, 3), (4160, 5)])
def test_fp8_a_in_tensor_memory(dev, dqd, monkeypatch, ntok, k, split):
    """FP8 at N <= 128 keeps the dequantised weights in tensor memory
    (tcgen05.st by the dequantising warps, A read from tensor memory by the
    MMA) in stages of two slabs, whose last one may lie beyond k (one-slab k,
    ragged k, an odd last split). Within tolerance of the oracle; within one
    bf16 ulp plus fp32 reordering error of the kernel with A in shared memory
    (the two issuers' partial sums are split differently); bit-identical on a
    rerun."""
    monkeypatch.setenv("DQD_GEMM_TC", "1")
    monkeypatch.setenv("DQD_GEMM_TC_N", str(ntok))
    monkeypatch.setenv("DQD_GEMM_SPLITS", str(split))
    monkeypatch.setenv("DQD_GEMM_TC_ATM", "1")  # tensor memory up to N = 128
    m, n = ntok - 3 if ntok > 16 else 11, 300
    w, host = _dense(dqd, dev, oracle.W_FP8_E4M3, n, k, seed=ntok + k)
    x = synth.normal_bf16(ntok + k + split, "x", (m, k))
    xd = bf(x, dev)
    a = dqd.dq_gemm(w, xd)
    assert np.array_equal(bits(a), bits(dqd.dq_gemm(w, xd)))
    assert_close(f64(a), oracle.dq_gemm(oracle.W_FP8_E4M3, *host, x), what=f"tc fp8 tmem-A N={ntok} k={k}")
    monkeypatch.setenv("DQD_GEMM_TC_ATM", "0")
    b = f64(dqd.dq_gemm(w, xd))
    # one bf16 ulp, plus what reordering an fp32 sum of k products can move
    # (some 256 sequential adds per accumulator at k = 8192, each within 2^-24
    # of the running sum; 1e-3 of the output rms bounds it here)
    tol = 2.0 ** -7 * np.maximum(np.abs(f64(a)), np.abs(b)) + 1e-3 * np.sqrt(np.mean(b ** 2))
    assert np.all(np.abs(f64(a) - b) <= tol)
    assert dqd.device_errors() == 0


@pytest.mark.parametrize("ntok", [16, 32, 48, 64, 96, 128])
@pytest.mark.parametrize("k,split", [(128, 1), (1024, 1), (8192, 1), (8192, 3), (4224, 5)])
def test_int4_a_in_tensor_memory(dev, dqd, monkeypatch, ntok, k, split):
    """INT4 with the dequantised weights in tensor memory, one 128-k group per
    stage, row-per-thread unpacking of the packed blocks: within tolerance of
    the oracle, within one bf16 ulp plus fp32 reordering of the form with A in
    shared memory, bit-identical on a rerun; ragged n (a partial row tile and
    a CTA with fewer than eight tiles), one-group k, split k."""
    monkeypatch.setenv("DQD_GEMM_TC", "1")
    monkeypatch.setenv("DQD_GEMM_TC_N", str(ntok))
    monkeypatch.setenv("DQD_GEMM_SPLITS", str(split))
    monkeypatch.setenv("DQD_GEMM_TC_ATM", "1")
    m, n = ntok - 3 if ntok > 16 else 11, 300
    wq, w = _weight(dqd, dev, n, k, seed=ntok + k)
    x = synth.normal_bf16(ntok + k + split, "x", (m, k))
    xd = bf(x, dev)
    a = dqd.dq_gemm(w, xd)
    assert np.array_equal(bits(a), bits(dqd.dq_gemm(w, xd)))
    assert_close(f64(a), oracle.dq_gemm(oracle.W_INT4_G128, wq.codes, wq.scales, wq.zeros, x),
                 what=f"tc int4 tmem-A N={ntok} k={k}")
    monkeypatch.setenv("DQD_GEMM_TC_ATM", "0")
    b = f64(dqd.dq_gemm(w, xd))
    tol = 2.0 ** -7 * np.maximum(np.abs(f64(a)), np.abs(b)) + 1e-3 * np.sqrt(np.mean(b ** 2))
    assert np.all(np.abs(f64(a) - b) <= tol)
    assert dqd.device_errors() == 0


@pytest.mark.parametrize("wtype", ["int4", "fp8"])
def test_one_hot_reads_back_tensor_memory_weights(dev, dqd, monkeypatch, wtype):
    """One-hot tokens through the tensor-memory form (N = 64): y[t] is the
    dequantised weight of column t, bit for bit, for every k position of two
    groups (every nibble and column of the unpacking), over ragged n."""
    monkeypatch.setenv("DQD_GEMM_TC", "1")
    monkeypatch.setenv("DQD_GEMM_TC_N", "64")
    monkeypatch.setenv("DQD_GEMM_SPLITS", "1")
    n, k = 200, 256
    if wtype == "int4":
        wq, w = _weight(dqd, dev, n, k, seed=23)
        deq = oracle.int4_dequant(wq.codes, wq.scales, wq.zeros)
        scale = None
    else:
        w, (rc, rs, _) = _dense(dqd, dev, oracle.W_FP8_E4M3, n, k, seed=23)
        deq, scale = None, rs
    for start in range(0, k, 64):
        x = np.zeros((64, k), np.uint16)
        x[np.arange(64), start + np.arange(64)] = 0x3F80
        y = dqd.dq_gemm(w, bf(x, dev))
        if wtype == "int4":
            assert np.array_equal(bits(y), deq[:, start:start + 64].T)
        else:
            # FP8: bf16(code value * row scale), the product of two exact factors rounded once
            ref = oracle.dq_gemm(oracle.W_FP8_E4M3, rc, rs, None, x.view(np.uint16))
            assert_close(f64(y), ref, what="fp8 one-hot")
    assert dqd.device_errors() == 0
