"""GPU parity of dq_gemm against the float64 oracle.

Dequantised weights must come back bit for bit through one-hot activations;
every other output must sit within |gpu - ref| <= 1e-2 (|ref| + rms(ref)).
Shapes span several 16-row tiles with ragged n, every m-tile width (1..64
and m-chunking past 64), split-K on and off, and ragged k for BF16/FP8."""
import os

import numpy as np
import pytest
import torch

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


@pytest.fixture
def splits(monkeypatch):
    def set_splits(v):
        if v is None:
            monkeypatch.delenv("DQD_GEMM_SPLITS", raising=False)
        else:
            monkeypatch.setenv("DQD_GEMM_SPLITS", str(v))
    yield set_splits
    monkeypatch.delenv("DQD_GEMM_SPLITS", raising=False)


def _f32(bits_):
    return (np.asarray(bits_, np.uint16).astype(np.uint32) << 16).view(np.float32)


class Case:
    """One weight in the three formats' host (oracle) and device forms."""

    def __init__(self, dqd, dev, wtype, n, k, seed=0, outliers=0):
        self.wtype, self.n, self.k = wtype, n, k
        if wtype == oracle.W_INT4_G128:
            self.wq = synth.int4_weight(seed, "w", n, k)
            p = dqd.pack_int4_g128(u8(self.wq.codes, dev), bf(self.wq.scales, dev), u8(self.wq.zeros, dev))
            self.weight = dqd.Weight.int4(p)
            self.host = (self.wq.codes, self.wq.scales, self.wq.zeros)
        else:
            w = synth.bf16_weight(seed, "w", n, k, std=0.02, outlier_channels=outliers)
            self.w16 = w
            if wtype == oracle.W_BF16:
                self.weight = dqd.Weight.bf16(bf(w, dev))
                self.host = (w, None, None)
            else:
                codes, scales = dqd.quant_fp8_rowwise(bf(w, dev))
                self.weight = dqd.Weight.fp8(codes, scales)
                rc, rs = oracle.quant_fp8_rowwise(w)       # the oracle's own codes
                self.host = (rc, rs, None)

    def ref(self, x, rows=None):
        return oracle.dq_gemm(self.wtype, *self.host, x, rows=rows)


WT = [oracle.W_BF16, oracle.W_FP8_E4M3, oracle.W_INT4_G128]
WT_IDS = ["bf16", "fp8", "int4"]


@pytest.mark.parametrize("wtype", WT, ids=WT_IDS)
@pytest.mark.parametrize("m,n,k", [(1, 1024, 1024), (1, 40, 384), (3, 17, 256), (8, 100, 512),
                                   (9, 64, 1024), (16, 33, 768), (32, 130, 512), (33, 48, 256),
                                   (64, 80, 384), (100, 50, 256), (1, 4096, 2048)])
def test_against_oracle(dev, dqd, monkeypatch, wtype, m, n, k):
    # the warp-MMA kernels at every m-tile count (wide m otherwise goes to tcgen05;
    # the warp-MMA kernels still take it where tcgen05 cannot, e.g. k % 16 != 0)
    monkeypatch.setenv("DQD_GEMM_TC", "0")
    c = Case(dqd, dev, wtype, n, k, seed=m * 31 + n, outliers=6 if wtype != oracle.W_INT4_G128 else 0)
    x = synth.normal_bf16(m + k, "x", (m, k))
    y = dqd.dq_gemm(c.weight, bf(x, dev))
    assert y.shape == (m, n)
    assert_close(f64(y), c.ref(x), what=f"dq_gemm {WT_IDS[wtype]} m={m} n={n} k={k}")


@pytest.mark.parametrize("k", [8, 24, 264])
@pytest.mark.parametrize("m", [1, 5])
def test_bf16_ragged_k(dev, dqd, m, k):
    c = Case(dqd, dev, oracle.W_BF16, 37, k, seed=k)
    x = synth.normal_bf16(k, "x", (m, k))
    assert_close(f64(dqd.dq_gemm(c.weight, bf(x, dev))), c.ref(x), what=f"bf16 k={k}")


@pytest.mark.parametrize("k", [16, 48, 272])
def test_fp8_ragged_k(dev, dqd, k):
    c = Case(dqd, dev, oracle.W_FP8_E4M3, 21, k, seed=k)
    x = synth.normal_bf16(k, "x", (2, k))
    assert_close(f64(dqd.dq_gemm(c.weight, bf(x, dev))), c.ref(x), what=f"fp8 k={k}")


@pytest.fixture
def cluster(monkeypatch):
    def set_cluster(on):
        monkeypatch.setenv("DQD_GEMM_CLUSTER", "1" if on else "0")
    yield set_cluster
    monkeypatch.delenv("DQD_GEMM_CLUSTER", raising=False)


@pytest.mark.parametrize("wtype", WT, ids=WT_IDS)
@pytest.mark.parametrize("split", [1, 2, 3, 7, 8, 64])
@pytest.mark.parametrize("m", [5, 20, 40])
@pytest.mark.parametrize("on", [True, False], ids=["dsmem", "global"])
def test_every_split_count(dev, dqd, monkeypatch, splits, cluster, wtype, split, m, on):
    """Up to 8 splits reduce inside a thread-block cluster; more, or with the
    cluster path switched off, through global partials and a ticket."""
    monkeypatch.setenv("DQD_GEMM_TC", "0")
    splits(split)
    cluster(on)
    c = Case(dqd, dev, wtype, 96, 2048, seed=split)
    x = synth.normal_bf16(split + m, "x", (m, 2048))
    y = dqd.dq_gemm(c.weight, bf(x, dev))
    assert_close(f64(y), c.ref(x), what=f"splits={split} m={m}")


@pytest.mark.parametrize("wtype", WT, ids=WT_IDS)
@pytest.mark.parametrize("on", [True, False], ids=["dsmem", "global"])
def test_deterministic_with_split_k(dev, dqd, splits, cluster, wtype, on):
    splits(4)
    cluster(on)
    c = Case(dqd, dev, wtype, 512, 4096, seed=9)
    x = bf(synth.normal_bf16(9, "x", (4, 4096)), dev)
    ws_need = dqd.dq_gemm_workspace_bytes(c.weight, 4)
    assert (ws_need == 0) if on else (ws_need > 0)  # split-K inside a cluster needs no workspace
    a = bits(dqd.dq_gemm(c.weight, x))
    b = bits(dqd.dq_gemm(c.weight, x))
    assert np.array_equal(a, b)
    assert dqd.device_errors() == 0


@pytest.mark.parametrize("slots", ["2", "3"])
@pytest.mark.parametrize("warps", ["4", "8"])
@pytest.mark.parametrize("split", [None, 1, 3])
@pytest.mark.parametrize("m,n,k", [(1, 1024, 1024), (5, 200, 640), (9, 72, 384), (16, 500, 1536)])
def test_int4_cta_widths(dev, dqd, splits, monkeypatch, slots, warps, split, m, n, k):
    """INT4 at m <= 16 runs 8 or 4 tile warps per CTA over a 2- or 3-slot ring
    (the planner picks both per shape); every combination agrees with the
    oracle, with and without split-K, on ragged tile counts."""
    monkeypatch.setenv("DQD_GEMM_WARPS", warps)
    monkeypatch.setenv("DQD_GEMM_INT4_NS", slots)
    splits(split)
    c = Case(dqd, dev, oracle.W_INT4_G128, n, k, seed=m + n)
    x = synth.normal_bf16(m, "x", (m, k))
    assert_close(f64(dqd.dq_gemm(c.weight, bf(x, dev))), c.ref(x), what=f"int4 warps={warps} split={split}")


def _one_hot(m_rows, k, cols):
    x = np.zeros((m_rows, k), np.uint16)
    x[np.arange(len(cols)), cols] = 0x3F80
    return x


@pytest.mark.parametrize("m_rows", [8, 64, 256])
def test_one_hot_reads_back_int4_deq_bit_exact(dev, dqd, m_rows):
    n, k = 48, 256
    c = Case(dqd, dev, oracle.W_INT4_G128, n, k, seed=m_rows)
    deq = oracle.int4_dequant(*c.host)
    for start in range(0, k, m_rows):
        cols = np.arange(start, min(k, start + m_rows))
        y = bits(dqd.dq_gemm(c.weight, bf(_one_hot(len(cols), k, cols), dev)))
        assert np.array_equal(y, deq[:, cols].T)


@pytest.mark.parametrize("m_rows", [8, 256])
def test_one_hot_reads_back_bf16_bit_exact(dev, dqd, m_rows):
    n, k = 40, 256
    c = Case(dqd, dev, oracle.W_BF16, n, k, seed=m_rows)
    for start in range(0, k, m_rows):
        cols = np.arange(start, min(k, start + m_rows))
        y = bits(dqd.dq_gemm(c.weight, bf(_one_hot(len(cols), k, cols), dev)))
        assert np.array_equal(y, c.w16[:, cols].T)


def test_one_hot_reads_back_every_fp8_code(dev, dqd):
    """Every finite E4M3 code (subnormals, +-0, +-448) through the public API:
    y = bf16(fp32(e4m3(code) * scale)), the scale applied in fp32."""
    k = 256
    all_codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    n = 32
    codes = np.resize(all_codes, (n, k)).astype(np.uint8)
    codes[:, :len(all_codes)] = np.roll(all_codes, 1)[None, :]
    scales = (2.0 ** np.random.default_rng(2).integers(-12, 4, n) *
              np.random.default_rng(3).uniform(1, 2, n)).astype(np.float32)
    scales[0] = 1.0
    w = dqd.Weight.fp8(u8(codes, dev), torch.from_numpy(scales).to(dev))
    vals = oracle.e4m3_decode(codes)
    want = oracle.bf16_round((vals * scales.astype(np.float64)[:, None]).astype(np.float32).astype(np.float64))
    # A dot product with +0 terms turns a -0 weight into +0 (IEEE: -0 + +0 = +0),
    # so zeros are compared by value.
    want = np.where(want == 0x8000, 0, want).astype(np.uint16)
    for start in range(0, k, 128):
        cols = np.arange(start, start + 128)
        y = bits(dqd.dq_gemm(w, bf(_one_hot(128, k, cols), dev)))
        assert np.array_equal(y, want[:, cols].T)


def test_int4_zero_point_equal_to_codes_gives_exact_zero(dev, dqd):
    n, k = 64, 512
    codes = np.repeat(np.random.default_rng(4).integers(0, 16, (n, 4)).astype(np.uint8), 128, axis=1)
    zeros = codes[:, ::128].copy()
    scales = synth.uniform_bf16(4, "s", (n, 4), 0.005, 0.02)
    p = dqd.pack_int4_g128(u8(codes, dev), bf(scales, dev), u8(zeros, dev))
    y = dqd.dq_gemm(dqd.Weight.int4(p), bf(synth.normal_bf16(4, "x", (7, k)), dev))
    assert torch.count_nonzero(y.float()).item() == 0


def test_bf16_gemm_on_dequantised_int4_matches_int4_gemm(dev, dqd):
    n, k = 96, 1024
    c = Case(dqd, dev, oracle.W_INT4_G128, n, k, seed=5)
    deq = oracle.int4_dequant(*c.host)
    x = bf(synth.normal_bf16(5, "x", (3, k)), dev)
    a = f64(dqd.dq_gemm(c.weight, x))
    b = f64(dqd.dq_gemm(dqd.Weight.bf16(bf(deq, dev)), x))
    assert_close(a, b, what="int4 vs bf16(deq)")


def test_empty_and_degenerate(dev, dqd):
    c = Case(dqd, dev, oracle.W_BF16, 16, 64)
    y = dqd.dq_gemm(c.weight, torch.empty((0, 64), dtype=torch.bfloat16, device=dev))
    assert y.shape == (0, 16)
    # k = 0: the empty sum is zero
    w0 = dqd.Weight.bf16(torch.empty((20, 0), dtype=torch.bfloat16, device=dev))
    y = dqd.dq_gemm(w0, torch.empty((3, 0), dtype=torch.bfloat16, device=dev))
    torch.cuda.synchronize()
    assert y.shape == (3, 20) and torch.count_nonzero(y.float()).item() == 0


def test_workspace_too_small_is_rejected(dev, dqd, cluster):
    cluster(False)  # the global split-K path needs a workspace
    c = Case(dqd, dev, oracle.W_INT4_G128, 256, 4096)
    need = dqd.dq_gemm_workspace_bytes(c.weight, 2)
    assert need > 0
    x = bf(synth.normal_bf16(1, "x", (2, 4096)), dev)
    small = torch.zeros(need - 16, dtype=torch.uint8, device=dev)
    with pytest.raises(dqd.DqdError) as e:
        dqd.dq_gemm(c.weight, x, ws=small)
    assert e.value.status == dqd.DQD_ERR_WORKSPACE


@pytest.mark.parametrize("wtype", WT, ids=WT_IDS)
@pytest.mark.parametrize("m,n,k", [(1, 16, 4096), (8, 16, 8192), (3, 48, 128), (1, 8, 256), (2, 40, 2048),
                                   (1, 17, 8192), (7, 4112, 1024)])
def test_small_m_stream_shapes(dev, dqd, wtype, m, n, k):
    """Small m over long k, a single 16-row tile, fewer tiles than warps per
    CTA, ragged n and wide grids."""
    c = Case(dqd, dev, wtype, n, k, seed=m + n + k)
    x = synth.normal_bf16(m * n + k, "x", (m, k))
    a = dqd.dq_gemm(c.weight, bf(x, dev))
    assert_close(f64(a), c.ref(x), what=f"stream {WT_IDS[wtype]} m={m} n={n} k={k}")
    b = dqd.dq_gemm(c.weight, bf(x, dev))
    assert np.array_equal(bits(a), bits(b))  # piece order fixed: bit-identical reruns


def test_no_device_error_flags(dev, dqd):
    assert dqd.device_errors() == 0
