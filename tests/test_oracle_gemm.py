"""Pins for the oracle's dq_gemm: y = x * deq(W)^T in float64.

Checked against NumPy matmul on weights decoded by torch's own casts (a
library path sharing nothing with the oracle's C), exact special cases, and
one-hot activations that read single weights back."""
import numpy as np
import pytest
import torch

from memory_bound_decode_dq_gb300 import synth
from oracle import W_BF16, W_FP8_E4M3, W_INT4_G128


def _f(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _torch_deq_int4(wq):
    s = np.repeat(_f(wq.scales), 128, axis=1).astype(np.float32)
    z = np.repeat(wq.zeros, 128, axis=1).astype(np.float32)
    prod = torch.from_numpy((wq.codes.astype(np.float32) - z) * s)
    return prod.to(torch.bfloat16).to(torch.float64).numpy()


@pytest.mark.parametrize("m,n,k", [(1, 64, 256), (3, 48, 256), (4, 17, 384)])
def test_bf16_against_numpy(oracle_lib, m, n, k):
    w = synth.bf16_weight(11, "w", n, k)
    x = synth.normal_bf16(11, "x", (m, k))
    y = oracle_lib.dq_gemm(W_BF16, w, None, None, x)
    np.testing.assert_allclose(y, _f(x) @ _f(w).T, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("m,n,k", [(1, 64, 256), (4, 33, 256)])
def test_fp8_against_torch_decode(oracle_lib, m, n, k):
    w = synth.bf16_weight(12, "w", n, k, outlier_channels=6)
    codes, scales = oracle_lib.quant_fp8_rowwise(w)
    x = synth.normal_bf16(12, "x", (m, k))
    y = oracle_lib.dq_gemm(W_FP8_E4M3, codes, scales, None, x)
    wv = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ref = (_f(x) @ wv.T) * scales.astype(np.float64)[None, :]
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    # and the FP8 GEMM stays close to the BF16 GEMM it approximates
    y16 = oracle_lib.dq_gemm(W_BF16, w, None, None, x)
    assert np.abs(y - y16).max() <= 0.07 * np.sqrt(np.mean(y16 ** 2))


@pytest.mark.parametrize("m,n,k", [(1, 64, 256), (4, 20, 512)])
def test_int4_against_torch_deq(oracle_lib, m, n, k):
    wq = synth.int4_weight(13, "w", n, k)
    x = synth.normal_bf16(13, "x", (m, k))
    y = oracle_lib.dq_gemm(W_INT4_G128, wq.codes, wq.scales, wq.zeros, x)
    np.testing.assert_allclose(y, _f(x) @ _torch_deq_int4(wq).T, rtol=1e-12, atol=1e-12)


def test_int4_zero_point_equal_to_codes_gives_zero(oracle_lib):
    n, k = 32, 256
    codes = np.repeat(np.random.default_rng(3).integers(0, 16, (n, 2)).astype(np.uint8), 128, axis=1)
    wq = synth.Int4Weight(codes=codes, scales=synth.uniform_bf16(3, "s", (n, 2), 0.005, 0.02),
                          zeros=codes[:, ::128].copy(), n=n, k=k)
    x = synth.normal_bf16(3, "x", (5, k))
    y = oracle_lib.dq_gemm(W_INT4_G128, wq.codes, wq.scales, wq.zeros, x)
    assert np.all(y == 0.0)


def test_one_hot_reads_back_weights(oracle_lib):
    n, k = 24, 256
    wq = synth.int4_weight(4, "w", n, k)
    eye = np.zeros((k, k), np.uint16)
    eye[np.arange(k), np.arange(k)] = 0x3F80           # bf16 1.0
    y = oracle_lib.dq_gemm(W_INT4_G128, wq.codes, wq.scales, wq.zeros, eye)
    assert np.array_equal(y.T, _f(oracle_lib.int4_dequant(wq.codes, wq.scales, wq.zeros)))
    w = synth.bf16_weight(4, "w16", n, k)
    y = oracle_lib.dq_gemm(W_BF16, w, None, None, eye)
    assert np.array_equal(y.T, _f(w))
    codes, scales = oracle_lib.quant_fp8_rowwise(w)
    y = oracle_lib.dq_gemm(W_FP8_E4M3, codes, scales, None, eye)
    assert np.array_equal(y.T, oracle_lib.e4m3_decode(codes) * scales.astype(np.float64)[:, None])


def test_row_subset_equals_full(oracle_lib):
    wq = synth.int4_weight(5, "w", 50, 256)
    x = synth.normal_bf16(5, "x", (3, 256))
    full = oracle_lib.dq_gemm(W_INT4_G128, wq.codes, wq.scales, wq.zeros, x)
    rows = np.array([49, 0, 17, 17, 3])
    sub = oracle_lib.dq_gemm(W_INT4_G128, wq.codes, wq.scales, wq.zeros, x, rows=rows)
    assert np.array_equal(sub, full[:, rows])


def test_bf16_gemm_on_dequantised_int4_equals_int4_gemm(oracle_lib):
    wq = synth.int4_weight(6, "w", 40, 384)
    x = synth.normal_bf16(6, "x", (2, 384))
    deq = oracle_lib.int4_dequant(wq.codes, wq.scales, wq.zeros)
    a = oracle_lib.dq_gemm(W_INT4_G128, wq.codes, wq.scales, wq.zeros, x)
    b = oracle_lib.dq_gemm(W_BF16, deq, None, None, x)
    assert np.array_equal(a, b)


def test_rejects_bad_arguments(oracle_lib):
    wq = synth.int4_weight(7, "w", 16, 128)
    with pytest.raises(ValueError):
        oracle_lib.dq_gemm(7, wq.codes, wq.scales, wq.zeros, synth.normal_bf16(7, "x", (1, 128)))
