"""GPU parity of the offline weight preparation: quant_fp8_rowwise and
pack_int4_g128 must match the oracle bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_decode_dq_gb300 import synth
from gpu_util import bf, bits, require_cuda, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_cuda()


@pytest.fixture(scope="module")
def dqd():
    from memory_bound_decode_dq_gb300 import dqd as m
    return m


@pytest.mark.parametrize("n,k,outliers", [(96, 512, 6), (33, 1024, 0), (1, 16, 0), (257, 4096, 6)])
def test_quant_fp8_bit_exact(dev, dqd, n, k, outliers):
    w = synth.bf16_weight(n + k, "q8", n, k, std=0.02, outlier_channels=outliers)
    codes, scales = dqd.quant_fp8_rowwise(bf(w, dev))
    rc, rs = oracle.quant_fp8_rowwise(w)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_quant_fp8_special_rows(dev, dqd):
    k = 64
    rows = [
        np.zeros(k, np.float32),                                  # all zero -> scale 1
        np.array([0.75, -0.75] * (k // 2), np.float32),           # equal magnitude -> +-448
        np.linspace(-1, 1, k).astype(np.float32),
        np.full(k, -1e-38, np.float32),                           # tiny
    ]
    w = synth.f32_to_bf16_bits(np.stack(rows))
    w[0, 5] = 0x8000                                              # -0.0 keeps its sign
    w[3, :8] = [0x0001, 0x8002, 0x0003, 0, 0x8000, 0x0010, 0x0007, 0x8001]   # subnormals
    codes, scales = dqd.quant_fp8_rowwise(bf(w, dev))
    rc, rs = oracle.quant_fp8_rowwise(w)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


@pytest.mark.parametrize("n,k", [(16, 128), (17, 256), (40, 384), (1, 128), (1024, 1024), (4100, 2048)])
def test_pack_int4_bit_exact(dev, dqd, n, k):
    wq = synth.int4_weight(n * 7 + k, "pk", n, k)
    p = dqd.pack_int4_g128(u8(wq.codes, dev), bf(wq.scales, dev), u8(wq.zeros, dev))
    pk, ps, pz = oracle.int4_pack(wq.codes, wq.scales, wq.zeros)
    assert np.array_equal(p.packed.cpu().numpy(), pk)
    assert np.array_equal(p.scales.cpu().numpy(), ps)
    assert np.array_equal(p.zeros.cpu().numpy(), pz)
    codes, scales, zeros, bad = oracle.int4_unpack(p.packed.cpu().numpy(), p.scales.cpu().numpy(),
                                                   p.zeros.cpu().numpy(), n, k)
    assert bad == 0
    assert np.array_equal(codes, wq.codes)
    assert np.array_equal(scales, wq.scales)
    assert np.array_equal(zeros, wq.zeros)


def test_pack_rejects_bad_shapes(dev, dqd):
    with pytest.raises(ValueError):
        dqd.pack_int4_g128(torch.zeros((16, 100), dtype=torch.uint8, device=dev),
                           torch.zeros((16, 1), dtype=torch.bfloat16, device=dev),
                           torch.zeros((16, 1), dtype=torch.uint8, device=dev))


def _int4_cases():
    rng = np.random.default_rng(11)
    w = rng.standard_normal((48, 1024)).astype(np.float32) * 0.02
    w[3, :128] = 0.0                                   # all-zero group
    w[4, 128:256] = 0.37                               # constant positive group
    w[5, 256:384] = -0.37                              # constant negative group
    w[6, :] = np.abs(w[6, :])                          # all-positive row
    w[7, :] = -np.abs(w[7, :])                         # all-negative row
    w[8, 384:512] = rng.standard_normal(128).astype(np.float32) * 1e-39   # bf16 subnormals
    w[9, 512:640] *= 1e4                               # wide range
    w[10, 700] = 3.0                                   # one outlier
    w[11, 0:128] = np.linspace(-1, 1, 128)             # many exact ties
    return synth.f32_to_bf16_bits(w)


@pytest.mark.parametrize("n,k,kind", [(48, 1024, "special"), (96, 4096, "normal"), (1, 128, "normal"),
                                      (257, 2048, "outliers")])
def test_quant_int4_bit_exact(dev, dqd, n, k, kind):
    if kind == "special":
        w = _int4_cases()
    else:
        w = synth.bf16_weight(n + k, "q4", n, k, std=0.02, outlier_channels=6 if kind == "outliers" else 0)
    codes, scales, zeros = dqd.quant_int4_g128(bf(w, dev))
    rc, rs, rz = oracle.int4_quant(w)
    assert np.array_equal(bits(scales), rs)
    assert np.array_equal(zeros.cpu().numpy(), rz)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_quant_int4_then_gemm(dev, dqd):
    """bf16 W -> quant_int4_g128 -> pack_int4_g128 -> dq_gemm agrees with the
    oracle's GEMM on the oracle's own quantisation of W."""
    n, k = 200, 2048
    w = synth.bf16_weight(5, "q4g", n, k, std=0.02, outlier_channels=4)
    codes, scales, zeros = dqd.quant_int4_g128(bf(w, dev))
    weight = dqd.Weight.int4(dqd.pack_int4_g128(codes, scales, zeros))
    x = synth.normal_bf16(5, "x", (3, k))
    from gpu_util import assert_close, f64
    y = dqd.dq_gemm(weight, bf(x, dev))
    rc, rs, rz = oracle.int4_quant(w)
    assert_close(f64(y), oracle.dq_gemm(oracle.W_INT4_G128, rc, rs, rz, x), what="quantise -> pack -> gemm")


def test_quant_int4_rejects_bad_shapes(dev, dqd):
    with pytest.raises(dqd.DqdError):
        dqd.quant_int4_g128(bf(np.zeros((4, 100), np.uint16), dev))
