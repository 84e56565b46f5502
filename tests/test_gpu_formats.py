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
