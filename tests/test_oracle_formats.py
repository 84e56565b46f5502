"""Pins for the oracle's weight formats: the FP8 row-wise quantiser, INT4 g128
dequantisation and the packed INT4 layout."""
import json
import os

import numpy as np
import pytest
import torch

from memory_bound_decode_dq_gb300 import synth

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")))


def _bits_to_f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ FP8 ----

def test_fp8_equal_magnitude_row_maps_to_448(oracle_lib):
    w = np.array([[0.75, -0.75, 0.75, -0.75] * 4], np.float32)
    codes, scales = oracle_lib.quant_fp8_rowwise(synth.f32_to_bf16_bits(w))
    assert scales[0] == np.float32(0.75) / np.float32(448.0)
    assert np.array_equal(codes[0], np.array([0x7E, 0xFE] * 8, np.uint8))


def test_fp8_zero_row_takes_unit_scale(oracle_lib):
    w = np.zeros((2, 32), np.uint16)
    w[1, 3] = 0x8000  # -0.0
    codes, scales = oracle_lib.quant_fp8_rowwise(w)
    assert np.all(scales == 1.0)
    assert np.all(codes[0] == 0) and codes[1, 3] == 0x80 and codes[1].sum() == 0x80


def test_fp8_matches_torch_cast(oracle_lib):
    """A second, independent quantiser built from torch's fp32 division and its
    float8_e4m3fn cast (RNE) gives the same codes and scales bit for bit."""
    w = synth.bf16_weight(2, "fp8pin", 96, 512, std=0.02, outlier_channels=6)
    codes, scales = oracle_lib.quant_fp8_rowwise(w)
    wf = torch.from_numpy(_bits_to_f32(w))
    amax = wf.abs().amax(dim=1)
    sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    ref = (wf / sc[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(scales, sc.numpy())
    assert np.array_equal(codes, ref)


def test_fp8_row_max_hits_448_and_error_within_half_step(oracle_lib):
    w = synth.bf16_weight(3, "fp8err", 64, 1024, std=0.02, outlier_channels=6)
    codes, scales = oracle_lib.quant_fp8_rowwise(w)
    wf = _bits_to_f32(w).astype(np.float64)
    val = oracle_lib.e4m3_decode(codes)
    amax_idx = np.abs(wf).argmax(axis=1)
    assert np.all(np.abs(val[np.arange(64), amax_idx]) == 448.0)
    v = wf / scales[:, None].astype(np.float64)          # exact quotient
    # E4M3 spacing at |v|: 2^(floor(log2|v|) - 3) for normals, 2^-9 below 2^-6
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -6)))
    half_step = 0.5 * 2.0 ** (e - 3)
    slack = np.abs(v) * 2.0 ** -23                      # the fp32 division's rounding
    assert np.all(np.abs(val - v) <= half_step + slack)


def test_fp8_tiny_row_uses_subnormal_scale(oracle_lib):
    w = np.zeros((1, 16), np.uint16)
    w[0, :4] = [0x0001, 0x8002, 0x0003, 0x0000]          # bf16 subnormals
    codes, scales = oracle_lib.quant_fp8_rowwise(w)
    assert scales[0] == np.float32(3 * 2.0 ** -133) / np.float32(448.0)
    assert codes[0, 2] == 0x7E


# ----------------------------------------------------------------- INT4 ----

def test_int4_dequant_matches_torch_rounding(oracle_lib):
    wq = synth.int4_weight(0, "deqpin", 40, 256)
    deq = oracle_lib.int4_dequant(wq.codes, wq.scales, wq.zeros)
    s = np.repeat(_bits_to_f32(wq.scales), 128, axis=1)
    z = np.repeat(wq.zeros, 128, axis=1).astype(np.float32)
    prod = (wq.codes.astype(np.float32) - z) * s         # exact in fp32
    ref = torch.from_numpy(prod).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(deq, ref)


def test_int4_dequant_special_cases(oracle_lib):
    n, k = 16, 256
    codes = np.random.default_rng(1).integers(0, 16, (n, k)).astype(np.uint8)
    zeros = np.zeros((n, k // 128), np.uint8)
    # scale 2^-5: exact, deq = q / 32
    scales = np.full((n, k // 128), 0x3D00, np.uint16)
    deq = oracle_lib.int4_dequant(codes, scales, zeros)
    assert np.array_equal(_bits_to_f32(deq), codes.astype(np.float32) / 32)
    # zero point equal to every code in its group -> exactly zero
    codes2 = np.repeat(np.arange(n * 2, dtype=np.uint8).reshape(n, 2) % 16, 128, axis=1)
    zeros2 = codes2[:, ::128].copy()
    deq2 = oracle_lib.int4_dequant(codes2, np.full((n, 2), 0x3C23, np.uint16), zeros2)
    assert np.all(_bits_to_f32(deq2) == 0.0)
    # q = 15, z = 0 and q = 0, z = 15 are negatives of each other
    a = oracle_lib.int4_dequant(np.full((1, 128), 15, np.uint8), np.full((1, 1), 0x3C23, np.uint16),
                                np.zeros((1, 1), np.uint8))
    b = oracle_lib.int4_dequant(np.zeros((1, 128), np.uint8), np.full((1, 1), 0x3C23, np.uint16),
                                np.full((1, 1), 15, np.uint8))
    assert np.all(_bits_to_f32(a) == -_bits_to_f32(b))


def test_int4_storage_matches_pages_bit_counts(oracle_lib):
    n = k = 4096
    nb, ns, nz = oracle_lib.int4_packed_sizes(n, k)
    bits = 8.0 * (nb + ns + nz) / (n * k)
    g = GOLDEN["int4_g128_bits"]
    # codes + bf16 scale per group alone: the pages' 4.125 bits
    assert 8.0 * (nb + ns) / (n * k) == g["scale_only"]
    # with the 4-bit zero point: 4.15625, the pages' "about 4.15"
    assert bits == 4.0 + 16 / 128 + 4 / 128
    assert abs(bits - g["gptq_estimate"]) < 0.01
    mb = GOLDEN["int4_4096_matrix_mb"]
    assert abs((nb + ns) / 1e6 - mb["value"]) < 0.01
    assert abs(2 * n * k / 1e6 - mb["bf16_mb"]) < 0.06


@pytest.mark.parametrize("n,k", [(16, 128), (1, 128), (15, 256), (17, 128), (40, 384), (64, 1024)])
def test_int4_pack_unpack_round_trip(oracle_lib, n, k):
    wq = synth.int4_weight(n * 1000 + k, "pack", n, k)
    pk, ps, pz = oracle_lib.int4_pack(wq.codes, wq.scales, wq.zeros)
    codes, scales, zeros, bad = oracle_lib.int4_unpack(pk, ps, pz, n, k)
    assert bad == 0
    assert np.array_equal(codes, wq.codes)
    assert np.array_equal(scales, wq.scales)
    assert np.array_equal(zeros, wq.zeros)


def test_int4_pack_is_a_permutation(oracle_lib):
    """Every (row, column) lands in exactly one nibble: pack a matrix whose
    codes are all zero but one, for every position of a 16x128 tile."""
    n, k = 16, 128
    scales = np.zeros((n, 1), np.uint16)
    zeros = np.zeros((n, 1), np.uint8)
    seen = set()
    for r in range(n):
        for c in range(k):
            codes = np.zeros((n, k), np.uint8)
            codes[r, c] = 15
            pk, _, _ = oracle_lib.int4_pack(codes, scales, zeros)
            words = pk.view(np.uint32)
            nz = np.flatnonzero(words)
            assert nz.size == 1
            word = int(nz[0])
            nib = int(words[word]).bit_length() // 4 - 1
            assert int(words[word]) == 15 << (4 * nib)
            seen.add((word, nib))
    assert len(seen) == n * k


def test_int4_pack_hand_checked_tile(oracle_lib):
    """16x128 tile with code(r, c) = (3r + c) mod 16, scale bits 0x3C80 + r and
    zero point r. The expected words are worked out by hand from the packed
    layout description (word w = 128h + 4l + j, nibble v -> row r0 + 8(v&1),
    column 32c + 8t + 4e + 2((v>>1)&1) + (v>>2)):
      word   0: h0 l0 j0 -> rows 0/8, columns 0..3   -> 0xB391A280
      word   5: h0 l1 j1 -> rows 0/8, columns 12..15 -> 0x7F5D6E4C
      word 255: h1 l31 j3 -> rows 7/15, columns 124..127 -> 0xC4A2B391
    scale word 3 = rows 3 and 11 -> 0x3C8B3C83; zero byte 5 = rows 5 and 13 -> 0xD5."""
    n, k = 16, 128
    r = np.arange(n)[:, None]
    c = np.arange(k)[None, :]
    codes = ((3 * r + c) % 16).astype(np.uint8)
    scales = (0x3C80 + np.arange(n, dtype=np.uint16))[:, None]
    zeros = np.arange(n, dtype=np.uint8)[:, None]
    pk, ps, pz = oracle_lib.int4_pack(codes, scales, zeros)
    words = pk.view(np.uint32)
    assert words[0] == 0xB391A280
    assert words[5] == 0x7F5D6E4C
    assert words[255] == 0xC4A2B391
    assert ps.view(np.uint32)[3] == 0x3C8B3C83
    assert pz[5] == 0xD5
