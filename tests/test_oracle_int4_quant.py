"""Pins for the oracle's asymmetric min/max INT4 quantiser.

Weights built on the grid, w = (q - z) s with both ends of 0..15 present and
a scale of at most 4 significant bits, come back as exactly (q, s, z); zero
stays exactly representable; every weight is reconstructed within a little
over half a step; and, as the granularity passage of the lecture notes says,
an outlier widens its own group's scale, so finer groups reconstruct a
matrix with outliers more accurately."""
import numpy as np
import pytest

from memory_bound_decode_dq_gb300 import synth


def _f(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _deq(codes, scales, zeros, group):
    s = np.repeat(_f(scales), group, axis=1)
    z = np.repeat(zeros.astype(np.float64), group, axis=1)
    return (codes.astype(np.float64) - z) * s


def test_weights_on_the_grid_are_recovered_exactly(oracle_lib):
    rng = np.random.default_rng(0)
    n, k = 24, 512
    G = k // 128
    # scales with 4 significant bits: (q - z) * s is exact in bf16
    mant = rng.integers(8, 16, (n, G))
    expo = rng.integers(-12, 2, (n, G))
    s = mant * np.exp2(expo - 3.0)
    z = rng.integers(0, 16, (n, G))
    q = rng.integers(0, 16, (n, k))
    q[:, ::128] = 0          # both ends of the grid in every group
    q[:, 1::128] = 15
    w = (q - np.repeat(z, 128, axis=1)) * np.repeat(s, 128, axis=1)
    wb = synth.f32_to_bf16_bits(w.astype(np.float32))
    assert np.array_equal(_f(wb), w)
    codes, scales, zeros = oracle_lib.int4_quant(wb)
    assert np.array_equal(_f(scales), s)
    assert np.array_equal(zeros, z)
    assert np.array_equal(codes, q)


def test_zero_is_exact_and_error_within_half_a_step(oracle_lib):
    w = synth.normal_bf16(1, "w", (64, 1024), std=0.02)
    w[:, 5] = 0
    codes, scales, zeros = oracle_lib.int4_quant(w)
    deq = _deq(codes, scales, zeros, 128)
    assert np.all(deq[:, 5] == 0)
    step = np.repeat(_f(scales), 128, axis=1)
    assert np.all(np.abs(deq - _f(w)) <= 0.55 * step)
    assert codes.max() <= 15 and zeros.max() <= 15


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_constant_and_zero_groups(oracle_lib, sign):
    w = np.zeros((2, 256), np.float32)
    w[0, :128] = sign * 3.0          # a constant group: 0 and c span the range
    wb = synth.f32_to_bf16_bits(w)
    codes, scales, zeros = oracle_lib.int4_quant(wb)
    deq = _deq(codes, scales, zeros, 128)
    assert np.abs(deq[0, :128] - sign * 3.0).max() <= 3.0 * 2.0 ** -8
    assert np.all(deq[0, 128:] == 0) and np.all(deq[1] == 0)
    assert scales[1, 0] == 0x3F80 and zeros[1, 0] == 0      # all-zero group: s = 1, z = 0


def test_finer_groups_contain_outliers(oracle_lib):
    """The granularity demo: a 512 x 512 matrix with 20 outliers. An outlier
    stretches its group's scale, so the other weights of that group lose
    resolution; smaller groups confine the damage."""
    rng = np.random.default_rng(3)
    w = rng.standard_normal((512, 512)).astype(np.float32)
    idx = rng.choice(512 * 512, 20, replace=False)
    w.reshape(-1)[idx] = rng.choice([-60.0, 60.0], 20)
    wb = synth.f32_to_bf16_bits(w)
    wf = _f(wb)
    err = {}
    for group in (512, 128, 32):
        deq = _deq(*oracle_lib.int4_quant(wb, group), group)
        err[group] = np.mean((deq - wf) ** 2)
    assert err[32] < err[128] < err[512]
    # inside g128, groups holding an outlier reconstruct their other weights worse
    codes, scales, zeros = oracle_lib.int4_quant(wb, 128)
    deq = _deq(codes, scales, zeros, 128)
    hit = np.zeros((512, 4), bool)
    for i in idx:
        hit[i // 512, (i % 512) // 128] = True
    e = ((deq - wf) ** 2).reshape(512, 4, 128)
    mask = np.ones(512 * 512, bool)
    mask[idx] = False
    mask = mask.reshape(512, 4, 128)
    per_group = np.array([[e[r, g][mask[r, g]].mean() for g in range(4)] for r in range(512)])
    assert per_group[hit].min() > 10 * np.median(per_group[~hit])
