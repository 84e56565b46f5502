"""Seeded synthetic inputs for the decode hot path.

This module only draws random numbers in the shapes and distributions of the
workloads; it holds none of the method's arithmetic (no dequantisation, no
quantiser, no attention). Both the CPU oracle and the CUDA path consume the
same bytes it produces.

Each tensor gets its own stream: ``numpy.random.default_rng`` seeded with
``(seed, crc32(name))``. Large tensors requested on a CUDA device are drawn by
torch's device generator instead (seeded the same way), because drawing
gigabytes on the host would dominate a benchmark run; tests that need the
oracle on such tensors copy the device bytes back to the host.
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass

import numpy as np

try:  # torch is only needed to build device tensors and bf16 bit patterns
    import torch
except ImportError:  # pragma: no cover
    torch = None

# Element count above which device tensors are drawn on the device.
DEVICE_DRAW_THRESHOLD = 1 << 24


def _seed_words(seed: int, name: str) -> list[int]:
    return [int(seed) & 0xFFFFFFFF, zlib.crc32(name.encode())]


def rng(seed: int, name: str) -> np.random.Generator:
    return np.random.default_rng(_seed_words(seed, name))


def _torch_gen(seed: int, name: str, device):
    g = torch.Generator(device=device)
    w = _seed_words(seed, name)
    g.manual_seed((w[0] << 32) | w[1])
    return g


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns via torch's round-to-nearest-even cast."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _is_cuda(device) -> bool:
    return device is not None and torch is not None and torch.device(device).type == "cuda"


def _out(bits: np.ndarray, device):
    """numpy array, or a torch tensor on ``device`` holding the same bytes."""
    if device is None:
        return bits
    t = torch.from_numpy(bits)
    if bits.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.to(device)


def normal_bf16(seed: int, name: str, shape, std: float = 1.0, device=None):
    """N(0, std^2) values rounded to bf16. numpy uint16 bit patterns when
    ``device`` is None, else a torch.bfloat16 tensor on ``device``."""
    shape = tuple(int(s) for s in shape)
    count = int(np.prod(shape)) if shape else 1
    if _is_cuda(device) and count >= DEVICE_DRAW_THRESHOLD:
        g = _torch_gen(seed, name, device)
        t = torch.empty(shape, dtype=torch.float32, device=device)
        t.normal_(0.0, std, generator=g)
        return t.to(torch.bfloat16)
    a = rng(seed, name).standard_normal(shape, dtype=np.float32) * np.float32(std)
    return _out(f32_to_bf16_bits(a), device)


def uniform_u8(seed: int, name: str, shape, lo: int, hi: int, device=None):
    """Integers uniform on [lo, hi] as uint8."""
    shape = tuple(int(s) for s in shape)
    count = int(np.prod(shape)) if shape else 1
    if _is_cuda(device) and count >= DEVICE_DRAW_THRESHOLD:
        g = _torch_gen(seed, name, device)
        return torch.randint(lo, hi + 1, shape, generator=g, device=device, dtype=torch.uint8)
    a = rng(seed, name).integers(lo, hi + 1, size=shape, dtype=np.uint8)
    return _out(a, device)


def uniform_bf16(seed: int, name: str, shape, lo: float, hi: float, device=None):
    """Values uniform on [lo, hi) rounded to bf16."""
    shape = tuple(int(s) for s in shape)
    a = rng(seed, name).uniform(lo, hi, size=shape).astype(np.float32)
    return _out(f32_to_bf16_bits(a), device)


# ------------------------------------------------------------- weights ----

@dataclass
class Int4Weight:
    """Logical INT4 g128 weight: codes [n,k] 0..15, bf16 scales [n,k/128],
    zero points [n,k/128] 0..15."""
    codes: object
    scales: object
    zeros: object
    n: int
    k: int


def int4_weight(seed: int, name: str, n: int, k: int, device=None) -> Int4Weight:
    """Asymmetric INT4 g128: codes and zero points uniform on 0..15, scales
    uniform on [0.005, 0.02)."""
    assert k % 128 == 0
    return Int4Weight(
        codes=uniform_u8(seed, name + ".codes", (n, k), 0, 15, device),
        scales=uniform_bf16(seed, name + ".scales", (n, k // 128), 0.005, 0.02, device),
        zeros=uniform_u8(seed, name + ".zeros", (n, k // 128), 0, 15, device),
        n=n, k=k)


def bf16_weight(seed: int, name: str, n: int, k: int, std: float = 0.02,
                outlier_channels: int = 0, outlier_gain: float = 20.0, device=None):
    """W [n,k] ~ N(0, std^2) in bf16; optionally ``outlier_channels`` input
    channels (columns, drawn without replacement) scaled by ``outlier_gain``."""
    w = normal_bf16(seed, name, (n, k), std, device=None if outlier_channels else device)
    if not outlier_channels:
        return w
    cols = rng(seed, name + ".outliers").choice(k, outlier_channels, replace=False)
    vals = (w.astype(np.uint32) << 16).view(np.float32)
    vals[:, cols] *= np.float32(outlier_gain)
    return _out(f32_to_bf16_bits(vals), device)


def bf16_weight_outliers_device(seed: int, name: str, n: int, k: int, std: float,
                                outlier_channels: int, outlier_gain: float, device):
    """Device-drawn variant of :func:`bf16_weight` for large matrices."""
    w = normal_bf16(seed, name, (n, k), std, device)
    cols = rng(seed, name + ".outliers").choice(k, outlier_channels, replace=False)
    idx = torch.as_tensor(cols, device=device, dtype=torch.long)
    w[:, idx] = (w[:, idx].float() * outlier_gain).to(torch.bfloat16)
    return w


# ------------------------------------------------------------ KV cache ----

@dataclass
class PagedKV:
    """Paged KV cache: pools [num_blocks, Hkv, 16, D], block table
    [B, max_blocks] int32 (unused entries 0), context lengths [B] int32."""
    k_pool: object
    v_pool: object
    block_table: np.ndarray
    context_lens: np.ndarray
    num_blocks: int


def block_table(seed: int, name: str, context_lens, shuffle: bool = True,
                spare_blocks: int = 0):
    """Assign ceil(ctx/16) physical blocks to each sequence: a random
    permutation of the pool (``shuffle``) or consecutive blocks. Returns
    (table [B, max_blocks] int32, num_blocks)."""
    ctx = np.asarray(context_lens, dtype=np.int64)
    need = (ctx + 15) // 16
    total = int(need.sum()) + int(spare_blocks)
    ids = rng(seed, name).permutation(total) if shuffle else np.arange(total)
    maxb = int(need.max()) if need.size else 0
    table = np.zeros((ctx.size, max(maxb, 1)), np.int32)
    pos = 0
    for b, nb in enumerate(need):
        table[b, :nb] = ids[pos:pos + nb]
        pos += nb
    return table, total


def paged_kv(seed: int, name: str, context_lens, hkv: int, d: int = 128,
             shuffle: bool = True, spare_blocks: int = 0, device=None) -> PagedKV:
    """K and V ~ N(0,1) bf16 in a paged pool addressed by a block table."""
    table, nblk = block_table(seed, name + ".table", context_lens, shuffle, spare_blocks)
    shape = (nblk, hkv, 16, d)
    return PagedKV(k_pool=normal_bf16(seed, name + ".k", shape, 1.0, device),
                   v_pool=normal_bf16(seed, name + ".v", shape, 1.0, device),
                   block_table=table,
                   context_lens=np.asarray(context_lens, dtype=np.int32),
                   num_blocks=nblk)


def context_lengths(seed: int, name: str, batch: int, lo: int, hi: int) -> np.ndarray:
    """Per-sequence context lengths uniform on [lo, hi]."""
    return rng(seed, name).integers(lo, hi + 1, size=batch).astype(np.int32)


def e4m3_codes(seed: int, name: str, shape, exp_lo: int = 0, exp_hi: int = 15, device=None):
    """FP8-E4M3 code bytes s.eeee.mmm drawn in code space: sign and 3-bit
    mantissa uniform, exponent field uniform on [exp_lo, exp_hi]. The NaN
    codes (0x7F, 0xFF) are replaced by the largest finite code of the same
    sign (0x7E, 0xFE)."""
    shape = tuple(int(s) for s in shape)
    count = int(np.prod(shape)) if shape else 1
    if _is_cuda(device) and count >= DEVICE_DRAW_THRESHOLD:
        g = _torch_gen(seed, name, device)
        sign = torch.randint(0, 2, shape, generator=g, device=device, dtype=torch.uint8)
        expo = torch.randint(exp_lo, exp_hi + 1, shape, generator=g, device=device, dtype=torch.uint8)
        mant = torch.randint(0, 8, shape, generator=g, device=device, dtype=torch.uint8)
        c = (sign << 7) | (expo << 3) | mant
        return torch.where((c & 0x7F) == 0x7F, c - 1, c)
    r = rng(seed, name)
    sign = r.integers(0, 2, size=shape, dtype=np.uint8)
    expo = r.integers(exp_lo, exp_hi + 1, size=shape, dtype=np.uint8)
    mant = r.integers(0, 8, size=shape, dtype=np.uint8)
    c = (sign << 7) | (expo << 3) | mant
    c[(c & 0x7F) == 0x7F] -= 1
    return _out(c, device)


@dataclass
class PagedKVFp8:
    """Paged FP8-E4M3 KV cache: code pools [num_blocks, Hkv, 16, D] uint8 plus
    the block table and context lengths of :class:`PagedKV`."""
    k_codes: object
    v_codes: object
    block_table: np.ndarray
    context_lens: np.ndarray
    num_blocks: int


def paged_kv_fp8(seed: int, name: str, context_lens, hkv: int, d: int = 128,
                 shuffle: bool = True, spare_blocks: int = 0, exp_lo: int = 0,
                 exp_hi: int = 15, device=None) -> PagedKVFp8:
    """K and V code pools from :func:`e4m3_codes` behind a block table. With
    the default exponent range the codes cover every finite E4M3 value,
    subnormals and both zeros included."""
    table, nblk = block_table(seed, name + ".table", context_lens, shuffle, spare_blocks)
    shape = (nblk, hkv, 16, d)
    return PagedKVFp8(k_codes=e4m3_codes(seed, name + ".k", shape, exp_lo, exp_hi, device),
                      v_codes=e4m3_codes(seed, name + ".v", shape, exp_lo, exp_hi, device),
                      block_table=table,
                      context_lens=np.asarray(context_lens, dtype=np.int32),
                      num_blocks=nblk)
