"""The synthetic decode workloads: shapes, distributions and seeds.

Each workload is named by what it is. Weight matrices are W [n out, k in].
Projections of a Llama-3-8B-shaped layer (hidden 4096, 32 q / 8 KV heads,
FFN 14336) and of the 80-layer 70B fixture (hidden 8192, 64 q / 8 KV heads,
FFN 28672); gate and up are fused into one [2*FFN, hidden] matrix.
"""
from __future__ import annotations

from dataclasses import dataclass, field

W_BF16, W_FP8_E4M3, W_INT4_G128 = 0, 1, 2
WTYPE_NAMES = {W_BF16: "bf16", W_FP8_E4M3: "fp8_e4m3", W_INT4_G128: "int4_g128"}

LLAMA3_8B_PROJ = (("qkv", 6144, 4096), ("o", 4096, 4096), ("gate_up", 28672, 4096),
                  ("down", 4096, 14336))
DENSE70B_PROJ = (("qkv", 10240, 8192), ("o", 8192, 8192), ("gate_up", 57344, 8192),
                 ("down", 8192, 28672))


@dataclass(frozen=True)
class GemmCase:
    name: str
    wtype: int
    m: int
    n: int
    k: int
    outliers: int = 0   # input channels scaled x20 (BF16/FP8 weights)


@dataclass(frozen=True)
class AttnCase:
    name: str
    batch: int
    width: int          # verify width W (1 = plain decode)
    hq: int
    hkv: int
    context: tuple      # per-sequence context lengths (include the W new tokens)
    shuffle: bool = True
    d: int = 128
    kv_fp8: bool = False  # FP8-E4M3 cache codes instead of bf16
    k_scale: float = 1.0  # FP8 cache: cached K = code * k_scale
    v_scale: float = 1.0  # FP8 cache: cached V = code * v_scale


@dataclass(frozen=True)
class VerifyCase:
    """Greedy verify of a draft block: target logits [batch, width, vocab] bf16."""
    name: str
    batch: int
    width: int
    vocab: int


@dataclass(frozen=True)
class RopeCase:
    """Rotary embedding of the new tokens' q, k and the append of k, v:
    qkv rows [batch * width, (hq + 2 hkv) * 128] bf16, bf16 paged cache."""
    name: str
    batch: int
    width: int
    hq: int
    hkv: int
    context: tuple
    rope_base: float = 500000.0
    d: int = 128


@dataclass(frozen=True)
class QkvRopeCase:
    """The QKV projection of the new tokens fused with RoPE and the KV append
    (dq_gemm_qkv_rope_append): x [batch * width, k], W [(hq + 2 hkv) * 128, k],
    bf16 paged cache."""
    name: str
    wtype: int
    batch: int
    width: int
    hq: int
    hkv: int
    k: int
    context: tuple
    rope_base: float = 500000.0
    d: int = 128


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    gemms: tuple = field(default_factory=tuple)
    attns: tuple = field(default_factory=tuple)
    verifies: tuple = field(default_factory=tuple)
    ropes: tuple = field(default_factory=tuple)
    qkv_ropes: tuple = field(default_factory=tuple)


def _ctx_uniform(seed: int, batch: int, lo: int, hi: int) -> tuple:
    from .synth import context_lengths
    return tuple(int(c) for c in context_lengths(seed, f"ctx.b{batch}", batch, lo, hi))


def tiny() -> Workload:
    """One INT4 g128 1024x1024 GEMV and one contiguous-KV decode attention
    (1 sequence, 8/2 heads, 256 cached tokens)."""
    return Workload("tiny_int4_1024_attn_ctx256", 0,
                    gemms=(GemmCase("proj_1024", W_INT4_G128, 1, 1024, 1024),),
                    attns=(AttnCase("attn_ctx256", 1, 1, 8, 2, (256,), shuffle=False),))


def llama3_8b_b1() -> Workload:
    """Llama-3-8B-shaped decode layer at batch 1: four projections in BF16 and
    INT4 g128, the BF16 QKV projection fused with the rotary embedding and KV
    append of the new token, attention 32/8 heads over 8192 paged tokens."""
    g = []
    for wt in (W_BF16, W_INT4_G128):
        for name, n, k in LLAMA3_8B_PROJ:
            if wt == W_BF16 and name == "qkv":
                continue  # fused with RoPE and the append below
            g.append(GemmCase(f"{name}_{WTYPE_NAMES[wt]}", wt, 1, n, k))
    return Workload("llama3_8b_decode_b1_ctx8192", 1, gemms=tuple(g),
                    attns=(AttnCase("attn_32_8_ctx8192", 1, 1, 32, 8, (8192,)),),
                    qkv_ropes=(QkvRopeCase("qkv_bf16_rope_append_32_8", W_BF16, 1, 1, 32, 8, 4096, (8192,)),))


def dense70b_b32() -> Workload:
    """70B-fixture decode layer at batch 32: projections in BF16 and FP8-E4M3
    (W ~ N(0, 0.02) with 6 outlier input channels x20), attention 64/8 heads
    over 2048 paged tokens per sequence."""
    g = []
    for wt in (W_BF16, W_FP8_E4M3):
        for name, n, k in DENSE70B_PROJ:
            g.append(GemmCase(f"{name}_{WTYPE_NAMES[wt]}", wt, 32, n, k, outliers=6))
    return Workload("dense70b_decode_b32_ctx2048", 2, gemms=tuple(g),
                    attns=(AttnCase("attn_64_8_b32_ctx2048", 32, 1, 64, 8, (2048,) * 32),))


LLAMA3_8B_VOCAB = 128256


def verify_8b() -> Workload:
    """Speculative verify on the 8B shapes: INT4 g128 projections at
    M = batch x (drafts + 1) for drafts in {5, 15} and batch in {1, 64},
    verify attention of width drafts + 1 over contexts uniform on [512, 4096],
    and the greedy accept step over the target's logits (vocabulary 128256)."""
    g, a, v = [], [], []
    for batch in (1, 64):
        for width in (6, 16):
            m = batch * width
            for name, n, k in LLAMA3_8B_PROJ:
                if name == "qkv" and batch == 64 and width == 16:
                    continue  # fused with RoPE and the append below
                g.append(GemmCase(f"{name}_int4_m{m}", W_INT4_G128, m, n, k))
            a.append(AttnCase(f"attn_verify_b{batch}_w{width}", batch, width, 32, 8,
                              _ctx_uniform(3, batch, 512, 4096)))
            v.append(VerifyCase(f"accept_greedy_b{batch}_w{width}", batch, width, LLAMA3_8B_VOCAB))
    r = (QkvRopeCase("qkv_int4_m1024_rope_append_b64_w16", W_INT4_G128, 64, 16, 32, 8, 4096,
                     _ctx_uniform(3, 64, 512, 4096)),)
    return Workload("verify_8b_int4", 3, gemms=tuple(g), attns=tuple(a), verifies=tuple(v), qkv_ropes=r)


def longctx_70b_b8() -> Workload:
    """Long-context step: 70B-fixture attention, 8 sequences x 131072 paged
    tokens (4 GiB of KV), plus the 70B projections at M = 8 in FP8 and INT4."""
    g = []
    for wt in (W_FP8_E4M3, W_INT4_G128):
        for name, n, k in DENSE70B_PROJ:
            g.append(GemmCase(f"{name}_{WTYPE_NAMES[wt]}", wt, 8, n, k,
                              outliers=6 if wt == W_FP8_E4M3 else 0))
    return Workload("longctx_70b_b8_ctx131072", 4, gemms=tuple(g),
                    attns=(AttnCase("attn_64_8_b8_ctx131072", 8, 1, 64, 8, (131072,) * 8),))


def longctx_70b_b1() -> Workload:
    """The long-context attention at one sequence (512 MiB of KV): the size
    used for Nsight Compute captures of the long-context kernel."""
    return Workload("longctx_70b_b1_ctx131072", 5,
                    attns=(AttnCase("attn_64_8_b1_ctx131072", 1, 1, 64, 8, (131072,)),))


# FP8 cache scales of the FP8-KV workloads: codes span +-448, so K = code/64
# and V = code/128 keep the cached values within a few units.
FP8_K_SCALE, FP8_V_SCALE = 1.0 / 64, 1.0 / 128


def int4_70b_b32_fp8kv() -> Workload:
    """70B-fixture decode layer at batch 32 with INT4 g128 projections and an
    FP8-E4M3 KV cache: attention 64/8 heads over 2048 paged tokens per
    sequence, codes drawn over every finite E4M3 value."""
    g = tuple(GemmCase(f"{name}_int4_g128", W_INT4_G128, 32, n, k) for name, n, k in DENSE70B_PROJ)
    return Workload("int4_70b_b32_fp8kv_ctx2048", 6, gemms=g,
                    attns=(AttnCase("attn_fp8kv_64_8_b32_ctx2048", 32, 1, 64, 8, (2048,) * 32,
                                    kv_fp8=True, k_scale=FP8_K_SCALE, v_scale=FP8_V_SCALE),))


def longctx_70b_b8_fp8kv() -> Workload:
    """The long-context attention of longctx_70b_b8 over an FP8-E4M3 cache:
    8 sequences x 131072 paged tokens, 64/8 heads (2 GiB of KV codes)."""
    return Workload("longctx_70b_b8_fp8kv_ctx131072", 7,
                    attns=(AttnCase("attn_fp8kv_64_8_b8_ctx131072", 8, 1, 64, 8, (131072,) * 8,
                                    kv_fp8=True, k_scale=FP8_K_SCALE, v_scale=FP8_V_SCALE),))


ALL = (tiny, llama3_8b_b1, dense70b_b32, verify_8b, longctx_70b_b8, longctx_70b_b1,
       int4_70b_b32_fp8kv, longctx_70b_b8_fp8kv)
