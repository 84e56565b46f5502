"""Byte accounting and the bandwidth bound model of a decode step.

Host-side arithmetic only (no kernels): the benchmark uses it to turn a
measured time into effective HBM bandwidth and a roofline fraction, and the
tests pin it to the figures the pages print.

Sources:
  "降低每個 Token 的生成成本" (Making each token cheaper), optiverse-tech.com:
    section "為何 Decode 通常受記憶體頻寬限制" (why decode is bandwidth-bound):
    memory_time = (weight bytes + batch x KV bytes per sequence) / bandwidth,
    compute_time = 2 x parameters x positions / peak, step >= max of the two;
    section "建立單一 Token 成本計算器" (the token_cost calculator) and its
    printed expected values.
  "LLM 推理是怎么变快的", §2.2: KV bytes = 2 x layers x kv_heads x head_dim
    x seq_len x dtype bytes x batch.
"""
from __future__ import annotations

import math

W_BF16, W_FP8_E4M3, W_INT4_G128 = 0, 1, 2


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, dtype_bytes: int = 2) -> int:
    """2 (K and V) x layers x kv_heads x head_dim x dtype bytes."""
    return 2 * layers * kv_heads * head_dim * dtype_bytes


def kv_bytes(layers: int, kv_heads: int, head_dim: int, seq_len: int, dtype_bytes: int = 2,
             batch: int = 1) -> int:
    return kv_bytes_per_token(layers, kv_heads, head_dim, dtype_bytes) * seq_len * batch


# ------------------------------------------------- algorithmic bytes/call ----

def weight_bytes(wtype: int, n: int, k: int) -> float:
    """Bytes the method must read once for W [n out, k in] with its metadata:
    BF16 2nk; FP8 nk + 4n (fp32 row scales); INT4 g128 nk/2 + 2.5 nk/128
    (bf16 scale and 4-bit zero point per 128-weight group)."""
    if wtype == W_BF16:
        return 2.0 * n * k
    if wtype == W_FP8_E4M3:
        return 1.0 * n * k + 4.0 * n
    if wtype == W_INT4_G128:
        return 0.5 * n * k + 2.5 * n * k / 128.0
    raise ValueError(wtype)


def dq_gemm_bytes(wtype: int, m: int, n: int, k: int) -> float:
    """Weights + activations x [m,k] bf16 + output y [m,n] bf16."""
    return weight_bytes(wtype, n, k) + 2.0 * m * k + 2.0 * m * n


def dq_gemm_flops(m: int, n: int, k: int) -> float:
    return 2.0 * m * n * k


def attn_bytes(context_lens, w: int, hq: int, hkv: int, d: int = 128, block: int = 16,
               kv_bytes_per_element: int = 2) -> float:
    """K and V of every cached token of every sequence (2 bytes per element in
    bf16, 1 in FP8), plus q and out (bf16), plus the block-table entries the
    call reads."""
    ctx = [int(c) for c in context_lens]
    b = len(ctx)
    kv = sum(ctx) * hkv * d * 2 * kv_bytes_per_element
    qo = 2 * (2 * b * w * hq * d)
    table = 4 * sum(math.ceil(c / block) for c in ctx)
    return float(kv + qo + table)


def rope_append_bytes(tokens: int, hq: int, hkv: int, d: int = 128, kv_bytes_per_element: int = 2) -> float:
    """RoPE + KV append: read each new token's qkv row (bf16), write its
    rotated q (bf16) and its k and v into the cache, plus the token's
    context length and block-table entry."""
    return float(tokens * ((hq + 2 * hkv) * d * 2 + hq * d * 2 + 2 * hkv * d * kv_bytes_per_element + 8))


def qkv_rope_append_bytes(wtype: int, tokens: int, k: int, hq: int, hkv: int, d: int = 128,
                          kv_bytes_per_element: int = 2) -> float:
    """The QKV projection fused with RoPE + KV append: the projection's
    weights and activations, then per token its rotated q (bf16), its k and v
    written into the cache, its context length and its block-table entry (the
    qkv row itself never reaches memory)."""
    n = (hq + 2 * hkv) * d
    return float(weight_bytes(wtype, n, k) + 2.0 * tokens * k +
                 tokens * (hq * d * 2 + 2 * hkv * d * kv_bytes_per_element + 8))


def verify_bytes(batch: int, width: int, vocab: int) -> float:
    """Greedy verify: the target's bf16 logits, the drafts, the predictions,
    the counts and the context lengths (read and written)."""
    return float(2 * batch * width * vocab + 4 * batch * (width - 1) + 4 * batch * width + 12 * batch)


def attn_flops(context_lens, w: int, hq: int, d: int = 128) -> float:
    """QK^T and PV over the visible keys (causal inside the verify block)."""
    total = 0
    for c in context_lens:
        for i in range(w):
            total += c - w + i + 1
    return 4.0 * total * hq * d


# ------------------------------------------------- step bound model ----

def step_bound_seconds(weight_bytes_total: float, batch: int, positions: int,
                       kv_bytes_per_sequence: float, parameters: float,
                       bandwidth: float, peak_flops: float) -> float:
    """Lower bound of one target forward: the larger of the time to stream
    weights plus every sequence's KV once and the time of 2 FLOPs per
    parameter per scored position."""
    stream = (weight_bytes_total + batch * kv_bytes_per_sequence) / bandwidth
    math_time = 2.0 * parameters * batch * positions / peak_flops
    return max(stream, math_time)


def expected_tokens_per_round(alpha: float, gamma: int) -> float:
    """Tokens a verify round yields when each of gamma drafts is accepted
    with probability alpha until the first rejection, plus the target's own
    token: 1 + alpha + ... + alpha^gamma."""
    return sum(alpha ** i for i in range(gamma + 1))


def fixture_70b_bounds(bits_per_weight: float, batch: int = 32, context: int = 2048,
                       gamma: int = 4, alpha: float = 0.8, draft_cost: float = 0.1,
                       bandwidth: float = 3.0e12, peak_flops: float = 1.0e15,
                       parameters: float = 70e9, kv_bytes_per_element: int = 2) -> dict:
    """Bound model of the 80-layer, 8-KV-head, head-dim-128 70B fixture on the
    pages' hypothetical 3.0 TB/s, 1,000 TFLOP/s device, for one weight
    format. Times in milliseconds."""
    kv_seq = kv_bytes(80, 8, 128, context, kv_bytes_per_element)
    wbytes = parameters * bits_per_weight / 8.0
    args = (kv_seq, parameters, bandwidth, peak_flops)
    plain = step_bound_seconds(wbytes, batch, 1, *args)
    verify = step_bound_seconds(wbytes, batch, gamma + 1, *args)
    tokens = expected_tokens_per_round(alpha, gamma)
    return {
        "weight_gb": wbytes / 1e9,
        "single_sequence_ms": 1e3 * wbytes / bandwidth,
        "batch_step_ms": 1e3 * plain,
        "verify_over_plain": verify / plain,
        "tokens_per_round": tokens,
        "speedup_free_verify": tokens / (1.0 + gamma * draft_cost),
        "speedup_at_batch": tokens / (verify / plain + gamma * draft_cost),
        "kv_bytes_per_sequence": kv_seq,
    }
