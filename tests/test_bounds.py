"""Pins for the host-side byte accounting and bound model against the figures
the pages print (tests/golden/pages_figures.json, each entry cited)."""
import json
import os

import pytest

from memory_bound_decode_dq_gb300 import bounds

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")))


@pytest.mark.parametrize("entry", G["kv_bytes_per_token"], ids=lambda e: e["model"])
def test_kv_bytes_per_token(entry):
    assert bounds.kv_bytes_per_token(entry["layers"], entry["kv_heads"], entry["head_dim"]) == entry["bytes"]


def test_kv_bytes_per_sequence():
    assert bounds.kv_bytes(80, 8, 128, 2048) == G["kv_bytes_per_sequence_2048"]["value"]
    # CS336 notes exercise 1(b): 128 KiB x 8192 x 32 ~ 34.4 GB
    assert abs(bounds.kv_bytes(32, 8, 128, 8192, batch=32) / 1e9 - 34.4) < 0.05


@pytest.mark.parametrize("fmt,bits", [("bf16", 16.0), ("fp8_e4m3", 8.0), ("int4_g128", 4.15)])
def test_fixture_bounds(fmt, bits):
    want = G["fixture_70b_bounds_ms"][fmt]
    got = bounds.fixture_70b_bounds(bits)
    assert got["weight_gb"] == pytest.approx(want["weight_gb"], abs=1e-9)
    assert got["single_sequence_ms"] == pytest.approx(want["batch1"], abs=5e-4)
    assert got["batch_step_ms"] == pytest.approx(want["batch32"], abs=5e-4)
    assert got["verify_over_plain"] == pytest.approx(want["verify_ratio"], abs=5e-5)


def test_speculation_figures():
    s = G["speculation"]
    bf = bounds.fixture_70b_bounds(16.0)
    i4 = bounds.fixture_70b_bounds(4.15)
    assert bf["tokens_per_round"] == pytest.approx(s["expected_tokens"], abs=5e-5)
    assert bf["speedup_free_verify"] == pytest.approx(s["speedup_free_verification"], abs=5e-5)
    assert i4["speedup_at_batch"] == pytest.approx(s["int4_speedup_at_batch"], abs=5e-5)


def test_fp8_kv_bound():
    got = bounds.fixture_70b_bounds(4.15, kv_bytes_per_element=1)["batch_step_ms"]
    assert got == pytest.approx(G["int4_b32_fp8_kv_ms"]["value"], abs=5e-4)


def test_algorithmic_bytes():
    # INT4 g128 with bf16 scale + 4-bit zero: 4.15625 bits per weight
    assert bounds.weight_bytes(bounds.W_INT4_G128, 4096, 4096) * 8 / 4096 ** 2 == 4.15625
    assert bounds.dq_gemm_bytes(bounds.W_BF16, 1, 4096, 4096) == 2 * 4096 * 4096 + 2 * 4096 + 2 * 4096
    assert bounds.dq_gemm_bytes(bounds.W_FP8_E4M3, 32, 10, 64) == 640 + 40 + 2 * 32 * 64 + 2 * 32 * 10
    # attention: 8192 tokens x 8 heads x 128 x 2 (K,V) x 2 B + q/out + table
    assert bounds.attn_bytes([8192], 1, 32, 8) == 8192 * 8 * 128 * 4 + 4 * 32 * 128 + 4 * 512
    assert bounds.attn_flops([10], 2, 1, 4) == 4.0 * (9 + 10) * 4


def test_algorithmic_bytes_of_the_next_rows():
    # FP8 cache: 8192 tokens x 8 heads x 128 x 2 (K, V) x 1 B, q and out in bf16, the table
    assert bounds.attn_bytes([8192], 1, 32, 8, kv_bytes_per_element=1) == 16_777_216 + 16_384 + 2_048
    # one new token, 32/8 heads: qkv row read (48 x 128 x 2), q written (32 x 128 x 2),
    # k and v appended (2 x 8 x 128 x 2 in bf16, x 1 in FP8), context length + table entry
    assert bounds.rope_append_bytes(1, 32, 8) == 12_288 + 8_192 + 4_096 + 8
    assert bounds.rope_append_bytes(1, 32, 8, kv_bytes_per_element=1) == 12_288 + 8_192 + 2_048 + 8
    # greedy verify, batch 64 x width 16 over 128256 logits: logits (bf16), drafts (64 x 15),
    # predictions (64 x 16), counts and context lengths read and written (64 x 12 B)
    assert bounds.verify_bytes(64, 16, 128256) == 262_668_288 + 3_840 + 4_096 + 768
