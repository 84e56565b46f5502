"""CPU oracle for the memory-bound decode hot path (Python side).

TEST INFRASTRUCTURE ONLY: the tests, the package's ``smoke()`` check and the
benchmark's CPU-baseline leg may use this module; the product path (the CUDA
library and its binding) never does, and this module imports nothing from it.

The arithmetic lives in ``dqd_oracle.c`` (plain C, double precision, OpenMP
over independent output rows). This file compiles it with the host C compiler
when the shared object is missing or older than the source, and wraps each
routine for NumPy arrays. Array layouts follow the C routines' comments.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dqd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libdqd_oracle.so")
_lock = threading.Lock()
_lib = None

W_BF16, W_FP8_E4M3, W_INT4_G128 = 0, 1, 2

_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-Wall"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``libdqd_oracle.so`` next to its source."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cc = os.environ.get("CC", "gcc")
            subprocess.run([cc, *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.orc_bf16_to_double.restype = ctypes.c_double
        lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_round.restype = ctypes.c_uint16
        lib.orc_bf16_round.argtypes = [ctypes.c_double]
        lib.orc_e4m3_decode.restype = ctypes.c_double
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        for name in ("orc_e4m3_decode_n", "orc_e4m3_encode_n", "orc_bf16_round_n"):
            getattr(lib, name).restype = None
            getattr(lib, name).argtypes = [P, I64, P]
        lib.orc_quant_fp8_rowwise.restype = None
        lib.orc_quant_fp8_rowwise.argtypes = [P, I64, I64, P, P]
        lib.orc_int4_dequant.restype = None
        lib.orc_int4_dequant.argtypes = [P, P, P, I64, I64, P]
        lib.orc_int4_quant.restype = None
        lib.orc_int4_quant.argtypes = [P, I64, I64, I64, P, P, P]
        lib.orc_int4_pack.restype = None
        lib.orc_int4_pack.argtypes = [P, P, P, I64, I64, P, P, P]
        lib.orc_int4_unpack.restype = I64
        lib.orc_int4_unpack.argtypes = [P, P, P, I64, I64, P, P, P]
        lib.orc_dq_gemm.restype = ctypes.c_int
        lib.orc_dq_gemm.argtypes = [ctypes.c_int, P, P, P, I64, I64, P, I64, P, I64, P]
        lib.orc_gqa_decode_attn.restype = ctypes.c_int
        lib.orc_gqa_decode_attn.argtypes = [P, P, P, P, I64, P, I64, I64, I64, I64, I64,
                                            I64, ctypes.c_double, P, I64, P]
        lib.orc_gqa_decode_attn_fp8kv.restype = ctypes.c_int
        lib.orc_gqa_decode_attn_fp8kv.argtypes = [P, P, P, ctypes.c_double, ctypes.c_double, P,
                                                  I64, P, I64, I64, I64, I64, I64, I64,
                                                  ctypes.c_double, P, I64, P]
        lib.orc_spec_verify_greedy.restype = None
        lib.orc_spec_verify_greedy.argtypes = [P, I64, I64, I64, P, P, P, P]
        lib.orc_spec_verify_sample.restype = None
        lib.orc_spec_verify_sample.argtypes = [P, P, P, P, P, I64, I64, I64, P, P, P]
        lib.orc_rope.restype = None
        lib.orc_rope.argtypes = [P, I64, I64, P, ctypes.c_double]
        lib.orc_rope_kv_append.restype = ctypes.c_int
        lib.orc_rope_kv_append.argtypes = [P, I64, I64, I64, I64, I64, ctypes.c_double, P, P, I64, I64,
                                           P, P, P, P]
        lib.orc_num_threads.restype = ctypes.c_int
        lib.orc_num_threads.argtypes = []
        lib.orc_set_num_threads.restype = None
        lib.orc_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def _p(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def num_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(_L().orc_num_threads())


def set_num_threads(n: int) -> None:
    """Threads for the oracle's later parallel loops."""
    _L().orc_set_num_threads(int(n))


# ---------------------------------------------------------------- codecs ----

def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values."""
    b = _c(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_round(values) -> np.ndarray:
    """Round float64 values to bf16 (RNE); returns uint16 bit patterns."""
    v = _c(values, np.float64)
    out = np.empty(v.shape, np.uint16)
    _L().orc_bf16_round_n(_p(v), v.size, _p(out))
    return out


def e4m3_decode(codes) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _L().orc_e4m3_decode_n(_p(c), c.size, _p(out))
    return out


def e4m3_encode(values) -> np.ndarray:
    """float32 values -> E4M3 codes (RNE, satfinite)."""
    v = _c(values, np.float32)
    out = np.empty(v.shape, np.uint8)
    _L().orc_e4m3_encode_n(_p(v), v.size, _p(out))
    return out


# --------------------------------------------------------- weight formats ----

def quant_fp8_rowwise(w_bf16) -> tuple[np.ndarray, np.ndarray]:
    """bf16 W [n, k] -> (E4M3 codes uint8 [n, k], fp32 scales [n])."""
    w = _c(w_bf16, np.uint16)
    n, k = w.shape
    codes = np.empty((n, k), np.uint8)
    scales = np.empty((n,), np.float32)
    _L().orc_quant_fp8_rowwise(_p(w), n, k, _p(codes), _p(scales))
    return codes, scales


def int4_dequant(codes, scales_bf16, zeros) -> np.ndarray:
    """INT4 g128 -> bf16 bit patterns [n, k] of bf16_RNE((q - z) * s)."""
    c = _c(codes, np.uint8)
    s = _c(scales_bf16, np.uint16)
    z = _c(zeros, np.uint8)
    n, k = c.shape
    assert k % 128 == 0 and s.shape == (n, k // 128) and z.shape == (n, k // 128)
    out = np.empty((n, k), np.uint16)
    _L().orc_int4_dequant(_p(c), _p(s), _p(z), n, k, _p(out))
    return out


def int4_quant(w_bf16, group: int = 128):
    """Asymmetric min/max INT4 quantiser (see orc_int4_quant): bf16 bit
    patterns [n, k] -> (codes u8 [n, k], scales bf16 bits [n, k/group],
    zeros u8 [n, k/group])."""
    w = _c(w_bf16, np.uint16)
    n, k = w.shape
    assert group >= 1 and k % group == 0
    codes = np.empty((n, k), np.uint8)
    scales = np.empty((n, k // group), np.uint16)
    zeros = np.empty((n, k // group), np.uint8)
    _L().orc_int4_quant(_p(w), n, k, group, _p(codes), _p(scales), _p(zeros))
    return codes, scales, zeros


def int4_packed_sizes(n: int, k: int) -> tuple[int, int, int]:
    """Bytes of (packed codes, packed scales, packed zeros)."""
    blocks = ((n + 15) // 16) * (k // 128)
    return blocks * 1024, blocks * 32, blocks * 8


def int4_pack(codes, scales_bf16, zeros):
    c = _c(codes, np.uint8)
    s = _c(scales_bf16, np.uint16)
    z = _c(zeros, np.uint8)
    n, k = c.shape
    nb, ns, nz = int4_packed_sizes(n, k)
    pk, ps, pz = np.empty(nb, np.uint8), np.empty(ns, np.uint8), np.empty(nz, np.uint8)
    _L().orc_int4_pack(_p(c), _p(s), _p(z), n, k, _p(pk), _p(ps), _p(pz))
    return pk, ps, pz


def int4_unpack(packed, packed_scales, packed_zeros, n: int, k: int):
    """Returns (codes [n,k] u8, scales [n,k/128] bf16 bits, zeros [n,k/128] u8,
    count of nonzero padding entries)."""
    pk = _c(packed, np.uint8)
    ps = _c(packed_scales, np.uint8)
    pz = _c(packed_zeros, np.uint8)
    nb, ns, nz = int4_packed_sizes(n, k)
    assert pk.size == nb and ps.size == ns and pz.size == nz
    codes = np.empty((n, k), np.uint8)
    scales = np.empty((n, k // 128), np.uint16)
    zeros = np.empty((n, k // 128), np.uint8)
    bad = _L().orc_int4_unpack(_p(pk), _p(ps), _p(pz), n, k, _p(codes), _p(scales), _p(zeros))
    return codes, scales, zeros, int(bad)


# -------------------------------------------------------------- dq_gemm ----

def dq_gemm(wtype: int, data, scales, zeros, x_bf16, rows=None) -> np.ndarray:
    """y = x * deq(W)^T in float64. ``data`` is bf16 bits [n,k] (BF16),
    E4M3 codes [n,k] (FP8, ``scales`` fp32 [n]) or logical INT4 codes [n,k]
    (``scales`` bf16 bits [n,k/128], ``zeros`` u8 [n,k/128]). Returns
    [m, len(rows)] (or [m, n] when rows is None)."""
    x = _c(x_bf16, np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    m, k = x.shape
    if wtype == W_BF16:
        d = _c(data, np.uint16)
        s = None
        z = None
    elif wtype == W_FP8_E4M3:
        d = _c(data, np.uint8)
        s = _c(scales, np.float32)
        z = None
    elif wtype == W_INT4_G128:
        d = _c(data, np.uint8)
        s = _c(scales, np.uint16)
        z = _c(zeros, np.uint8)
    else:
        raise ValueError(wtype)
    n, kk = d.shape
    assert kk == k
    r = None if rows is None else _c(rows, np.int64)
    nrows = n if r is None else r.size
    y = np.empty((m, nrows), np.float64)
    rc = _L().orc_dq_gemm(int(wtype), _p(d), _p(s), _p(z), n, k, _p(x), m, _p(r), nrows, _p(y))
    if rc != 0:
        raise ValueError("orc_dq_gemm rejected its arguments")
    return y


# ------------------------------------------------------------ attention ----

def gqa_decode_attn(q_bf16, k_pool, v_pool, block_table, context_lens, hkv: int,
                    softmax_scale: float, rows=None) -> np.ndarray:
    """Paged GQA decode/verify attention in float64.

    q [B, W, Hq, D] bf16 bits; k_pool, v_pool [blocks, Hkv, 16, D] bf16 bits;
    block_table int32 [B, max_blocks]; context_lens int32 [B]. Returns
    [B, W, Hq, D] (rows None) or [len(rows), D] for flattened row ids
    r = (b*W + i)*Hq + h."""
    q = _c(q_bf16, np.uint16)
    kp = _c(k_pool, np.uint16)
    vp = _c(v_pool, np.uint16)
    bt = _c(block_table, np.int32)
    cl = _c(context_lens, np.int32)
    B, W, Hq, D = q.shape
    nblk = kp.shape[0]
    assert kp.shape == (nblk, hkv, 16, D) and vp.shape == kp.shape
    assert bt.ndim == 2 and bt.shape[0] == B and cl.shape == (B,)
    r = None if rows is None else _c(rows, np.int64)
    nrows = B * W * Hq if r is None else r.size
    out = np.empty((nrows, D), np.float64)
    rc = _L().orc_gqa_decode_attn(_p(q), _p(kp), _p(vp), _p(bt), bt.shape[1], _p(cl), nblk,
                                  B, W, Hq, hkv, D, float(softmax_scale), _p(r), nrows, _p(out))
    if rc != 0:
        raise ValueError("orc_gqa_decode_attn rejected its arguments")
    return out.reshape(B, W, Hq, D) if r is None else out


def gqa_decode_attn_fp8kv(q_bf16, k_codes, v_codes, block_table, context_lens, hkv: int,
                          softmax_scale: float, k_scale: float, v_scale: float,
                          rows=None) -> np.ndarray:
    """:func:`gqa_decode_attn` over an FP8-E4M3 cache, in float64.

    k_codes, v_codes [blocks, Hkv, 16, D] uint8 E4M3 codes; the cached values
    are decode(code) * k_scale and decode(code) * v_scale. Other arguments and
    the result as in :func:`gqa_decode_attn`."""
    q = _c(q_bf16, np.uint16)
    kp = _c(k_codes, np.uint8)
    vp = _c(v_codes, np.uint8)
    bt = _c(block_table, np.int32)
    cl = _c(context_lens, np.int32)
    B, W, Hq, D = q.shape
    nblk = kp.shape[0]
    assert kp.shape == (nblk, hkv, 16, D) and vp.shape == kp.shape
    assert bt.ndim == 2 and bt.shape[0] == B and cl.shape == (B,)
    r = None if rows is None else _c(rows, np.int64)
    nrows = B * W * Hq if r is None else r.size
    out = np.empty((nrows, D), np.float64)
    rc = _L().orc_gqa_decode_attn_fp8kv(_p(q), _p(kp), _p(vp), float(k_scale), float(v_scale),
                                        _p(bt), bt.shape[1], _p(cl), nblk, B, W, Hq, hkv, D,
                                        float(softmax_scale), _p(r), nrows, _p(out))
    if rc != 0:
        raise ValueError("orc_gqa_decode_attn_fp8kv rejected its arguments")
    return out.reshape(B, W, Hq, D) if r is None else out


# ------------------------------------------------------------ verify ----

def spec_verify_greedy(logits_bf16, draft, context_lens=None):
    """Greedy verify (orc_spec_verify_greedy). logits bf16 bits [b, w, vocab];
    draft int32 [b, w-1]. Returns (out int32 [b, w] with -1 past count,
    count int32 [b], new context_lens or None)."""
    lg = _c(logits_bf16, np.uint16)
    B, W, V = lg.shape
    d = _c(draft, np.int32).reshape(B, W - 1)
    out = np.full((B, W), -1, np.int32)
    cnt = np.zeros(B, np.int32)
    ctx = None if context_lens is None else _c(context_lens, np.int32).copy()
    _L().orc_spec_verify_greedy(_p(lg), B, W, V, _p(d), _p(out), _p(cnt), _p(ctx))
    out[np.arange(W)[None, :] >= cnt[:, None]] = -1
    return out, cnt, ctx


def spec_verify_sample(p, q, draft, u_accept, u_sample, context_lens=None):
    """Speculative sampling (orc_spec_verify_sample). p f32 [b, k, vocab];
    q f32 [b, k+1, vocab]; draft int32 [b, k]; u_accept f32 [b, k]; u_sample
    f32 [b]. Returns (out int32 [b, k+1] with -1 past count, count, ctx)."""
    pp = _c(p, np.float32)
    qq = _c(q, np.float32)
    B, K, V = pp.shape
    assert qq.shape == (B, K + 1, V)
    d = _c(draft, np.int32).reshape(B, K)
    ua = _c(u_accept, np.float32).reshape(B, K)
    us = _c(u_sample, np.float32).reshape(B)
    out = np.full((B, K + 1), -1, np.int32)
    cnt = np.zeros(B, np.int32)
    ctx = None if context_lens is None else _c(context_lens, np.int32).copy()
    _L().orc_spec_verify_sample(_p(pp), _p(qq), _p(d), _p(ua), _p(us), B, K, V, _p(out), _p(cnt), _p(ctx))
    out[np.arange(K + 1)[None, :] >= cnt[:, None]] = -1
    return out, cnt, ctx


# -------------------------------------------------------- RoPE / append ----

def rope(x, pos, base: float = 10000.0) -> np.ndarray:
    """Rotary embedding of head vectors x [rows, d] (float64) at positions
    pos [rows]: dims (2i, 2i+1) rotate by pos * base^(-2i/d)."""
    v = _c(x, np.float64).copy()
    rows, d = v.shape
    ps = _c(pos, np.float64).reshape(rows)
    _L().orc_rope(_p(v), rows, d, _p(ps), float(base))
    return v


def rope_kv_append(qkv_bf16, B: int, W: int, hq: int, hkv: int, base: float, context_lens, block_table,
                   num_blocks: int):
    """orc_rope_kv_append: returns (q [B, W, hq, d], k [B, W, hkv, d],
    v [B, W, hkv, d] as float64, slot int64 [B, W]: pool row
    phys * hkv * 16 + pos % 16 (add head * 16), -1 for no append)."""
    x = _c(qkv_bf16, np.uint16)
    d = x.shape[-1] // (hq + 2 * hkv)
    bt = _c(block_table, np.int32)
    ctx = _c(context_lens, np.int32)
    q = np.empty((B, W, hq, d))
    k = np.empty((B, W, hkv, d))
    v = np.empty((B, W, hkv, d))
    slot = np.empty((B, W), np.int64)
    rc = _L().orc_rope_kv_append(_p(x), B, W, hq, hkv, d, float(base), _p(ctx), _p(bt), bt.shape[1],
                                 num_blocks, _p(q), _p(k), _p(v), _p(slot))
    if rc != 0:
        raise ValueError("orc_rope_kv_append rejected its arguments")
    return q, k, v, slot
