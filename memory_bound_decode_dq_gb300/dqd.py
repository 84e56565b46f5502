"""Thin ctypes binding of libdqd over torch tensors.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libdqd.so (built by ``memory_bound_decode_dq_gb300.build``). The
names are the C names declared in ``include/dqd.h``. There is no fallback: if
the library is missing, importing this module raises ImportError.

torch provides device memory and streams: tensors' ``data_ptr()`` and the
current stream's handle are passed to the C calls unchanged.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdqd.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"` "
        "or `python memory_bound_decode_dq_gb300/build.py` (needs nvcc)")

_lib = ctypes.CDLL(LIB_PATH)

DQD_OK, DQD_ERR_INVALID_ARG, DQD_ERR_UNSUPPORTED, DQD_ERR_WORKSPACE, DQD_ERR_CUDA = range(5)
DQD_W_BF16, DQD_W_FP8_E4M3, DQD_W_INT4_G128 = 0, 1, 2
DQD_WS_COUNTER_BYTES = 65536
DQD_DEVICE_ERR_WAIT_TIMEOUT, DQD_DEVICE_ERR_BAD_INPUT = 1, 2


class _WeightDesc(ctypes.Structure):
    _fields_ = [("type", ctypes.c_int32), ("n", ctypes.c_int64), ("k", ctypes.c_int64),
                ("data", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("zeros", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I32, _I64, _SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_SIGS = {
    "dqd_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "dqd_last_error": (ctypes.c_char_p, []),
    "dqd_version": (ctypes.c_char_p, []),
    "dqd_device_errors": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32)]),
    "dqd_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint32, _P]),
    "pack_int4_g128_bytes": (_SZ, [_I64, _I64, ctypes.c_int]),
    "pack_int4_g128": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _P, _P, _P, _P]),
    "quant_fp8_rowwise": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P]),
    "quant_int4_g128": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P, _P]),
    "spec_verify_greedy": (ctypes.c_int, [_P, _I32, _I32, _I64, _P, _P, _P, _P, _P]),
    "rope_kv_append": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _I32, ctypes.c_float, _P, _I32, _P, _I64,
                                      _P, _P, _I32, ctypes.c_float, ctypes.c_float, _P, _P]),
    "spec_verify_sample": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _I32, _I64, _P, _P, _P, _P]),
    "dq_gemm_qkv_rope_append": (ctypes.c_int, [ctypes.POINTER(_WeightDesc), _P, _I32, _I32, _I32, _I32, _I32,
                                               ctypes.c_float, _P, _I32, _P, _I64, _P, _P, _I32, ctypes.c_float,
                                               ctypes.c_float, _P, _P, _SZ, _P]),
    "dq_gemm_workspace_bytes": (ctypes.c_int, [ctypes.POINTER(_WeightDesc), _I64, ctypes.POINTER(_SZ)]),
    "dq_gemm": (ctypes.c_int, [ctypes.POINTER(_WeightDesc), _P, _I64, _P, _P, _SZ, _P]),
    "gqa_decode_attn_workspace_bytes": (ctypes.c_int, [_I32, _I32, _I32, _I32, _I32, _I32,
                                                       ctypes.POINTER(_SZ)]),
    "gqa_decode_attn": (ctypes.c_int, [_P, _P, _P, _I64, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32,
                                       _I32, ctypes.c_float, _P, _P, _SZ, _P]),
    "gqa_decode_attn_fp8kv_workspace_bytes": (ctypes.c_int, [_I32, _I32, _I32, _I32, _I32, _I32,
                                                             ctypes.POINTER(_SZ)]),
    "gqa_decode_attn_fp8kv": (ctypes.c_int, [_P, _P, _P, _I64, _P, _I32, _P, _I32, _I32, _I32, _I32,
                                             _I32, _I32, ctypes.c_float, ctypes.c_float,
                                             ctypes.c_float, _P, _P, _SZ, _P]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class DqdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = _lib.dqd_status_string(status).decode()
        detail = _lib.dqd_last_error().decode()
        super().__init__(f"{where}: {name}: {detail}")


def _check(status: int, where: str) -> None:
    if status != DQD_OK:
        raise DqdError(status, where)


def version() -> str:
    return _lib.dqd_version().decode()


def device_errors() -> int:
    """OR of the kernels' device error flags since the last call (0: none;
    DQD_DEVICE_ERR_WAIT_TIMEOUT: a bounded wait on an asynchronous copy gave
    up; DQD_DEVICE_ERR_BAD_INPUT: an input outside its documented range was
    clamped). Synchronises and clears the flags."""
    v = ctypes.c_uint32(0)
    _check(_lib.dqd_device_errors(ctypes.byref(v)), "dqd_device_errors")
    return int(v.value)


def selftest_wait_timeout(polls: int = 1 << 16, stream=None) -> None:
    """Run one bounded wait that runs out (see dqd_selftest_wait_timeout)."""
    _check(_lib.dqd_selftest_wait_timeout(int(polls), _stream(stream)), "dqd_selftest_wait_timeout")


def library() -> ctypes.CDLL:
    """The loaded libdqd handle (for callers that want the raw C ABI)."""
    return _lib


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name: str, dtypes, device=None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


_U8 = (torch.uint8,)
_B16 = (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (torch.bfloat16, torch.int16)
_F32 = (torch.float32,)
_I32T = (torch.int32,)


# ------------------------------------------------------------ workspace ----

_ws_lock = threading.Lock()
_ws_cache: dict = {}


def workspace(nbytes: int, device, stream=None) -> torch.Tensor | None:
    """A zero-initialised workspace of at least ``nbytes`` for ``device``,
    cached per (device, stream). Every library call leaves the counter region
    zero, so a cached buffer can be reused by later calls on the same stream."""
    if nbytes == 0:
        return None
    dev = torch.device(device)
    sid = (stream or torch.cuda.current_stream(dev)).cuda_stream
    key = (dev.index, sid)
    with _ws_lock:
        buf = _ws_cache.get(key)
        if buf is None or buf.numel() < nbytes:
            size = max(nbytes, 2 * (buf.numel() if buf is not None else 0))
            buf = torch.zeros(size, dtype=torch.uint8, device=dev)
            _ws_cache[key] = buf
        return buf


# --------------------------------------------------------------- weights ----

@dataclass
class Int4Packed:
    """INT4 g128 weight in the packed layout of include/dqd.h."""
    packed: torch.Tensor
    scales: torch.Tensor
    zeros: torch.Tensor
    n: int
    k: int


@dataclass
class Weight:
    """W [n out, k in] for dq_gemm. ``type`` is DQD_W_BF16, DQD_W_FP8_E4M3 or
    DQD_W_INT4_G128; the tensors stay referenced for the call's lifetime."""
    type: int
    n: int
    k: int
    data: torch.Tensor
    scales: torch.Tensor | None = None
    zeros: torch.Tensor | None = None

    @staticmethod
    def bf16(w: torch.Tensor) -> "Weight":
        _need(w, "w", _B16)
        return Weight(DQD_W_BF16, w.shape[0], w.shape[1], w)

    @staticmethod
    def fp8(codes: torch.Tensor, scales: torch.Tensor) -> "Weight":
        _need(codes, "codes", _U8 + ((torch.float8_e4m3fn,) if hasattr(torch, "float8_e4m3fn") else ()))
        _need(scales, "scales", _F32)
        return Weight(DQD_W_FP8_E4M3, codes.shape[0], codes.shape[1], codes, scales)

    @staticmethod
    def int4(p: Int4Packed) -> "Weight":
        return Weight(DQD_W_INT4_G128, p.n, p.k, p.packed, p.scales, p.zeros)

    def desc(self) -> _WeightDesc:
        return _WeightDesc(int(self.type), int(self.n), int(self.k), _ptr(self.data),
                           _ptr(self.scales), _ptr(self.zeros))


# ------------------------------------------------------------ functions ----

def pack_int4_g128_bytes(n: int, k: int, which: int) -> int:
    return int(_lib.pack_int4_g128_bytes(n, k, which))


def pack_int4_g128(codes: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor,
                   stream=None) -> Int4Packed:
    """Logical INT4 g128 (codes u8 [n,k], bf16 scales [n,k/128], u8 zeros
    [n,k/128]) -> packed layout, on the GPU."""
    _need(codes, "codes", _U8)
    dev = codes.device
    _need(scales, "scales", _B16, dev)
    _need(zeros, "zeros", _U8, dev)
    n, k = codes.shape
    sizes = [pack_int4_g128_bytes(n, k, i) for i in range(3)]
    if 0 in sizes:
        raise ValueError(f"pack_int4_g128: unsupported shape n={n} k={k} (k must be a multiple of 128)")
    if scales.shape != (n, k // 128) or zeros.shape != (n, k // 128):
        raise ValueError("pack_int4_g128: scales and zeros must be [n, k/128]")
    out = [torch.empty(s, dtype=torch.uint8, device=dev) for s in sizes]
    _check(_lib.pack_int4_g128(_ptr(codes), _ptr(scales), _ptr(zeros), n, k, _ptr(out[0]),
                               _ptr(out[1]), _ptr(out[2]), _stream(stream)), "pack_int4_g128")
    return Int4Packed(out[0], out[1], out[2], n, k)


def quant_fp8_rowwise(w: torch.Tensor, stream=None):
    """bf16 W [n, k] -> (E4M3 codes u8 [n, k], fp32 scales [n])."""
    _need(w, "w", _B16)
    n, k = w.shape
    codes = torch.empty((n, k), dtype=torch.uint8, device=w.device)
    scales = torch.empty((n,), dtype=torch.float32, device=w.device)
    _check(_lib.quant_fp8_rowwise(_ptr(w), n, k, _ptr(codes), _ptr(scales), _stream(stream)),
           "quant_fp8_rowwise")
    return codes, scales


def quant_int4_g128(w: torch.Tensor, stream=None):
    """bf16 W [n, k] -> (codes u8 [n, k] in 0..15, bf16 scales [n, k/128],
    zero points u8 [n, k/128]): asymmetric min/max per 128-group."""
    _need(w, "w", _B16)
    n, k = w.shape
    codes = torch.empty((n, k), dtype=torch.uint8, device=w.device)
    scales = torch.empty((n, k // 128), dtype=torch.bfloat16, device=w.device)
    zeros = torch.empty((n, k // 128), dtype=torch.uint8, device=w.device)
    _check(_lib.quant_int4_g128(_ptr(w), n, k, _ptr(codes), _ptr(scales), _ptr(zeros), _stream(stream)),
           "quant_int4_g128")
    return codes, scales, zeros


def dq_gemm_workspace_bytes(weight: Weight, m: int) -> int:
    out = _SZ(0)
    d = weight.desc()
    _check(_lib.dq_gemm_workspace_bytes(ctypes.byref(d), int(m), ctypes.byref(out)),
           "dq_gemm_workspace_bytes")
    return int(out.value)


def dq_gemm(weight: Weight, x: torch.Tensor, y: torch.Tensor | None = None,
            ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = x * deq(W)^T. x bf16 [m, k] (or [k]); returns bf16 [m, n]."""
    _need(x, "x", _B16)
    squeeze = x.dim() == 1
    x2 = x.view(1, -1) if squeeze else x
    m, k = x2.shape
    if k != weight.k:
        raise ValueError(f"dq_gemm: x has k={k}, weight has k={weight.k}")
    if y is None:
        y = torch.empty((m, weight.n), dtype=torch.bfloat16, device=x.device)
    else:
        _need(y, "y", _B16, x.device)
        if tuple(y.shape) not in ((m, weight.n),) + (((weight.n,),) if squeeze else ()):
            raise ValueError("dq_gemm: y must be [m, n]")
    d = weight.desc()
    need = dq_gemm_workspace_bytes(weight, m)
    if ws is None:
        ws = workspace(need, x.device, stream)
    _check(_lib.dq_gemm(ctypes.byref(d), _ptr(x2), m, _ptr(y), _ptr(ws),
                        0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
           "dq_gemm")
    return y.view(-1) if squeeze and y.dim() == 2 else y


def gqa_decode_attn_workspace_bytes(b: int, w: int, hq: int, hkv: int, d: int, max_context: int) -> int:
    out = _SZ(0)
    _check(_lib.gqa_decode_attn_workspace_bytes(b, w, hq, hkv, d, max_context, ctypes.byref(out)),
           "gqa_decode_attn_workspace_bytes")
    return int(out.value)


def gqa_decode_attn_fp8kv_workspace_bytes(b: int, w: int, hq: int, hkv: int, d: int,
                                          max_context: int) -> int:
    out = _SZ(0)
    _check(_lib.gqa_decode_attn_fp8kv_workspace_bytes(b, w, hq, hkv, d, max_context,
                                                      ctypes.byref(out)),
           "gqa_decode_attn_fp8kv_workspace_bytes")
    return int(out.value)


def _attn_args(name, q, k_pool, v_pool, pool_types, block_table, context_lens, softmax_scale, out):
    _need(q, "q", _B16)
    dev = q.device
    _need(k_pool, "k_pool", pool_types, dev)
    _need(v_pool, "v_pool", pool_types, dev)
    _need(block_table, "block_table", _I32T, dev)
    _need(context_lens, "context_lens", _I32T, dev)
    B, W, Hq, D = q.shape
    nblk, Hkv, bs, D2 = k_pool.shape
    if bs != 16 or D2 != D or v_pool.shape != k_pool.shape:
        raise ValueError(f"{name}: pools must be [num_blocks, Hkv, 16, D] and equal shapes")
    if block_table.dim() != 2 or block_table.shape[0] != B or context_lens.shape != (B,):
        raise ValueError(f"{name}: block_table must be [B, max_blocks], context_lens [B]")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q, dtype=torch.bfloat16)
    else:
        _need(out, "out", _B16, dev)
        if out.shape != q.shape:
            raise ValueError(f"{name}: out must have q's shape")
    return (B, W, Hq, Hkv, D, nblk), float(softmax_scale), out


def gqa_decode_attn(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                    block_table: torch.Tensor, context_lens: torch.Tensor, max_context: int,
                    softmax_scale: float | None = None, out: torch.Tensor | None = None,
                    ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Paged GQA decode/verify attention. q bf16 [B, W, Hq, D]; pools bf16
    [num_blocks, Hkv, 16, D]; block_table int32 [B, max_blocks]; context_lens
    int32 [B] (device, includes the W new tokens); max_context: host bound."""
    (B, W, Hq, Hkv, D, nblk), scale, out = _attn_args(
        "gqa_decode_attn", q, k_pool, v_pool, _B16, block_table, context_lens, softmax_scale, out)
    need = gqa_decode_attn_workspace_bytes(B, W, Hq, Hkv, D, int(max_context))
    if ws is None:
        ws = workspace(need, q.device, stream)
    _check(_lib.gqa_decode_attn(_ptr(q), _ptr(k_pool), _ptr(v_pool), nblk, _ptr(block_table),
                                block_table.shape[1], _ptr(context_lens), int(max_context), B, W, Hq,
                                Hkv, D, scale, _ptr(out), _ptr(ws),
                                0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
           "gqa_decode_attn")
    return out


def gqa_decode_attn_fp8kv(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                          block_table: torch.Tensor, context_lens: torch.Tensor, max_context: int,
                          k_scale: float, v_scale: float, softmax_scale: float | None = None,
                          out: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                          stream=None) -> torch.Tensor:
    """:func:`gqa_decode_attn` over an FP8-E4M3 cache: pools uint8 (or
    float8_e4m3fn) codes [num_blocks, Hkv, 16, D]; cached values are
    code * k_scale and code * v_scale."""
    pool_types = _U8 + ((torch.float8_e4m3fn,) if hasattr(torch, "float8_e4m3fn") else ())
    (B, W, Hq, Hkv, D, nblk), scale, out = _attn_args(
        "gqa_decode_attn_fp8kv", q, k_pool, v_pool, pool_types, block_table, context_lens,
        softmax_scale, out)
    need = gqa_decode_attn_fp8kv_workspace_bytes(B, W, Hq, Hkv, D, int(max_context))
    if ws is None:
        ws = workspace(need, q.device, stream)
    _check(_lib.gqa_decode_attn_fp8kv(_ptr(q), _ptr(k_pool), _ptr(v_pool), nblk, _ptr(block_table),
                                      block_table.shape[1], _ptr(context_lens), int(max_context), B,
                                      W, Hq, Hkv, D, scale, float(k_scale), float(v_scale), _ptr(out),
                                      _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                      _stream(stream)),
           "gqa_decode_attn_fp8kv")
    return out


# ---------------------------------------------------------------- verify ----

def spec_verify_greedy(logits: torch.Tensor, draft: torch.Tensor | None,
                       context_lens: torch.Tensor | None = None, out: torch.Tensor | None = None,
                       count: torch.Tensor | None = None, stream=None):
    """Greedy verify. logits bf16 [b, w, vocab]; draft int32 [b, w-1];
    context_lens int32 [b] updated in place (None: left alone). Returns
    (out int32 [b, w] = the target's predictions, count int32 [b]): the
    round emits out[r, :count[r]]."""
    _need(logits, "logits", _B16)
    dev = logits.device
    b, w, vocab = logits.shape
    if w > 1:
        _need(draft, "draft", _I32T, dev)
        if tuple(draft.shape) != (b, w - 1):
            raise ValueError("spec_verify_greedy: draft must be [b, w-1]")
    if context_lens is not None:
        _need(context_lens, "context_lens", _I32T, dev)
    out = torch.empty((b, w), dtype=torch.int32, device=dev) if out is None else out
    count = torch.empty((b,), dtype=torch.int32, device=dev) if count is None else count
    _need(out, "out", _I32T, dev)
    _need(count, "count", _I32T, dev)
    _check(_lib.spec_verify_greedy(_ptr(logits), b, w, vocab, _ptr(draft) if w > 1 else None, _ptr(out),
                                   _ptr(count), _ptr(context_lens), _stream(stream)), "spec_verify_greedy")
    return out, count


def spec_verify_sample(p: torch.Tensor, q: torch.Tensor, draft: torch.Tensor, u_accept: torch.Tensor,
                       u_sample: torch.Tensor, context_lens: torch.Tensor | None = None, stream=None):
    """Speculative sampling. p f32 [b, k, vocab]; q f32 [b, k+1, vocab];
    draft int32 [b, k]; u_accept f32 [b, k]; u_sample f32 [b]. Returns
    (out int32 [b, k+1], count int32 [b]); context_lens updated in place."""
    _need(q, "q", _F32)
    dev = q.device
    b, k1, vocab = q.shape
    k = k1 - 1
    for t, name in ((p, "p"), (u_accept, "u_accept"), (u_sample, "u_sample")):
        _need(t, name, _F32, dev)
    _need(draft, "draft", _I32T, dev)
    if tuple(p.shape) != (b, k, vocab) or tuple(draft.shape) != (b, k) or tuple(u_accept.shape) != (b, k) \
            or tuple(u_sample.shape) != (b,):
        raise ValueError("spec_verify_sample: shapes must be p [b,k,V], draft/u_accept [b,k], u_sample [b]")
    if context_lens is not None:
        _need(context_lens, "context_lens", _I32T, dev)
    out = torch.full((b, k + 1), -1, dtype=torch.int32, device=dev)
    count = torch.empty((b,), dtype=torch.int32, device=dev)
    _check(_lib.spec_verify_sample(_ptr(p), _ptr(q), _ptr(draft), _ptr(u_accept), _ptr(u_sample), b, k, vocab,
                                   _ptr(out), _ptr(count), _ptr(context_lens), _stream(stream)),
           "spec_verify_sample")
    return out, count


# ------------------------------------------------------ RoPE and append ----

def rope_kv_append(qkv: torch.Tensor, b: int, w: int, hq: int, hkv: int, k_pool: torch.Tensor,
                   v_pool: torch.Tensor, block_table: torch.Tensor, context_lens: torch.Tensor,
                   rope_base: float = 10000.0, k_scale: float = 1.0, v_scale: float = 1.0,
                   q_out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Rotate the new tokens' q and k, append k and v to the paged cache.
    qkv bf16 [b*w, (hq + 2*hkv) * d]; pools [num_blocks, hkv, 16, d], bf16
    or uint8 / float8_e4m3fn (FP8 cache with k_scale, v_scale). Returns
    q_out bf16 [b, w, hq, d]."""
    _need(qkv, "qkv", _B16)
    dev = qkv.device
    f8_types = _U8 + ((torch.float8_e4m3fn,) if hasattr(torch, "float8_e4m3fn") else ())
    fp8 = k_pool.dtype in f8_types
    _need(k_pool, "k_pool", f8_types if fp8 else _B16, dev)
    _need(v_pool, "v_pool", f8_types if fp8 else _B16, dev)
    _need(block_table, "block_table", _I32T, dev)
    _need(context_lens, "context_lens", _I32T, dev)
    rows, width = qkv.shape
    d = width // (hq + 2 * hkv)
    if rows != b * w or width != (hq + 2 * hkv) * d or tuple(k_pool.shape[1:]) != (hkv, 16, d) \
            or v_pool.shape != k_pool.shape:
        raise ValueError("rope_kv_append: qkv must be [b*w, (hq+2*hkv)*d], pools [num_blocks, hkv, 16, d]")
    if q_out is None:
        q_out = torch.empty((b, w, hq, d), dtype=torch.bfloat16, device=dev)
    _need(q_out, "q_out", _B16, dev)
    _check(_lib.rope_kv_append(_ptr(qkv), b, w, hq, hkv, d, float(rope_base), _ptr(block_table),
                               block_table.shape[1], _ptr(context_lens), k_pool.shape[0], _ptr(k_pool),
                               _ptr(v_pool), 1 if fp8 else 0, float(k_scale), float(v_scale), _ptr(q_out),
                               _stream(stream)), "rope_kv_append")
    return q_out


def dq_gemm_qkv_rope_append(weight: Weight, x: torch.Tensor, b: int, w: int, hq: int, hkv: int,
                            k_pool: torch.Tensor, v_pool: torch.Tensor, block_table: torch.Tensor,
                            context_lens: torch.Tensor, rope_base: float = 10000.0, k_scale: float = 1.0,
                            v_scale: float = 1.0, q_out: torch.Tensor | None = None,
                            ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The QKV projection of the new tokens fused with rope_kv_append: x bf16
    [b*w, k], weight [(hq + 2*hkv) * 128, k]; rotates q and k, appends k and v
    to the paged cache (bf16 pools, or uint8 / float8_e4m3fn for an FP8 cache
    with k_scale, v_scale). Returns q_out bf16 [b, w, hq, 128]."""
    _need(x, "x", _B16)
    dev = x.device
    f8_types = _U8 + ((torch.float8_e4m3fn,) if hasattr(torch, "float8_e4m3fn") else ())
    fp8 = k_pool.dtype in f8_types
    _need(k_pool, "k_pool", f8_types if fp8 else _B16, dev)
    _need(v_pool, "v_pool", f8_types if fp8 else _B16, dev)
    _need(block_table, "block_table", _I32T, dev)
    _need(context_lens, "context_lens", _I32T, dev)
    d = 128
    if tuple(x.shape) != (b * w, weight.k) or weight.n != (hq + 2 * hkv) * d \
            or tuple(k_pool.shape[1:]) != (hkv, 16, d) or v_pool.shape != k_pool.shape:
        raise ValueError("dq_gemm_qkv_rope_append: x must be [b*w, k], W [(hq+2*hkv)*128, k], "
                         "pools [num_blocks, hkv, 16, 128]")
    if q_out is None:
        q_out = torch.empty((b, w, hq, d), dtype=torch.bfloat16, device=dev)
    _need(q_out, "q_out", _B16, dev)
    need = dq_gemm_workspace_bytes(weight, b * w)
    if ws is None:
        ws = workspace(need, dev, stream)
    desc = weight.desc()
    _check(_lib.dq_gemm_qkv_rope_append(ctypes.byref(desc), _ptr(x), b, w, hq, hkv, d, float(rope_base),
                                        _ptr(block_table), block_table.shape[1], _ptr(context_lens),
                                        k_pool.shape[0], _ptr(k_pool), _ptr(v_pool), 1 if fp8 else 0,
                                        float(k_scale), float(v_scale), _ptr(q_out), _ptr(ws),
                                        0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
           "dq_gemm_qkv_rope_append")
    return q_out
