"""GB300-native kernels for the memory-bound LLM decode step.

The compute lives in ``libdqd.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/dqd.h``). ``memory_bound_decode_dq_gb300.dqd``
is the thin ctypes binding over torch tensors; its names are the C names.
The binding is imported lazily so that the host-only modules (``synth``,
``bounds``, ``configs``) work on machines without the library or a GPU.
"""

_BINDING_NAMES = (
    "dq_gemm", "gqa_decode_attn", "pack_int4_g128", "quant_fp8_rowwise",
    "dq_gemm_workspace_bytes", "gqa_decode_attn_workspace_bytes",
    "pack_int4_g128_bytes", "DqdError", "Int4Packed", "Weight",
)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import dqd
        return getattr(dqd, name)
    raise AttributeError(name)
