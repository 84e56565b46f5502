"""gqa_decode_attn_static_ws: attention for callers that cannot allocate
device memory.

Some callers (a serving runtime that forbids cudaMalloc after start-up, a
plug-in inside a process whose allocator it does not own) cannot hand the
library a workspace. This entry point uses a fixed scratch array inside the
library instead. The test calls it through the C ABI and checks it against
gqa_decode_attn (caller workspace) on two different calls in a row, so the
second call runs over whatever the first left in the shared scratch: the two
run the same plan and kernels, so they must agree bit for bit. The first pair
is also checked against the float64 oracle (a defect shared by both entry
points would pass the bit comparison). After a warm-up call, a further call
must leave the device's free memory unchanged, and an oversized call is
refused before any launch.

This file is collected last on purpose, and it passes both on its own in a
fresh process and after the rest of the suite."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from memory_bound_decode_dq_gb300 import synth
from gpu_util import assert_close, bf, bits, f64, i32, require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_cuda()


@pytest.fixture(scope="module")
def dqd():
    from memory_bound_decode_dq_gb300 import dqd as m
    return m


def static_ws_call(dqd, q, kp, vp, table, ctx, max_context, out, scale):
    lib = dqd.library()
    f = lib.gqa_decode_attn_static_ws
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p] + \
                 [ctypes.c_int32] * 6 + [ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
    B, W, Hq, D = q.shape
    nblk, Hkv = kp.shape[0], kp.shape[1]
    return f(q.data_ptr(), kp.data_ptr(), vp.data_ptr(), nblk, table.data_ptr(), table.shape[1],
             ctx.data_ptr(), max_context, B, W, Hq, Hkv, D, scale, out.data_ptr(),
             torch.cuda.current_stream().cuda_stream)


def make_case(dev, seed, B, W, hq, hkv, ctx):
    kv = synth.paged_kv(seed, "kv", ctx, hkv)
    q = synth.normal_bf16(seed, "q", (B, W, hq, 128))
    dev_args = (bf(q, dev), bf(kv.k_pool, dev), bf(kv.v_pool, dev), i32(kv.block_table, dev),
                i32(kv.context_lens, dev), int(max(ctx)))
    return dev_args, (q, kv)


@pytest.mark.parametrize("first,second", [
    ((1, 1, 32, 8, (8192,)), (3, 4, 8, 2, (70, 1000, 333))),
    ((2, 16, 32, 8, (600, 2000)), (1, 1, 64, 8, (5000,))),
])
def test_matches_workspace_entry_point_on_two_calls_in_a_row(dev, dqd, first, second):
    for i, (B, W, hq, hkv, ctx) in enumerate((first, second)):
        (q, kp, vp, table, cl, maxc), (qh, kv) = make_case(dev, 100 + i, B, W, hq, hkv, ctx)
        need = dqd.gqa_decode_attn_workspace_bytes(B, W, hq, hkv, 128, maxc)
        assert need > 0, "the case must exercise the split-KV scratch"
        want = dqd.gqa_decode_attn(q, kp, vp, table, cl, maxc)
        out = torch.full_like(q, float("nan"))
        st = static_ws_call(dqd, q, kp, vp, table, cl, maxc, out, 1 / math.sqrt(128))
        assert st == dqd.DQD_OK, dqd.library().dqd_last_error()
        torch.cuda.synchronize()
        # same plan, same kernels: identical bits, whatever the scratch held before
        assert np.array_equal(bits(out), bits(want)), f"static scratch, call {i + 1}: differs from gqa_decode_attn"
        if i == 0:
            ref = oracle.gqa_decode_attn(qh, kv.k_pool, kv.v_pool, kv.block_table, kv.context_lens, hkv,
                                         1 / math.sqrt(128))
            assert_close(f64(out), ref, what="static scratch against the oracle")
    assert dqd.device_errors() == 0


def test_warm_call_leaves_free_device_memory_unchanged(dev, dqd):
    """Once the first call has set the scratch up, a call reserves no device
    memory: the device's free memory is the same before and after it."""
    (q, kp, vp, table, cl, maxc), _ = make_case(dev, 300, 2, 6, 32, 8, (3000, 800))
    out = torch.empty_like(q)
    assert static_ws_call(dqd, q, kp, vp, table, cl, maxc, out, 0.088) == dqd.DQD_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    assert static_ws_call(dqd, q, kp, vp, table, cl, maxc, out, 0.088) == dqd.DQD_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 == free0


def test_oversized_call_is_refused_without_launch(dev, dqd, monkeypatch):
    # one 16-token chunk per CTA over 64 x 16 x 32 query rows needs far more
    # than the fixed scratch
    monkeypatch.setenv("DQD_ATTN_CHUNK_BLOCKS", "1")
    (q, kp, vp, table, cl, maxc), _ = make_case(dev, 7, 64, 16, 32, 8, tuple([512] * 64))
    out = torch.zeros_like(q)
    st = static_ws_call(dqd, q, kp, vp, table, cl, maxc, out, 0.088)
    assert st == dqd.DQD_ERR_WORKSPACE
    msg = dqd.library().dqd_last_error().decode()
    assert "static scratch" in msg and "gqa_decode_attn" in msg
    torch.cuda.synchronize()
    assert torch.count_nonzero(out.float()).item() == 0
