"""Failure detection on the GPU without a fault: a bounded wait on a barrier
that nothing completes gives up, the sticky device error flag reports it
once, and the context keeps working (a following attention call is correct
and raises no flag)."""
import math

import numpy as np
import pytest

import oracle
from memory_bound_decode_dq_gb300 import synth
from gpu_util import assert_close, bf, f64, i32, require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_cuda()


@pytest.fixture(scope="module")
def dqd():
    from memory_bound_decode_dq_gb300 import dqd as m
    return m


def test_bounded_wait_gives_up_and_reports(dev, dqd):
    assert dqd.device_errors() == 0
    dqd.selftest_wait_timeout(1 << 12)
    flags = dqd.device_errors()
    assert flags & 1                       # the wait gave up and said so
    assert dqd.device_errors() == 0        # reading clears the flag


def test_context_stays_usable(dev, dqd):
    dqd.selftest_wait_timeout(1 << 10)
    assert dqd.device_errors() & 1
    kv = synth.paged_kv(3, "kv", (300,), 2)
    q = synth.normal_bf16(3, "q", (1, 1, 8, 128))
    out = dqd.gqa_decode_attn(bf(q, dev), bf(kv.k_pool, dev), bf(kv.v_pool, dev), i32(kv.block_table, dev),
                              i32(kv.context_lens, dev), 300)
    ref = oracle.gqa_decode_attn(q, kv.k_pool, kv.v_pool, kv.block_table, kv.context_lens, 2, 1 / math.sqrt(128))
    assert_close(f64(out), ref, what="attention after a timed-out wait")
    assert dqd.device_errors() == 0


def test_rejects_bad_poll_counts(dev, dqd):
    with pytest.raises(dqd.DqdError):
        dqd.selftest_wait_timeout(0)
    with pytest.raises(dqd.DqdError):
        dqd.selftest_wait_timeout((1 << 22) + 1)
