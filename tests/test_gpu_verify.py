"""GPU parity of the speculative verify step (spec_verify_greedy,
spec_verify_sample) against the oracle: token ids, counts and context
lengths are integers and must match exactly."""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_decode_dq_gb300 import synth
from gpu_util import bf, i32, require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_cuda()


@pytest.fixture(scope="module")
def dqd():
    from memory_bound_decode_dq_gb300 import dqd as m
    return m


def _greedy_case(seed, b, w, vocab, match=0.7):
    """Logits ~ N(0, 1) bf16 and drafts that follow the target's argmax with
    probability `match` per position (so accepted lengths vary)."""
    rng = np.random.default_rng(seed)
    lg = synth.normal_bf16(seed, "logits", (b, w, vocab))
    f = (lg.astype(np.uint32) << 16).view(np.float32)
    t = f.argmax(axis=2)
    draft = np.where(rng.random((b, w - 1)) < match, t[:, :w - 1], rng.integers(0, vocab, (b, w - 1)))
    ctx = rng.integers(w, 5000, b).astype(np.int32)
    return lg, draft.astype(np.int32), ctx


def _run_greedy(dqd, dev, lg, draft, ctx):
    ctx_d = i32(ctx, dev)
    out, cnt = dqd.spec_verify_greedy(bf(lg, dev), i32(draft, dev) if draft.shape[1] else None, ctx_d)
    return out.cpu().numpy(), cnt.cpu().numpy(), ctx_d.cpu().numpy()


@pytest.mark.parametrize("b,w,vocab", [(1, 6, 32000), (64, 6, 1000), (8, 16, 128256), (3, 1, 4096),
                                       (5, 4, 50257), (2, 3, 1), (7, 5, 13)])
def test_greedy_against_oracle(dev, dqd, b, w, vocab):
    lg, draft, ctx = _greedy_case(b * 31 + w + vocab, b, w, vocab)
    out, cnt, ctx2 = _run_greedy(dqd, dev, lg, draft, ctx)
    rout, rcnt, rctx = oracle.spec_verify_greedy(lg, draft, ctx)
    assert np.array_equal(cnt, rcnt)
    assert np.array_equal(ctx2, rctx)
    keep = np.arange(w)[None, :] < rcnt[:, None]
    assert np.array_equal(out[keep], rout[keep])
    assert np.all(cnt >= 1) and np.all(cnt <= w)


def test_greedy_ties_infinities_and_bad_ids(dev, dqd):
    V = 1000
    lg = np.zeros((4, 3, V), np.float32)
    lg[0, :, [17, 900]] = 5.0                           # ties: the smaller id
    lg[1, :, :] = -np.inf                               # all -inf: token 0
    lg[2, :, 250] = np.inf
    lg[3, :, 3] = 1.0
    bits_ = synth.f32_to_bf16_bits(lg)
    draft = np.array([[17, 17], [0, 5], [250, 250], [3 + V, 3]], np.int32)   # last: an id out of range
    ctx = np.full(4, 40, np.int32)
    out, cnt, ctx2 = _run_greedy(dqd, dev, bits_, draft, ctx)
    rout, rcnt, rctx = oracle.spec_verify_greedy(bits_, draft, ctx)
    assert list(cnt) == list(rcnt) == [3, 2, 3, 1]
    assert list(ctx2) == list(rctx) == [40, 39, 40, 38]
    assert out[0, 0] == 17 and out[1, 0] == 0 and out[2, 0] == 250 and out[3, 0] == 3


def test_greedy_rounds_reproduce_plain_greedy(dev, dqd):
    """Several draft + verify rounds through the GPU kernel emit exactly the
    token sequence of plain greedy decoding of the same synthetic target."""
    V, k, steps = 5003, 7, 80

    def target_next(prefix):
        h = 2166136261
        for t in prefix:
            h = (h * 16777619 + t + 3) % 1000003
        return h % V

    plain = [1]
    while len(plain) < 1 + steps:
        plain.append(target_next(plain))
    rng = np.random.default_rng(4)
    seq, ctx = [1], np.array([1 + k], np.int32)
    while len(seq) < 1 + steps:
        d, pref = [], list(seq)
        for _ in range(k):
            t = target_next(pref) if rng.random() < 0.6 else int(rng.integers(V))
            d.append(t)
            pref.append(t)
        block = [target_next(seq + d[:i]) for i in range(k + 1)]
        lg = rng.standard_normal((1, k + 1, V)).astype(np.float32)
        lg[0, np.arange(k + 1), block] = 20.0
        out, cnt, ctx2 = _run_greedy(dqd, dev, synth.f32_to_bf16_bits(lg), np.array([d], np.int32), ctx)
        seq.extend(int(t) for t in out[0, :cnt[0]])
        # the cache keeps the round's input and the accepted drafts
        assert ctx2[0] == ctx[0] - (k - (cnt[0] - 1))
    assert seq[:len(plain)] == plain


def _dists(rng, b, rows, vocab, peaked):
    x = rng.standard_normal((b, rows, vocab)) * (4.0 if peaked else 1.0)
    e = np.exp(x - x.max(axis=2, keepdims=True))
    return (e / e.sum(axis=2, keepdims=True)).astype(np.float32)


@pytest.mark.parametrize("b,k,vocab", [(1, 4, 32000), (16, 1, 1000), (64, 5, 4096), (4, 15, 50257),
                                       (9, 0, 777), (2, 3, 1)])
def test_sample_against_oracle(dev, dqd, b, k, vocab):
    rng = np.random.default_rng(b * 13 + k + vocab)
    q = _dists(rng, b, k + 1, vocab, peaked=True)
    p = _dists(rng, b, k, vocab, peaked=True)
    # drafts drawn from p; a few out-of-range ids
    draft = np.zeros((b, k), np.int32)
    for r in range(b):
        for i in range(k):
            draft[r, i] = rng.choice(vocab, p=p[r, i] / p[r, i].sum())
    if b * k > 3:
        draft.reshape(-1)[2] = vocab + 5
    ua = rng.random((b, k)).astype(np.float32)
    us = rng.random(b).astype(np.float32)
    ctx = rng.integers(k + 1, 9000, b).astype(np.int32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    ctx_d = t(ctx)
    out, cnt = dqd.spec_verify_sample(t(p), t(q), t(draft), t(ua), t(us), ctx_d)
    rout, rcnt, rctx = oracle.spec_verify_sample(p, q, draft, ua, us, ctx)
    assert np.array_equal(cnt.cpu().numpy(), rcnt)
    assert np.array_equal(out.cpu().numpy(), rout)
    assert np.array_equal(ctx_d.cpu().numpy(), rctx)


def test_sample_exercise_distribution(dev, dqd):
    """p = (0.2, 0.2, 0.6), q = (0.5, 0.3, 0.2): over stratified grids of the
    draft draw and both uniforms, acceptance is 0.6 and the output is
    distributed exactly as q."""
    p, q = [0.2, 0.2, 0.6], [0.5, 0.3, 0.2]
    cp = np.cumsum(p)
    xs = [int(np.searchsorted(cp, (i + 0.5) / 50, side="right")) for i in range(50)]
    us = (np.arange(24) + 0.5) / 24
    xx, ua, us_ = np.meshgrid(np.array(xs), us, us, indexing="ij")
    n = xx.size
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    P = np.broadcast_to(np.array(p, np.float32), (n, 1, 3))
    Q = np.broadcast_to(np.array([q, q], np.float32), (n, 2, 3))
    out, cnt = dqd.spec_verify_sample(t(P), t(Q), t(xx.reshape(n, 1).astype(np.int32)),
                                      t(ua.reshape(n, 1).astype(np.float32)), t(us_.reshape(n).astype(np.float32)))
    first = out[:, 0].cpu().numpy()
    assert np.sum(cnt.cpu().numpy() == 2) * 5 == n * 3
    assert [int(np.sum(first == v)) * 10 for v in range(3)] == [5 * n, 3 * n, 2 * n]


def test_rejects_bad_arguments(dev, dqd):
    lg = torch.zeros((2, 3, 8), dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError):
        dqd.spec_verify_greedy(lg, torch.zeros((2, 3), dtype=torch.int32, device=dev))
    lib = dqd.library()
    assert lib.spec_verify_greedy(None, 2, 3, 8, None, None, None, None, None) != dqd.DQD_OK
    assert lib.spec_verify_sample(None, None, None, None, None, 1, -1, 8, None, None, None, None) != dqd.DQD_OK


def test_no_device_error_flags(dev, dqd):
    assert dqd.device_errors() == 0


def test_sample_at_full_vocabulary(dev, dqd):
    """Speculative sampling at the 8B vocabulary (128256), batch 64, 5 drafts:
    tokens, counts and contexts equal the oracle's for every request."""
    b, k, vocab = 64, 5, 128256
    rng = np.random.default_rng(77)
    g = torch.Generator(device=dev)
    g.manual_seed(77)
    logits_q = torch.randn((b, k + 1, vocab), generator=g, device=dev) * 3.0
    logits_p = logits_q[:, :k] + torch.randn((b, k, vocab), generator=g, device=dev)  # a draft close to the target
    q = torch.softmax(logits_q, dim=2).contiguous()
    p = torch.softmax(logits_p, dim=2).contiguous()
    draft = torch.multinomial(p.view(-1, vocab), 1, generator=g).view(b, k).to(torch.int32)
    ua = torch.from_numpy(rng.random((b, k)).astype(np.float32)).to(dev)
    us = torch.from_numpy(rng.random(b).astype(np.float32)).to(dev)
    ctx = torch.full((b,), 3000, dtype=torch.int32, device=dev)
    out, cnt = dqd.spec_verify_sample(p, q, draft, ua, us, ctx)
    rout, rcnt, rctx = oracle.spec_verify_sample(p.cpu().numpy(), q.cpu().numpy(), draft.cpu().numpy(),
                                                 ua.cpu().numpy(), us.cpu().numpy(), np.full(b, 3000, np.int32))
    assert np.array_equal(cnt.cpu().numpy(), rcnt)
    assert np.array_equal(out.cpu().numpy(), rout)
    assert np.array_equal(ctx.cpu().numpy(), rctx)
    assert 1 < rcnt.mean() < k + 1          # the drafts are accepted some of the time
