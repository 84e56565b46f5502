"""Parity at the full workload sizes, in the launch configuration the
benchmark times. The oracle evaluates sampled output rows (every row where it
finishes in seconds); inputs are drawn once per case on the device and the
sampled slices are copied back for the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from memory_bound_decode_dq_gb300 import configs, synth
from gpu_util import assert_close, bits, f64, require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_cuda()


@pytest.fixture(scope="module")
def dqd():
    from memory_bound_decode_dq_gb300 import dqd as m
    return m


def sample_rows(n: int, count: int, seed: int) -> np.ndarray:
    if count >= n:
        return np.arange(n)
    r = np.random.default_rng(seed).choice(n, count - 2, replace=False)
    return np.unique(np.concatenate([[0, n - 1], r]))


def check_gemm(dqd, dev, case, seed, max_oracle_macs=4e8):
    n, k, m = case.n, case.k, case.m
    x = synth.normal_bf16(seed, case.name + ".x", (m, k), device=dev)
    rows = sample_rows(n, max(16, int(max_oracle_macs // (m * k))), seed)
    ridx = torch.as_tensor(rows, device=dev)
    if case.wtype == oracle.W_INT4_G128:
        wq = synth.int4_weight(seed, case.name, n, k, device=dev)
        weight = dqd.Weight.int4(dqd.pack_int4_g128(wq.codes, wq.scales, wq.zeros))
        host = (wq.codes[ridx].cpu().numpy(), bits(wq.scales[ridx]), wq.zeros[ridx].cpu().numpy())
    else:
        if case.outliers:
            w = synth.bf16_weight_outliers_device(seed, case.name, n, k, 0.02, case.outliers, 20.0, dev)
        else:
            w = synth.normal_bf16(seed, case.name, (n, k), 0.02, device=dev)
        if case.wtype == oracle.W_BF16:
            weight = dqd.Weight.bf16(w)
            host = (bits(w[ridx]), None, None)
        else:
            codes, scales = dqd.quant_fp8_rowwise(w)
            weight = dqd.Weight.fp8(codes, scales)
            rc, rs = oracle.quant_fp8_rowwise(bits(w[ridx]))
            assert np.array_equal(codes[ridx].cpu().numpy(), rc), "GPU FP8 codes differ from the oracle's"
            assert np.array_equal(scales[ridx].cpu().numpy(), rs)
            host = (rc, rs, None)
    y = dqd.dq_gemm(weight, x)
    ref = oracle.dq_gemm(case.wtype, *host, bits(x))
    assert_close(f64(y[:, ridx]), ref, what=case.name)


def check_attn(dqd, dev, case, seed, max_groups=None):
    B, W, hq, hkv = case.batch, case.width, case.hq, case.hkv
    G = hq // hkv
    ctx = np.asarray(case.context, np.int32)
    table, nblk = synth.block_table(seed, case.name + ".table", ctx, case.shuffle)
    shape = (nblk, hkv, 16, 128)
    if case.kv_fp8:
        kp = synth.e4m3_codes(seed, case.name + ".k", shape, device=dev)
        vp = synth.e4m3_codes(seed, case.name + ".v", shape, device=dev)
    else:
        kp = synth.normal_bf16(seed, case.name + ".k", shape, 1.0, device=dev)
        vp = synth.normal_bf16(seed, case.name + ".v", shape, 1.0, device=dev)
    q = synth.normal_bf16(seed, case.name + ".q", (B, W, hq, 128), device=dev)
    args = (q, kp, vp, torch.from_numpy(table).to(dev), torch.from_numpy(ctx).to(dev), int(ctx.max()))
    if case.kv_fp8:
        out = dqd.gqa_decode_attn_fp8kv(*args, case.k_scale, case.v_scale)
    else:
        out = dqd.gqa_decode_attn(*args)
    groups = [(b, g) for b in range(B) for g in range(hkv)]
    if max_groups is not None and len(groups) > max_groups:
        pick = np.random.default_rng(seed).choice(len(groups), max_groups, replace=False)
        groups = [groups[i] for i in sorted(pick)]
    tab_dev = torch.from_numpy(table).to(dev)
    for b, g in groups:
        nb = (int(ctx[b]) + 15) // 16
        blocks = tab_dev[b, :nb].long()
        qsub = bits(q[b:b + 1, :, g * G:(g + 1) * G].contiguous())  # [1, W, G, 128]
        local = np.arange(nb, dtype=np.int32)[None, :]
        if case.kv_fp8:
            ksub = kp[blocks, g].unsqueeze(1).contiguous().cpu().numpy()   # [nb, 1, 16, 128]
            vsub = vp[blocks, g].unsqueeze(1).contiguous().cpu().numpy()
            ref = oracle.gqa_decode_attn_fp8kv(qsub, ksub, vsub, local, ctx[b:b + 1], 1, 1 / math.sqrt(128),
                                               case.k_scale, case.v_scale)
        else:
            ksub = bits(kp[blocks, g].unsqueeze(1).contiguous())
            vsub = bits(vp[blocks, g].unsqueeze(1).contiguous())
            ref = oracle.gqa_decode_attn(qsub, ksub, vsub, local, ctx[b:b + 1], 1, 1 / math.sqrt(128))
        got = f64(out[b:b + 1, :, g * G:(g + 1) * G])
        assert_close(got, ref, what=f"{case.name} b={b} g={g}")


WORKLOADS = {w.__name__: w() for w in configs.ALL}


@pytest.mark.parametrize("case", WORKLOADS["tiny"].gemms, ids=lambda c: c.name)
def test_tiny_gemm(dev, dqd, case):
    check_gemm(dqd, dev, case, WORKLOADS["tiny"].seed)


@pytest.mark.parametrize("case", WORKLOADS["tiny"].attns, ids=lambda c: c.name)
def test_tiny_attn(dev, dqd, case):
    check_attn(dqd, dev, case, WORKLOADS["tiny"].seed)


@pytest.mark.parametrize("case", WORKLOADS["llama3_8b_b1"].gemms, ids=lambda c: c.name)
def test_llama3_8b_gemm(dev, dqd, case):
    check_gemm(dqd, dev, case, WORKLOADS["llama3_8b_b1"].seed, max_oracle_macs=2e8)


@pytest.mark.parametrize("case", WORKLOADS["llama3_8b_b1"].attns, ids=lambda c: c.name)
def test_llama3_8b_attn(dev, dqd, case):
    check_attn(dqd, dev, case, WORKLOADS["llama3_8b_b1"].seed)


@pytest.mark.parametrize("case", WORKLOADS["dense70b_b32"].gemms, ids=lambda c: c.name)
def test_dense70b_gemm(dev, dqd, case):
    check_gemm(dqd, dev, case, WORKLOADS["dense70b_b32"].seed)


@pytest.mark.parametrize("case", WORKLOADS["dense70b_b32"].attns, ids=lambda c: c.name)
def test_dense70b_attn(dev, dqd, case):
    check_attn(dqd, dev, case, WORKLOADS["dense70b_b32"].seed, max_groups=24)


@pytest.mark.parametrize("case", WORKLOADS["verify_8b"].gemms, ids=lambda c: c.name)
def test_verify_gemm(dev, dqd, case):
    check_gemm(dqd, dev, case, WORKLOADS["verify_8b"].seed)


@pytest.mark.parametrize("case", WORKLOADS["verify_8b"].attns, ids=lambda c: c.name)
def test_verify_attn(dev, dqd, case):
    check_attn(dqd, dev, case, WORKLOADS["verify_8b"].seed, max_groups=24)


@pytest.mark.parametrize("case", WORKLOADS["longctx_70b_b8"].gemms, ids=lambda c: c.name)
def test_longctx_gemm(dev, dqd, case):
    check_gemm(dqd, dev, case, WORKLOADS["longctx_70b_b8"].seed)


@pytest.mark.parametrize("case", WORKLOADS["longctx_70b_b8"].attns, ids=lambda c: c.name)
def test_longctx_attn(dev, dqd, case):
    check_attn(dqd, dev, case, WORKLOADS["longctx_70b_b8"].seed, max_groups=3)


@pytest.mark.parametrize("case", WORKLOADS["int4_70b_b32_fp8kv"].gemms, ids=lambda c: c.name)
def test_int4_70b_fp8kv_gemm(dev, dqd, case):
    check_gemm(dqd, dev, case, WORKLOADS["int4_70b_b32_fp8kv"].seed)


@pytest.mark.parametrize("case", WORKLOADS["int4_70b_b32_fp8kv"].attns, ids=lambda c: c.name)
def test_int4_70b_fp8kv_attn(dev, dqd, case):
    check_attn(dqd, dev, case, WORKLOADS["int4_70b_b32_fp8kv"].seed, max_groups=24)


@pytest.mark.parametrize("case", WORKLOADS["longctx_70b_b8_fp8kv"].attns, ids=lambda c: c.name)
def test_longctx_fp8kv_attn(dev, dqd, case):
    check_attn(dqd, dev, case, WORKLOADS["longctx_70b_b8_fp8kv"].seed, max_groups=3)


def check_verify(dqd, dev, case, seed, max_reqs=8):
    """The bench's greedy verify call at full size: the logits are drawn on the
    device, sampled requests are copied back for the oracle."""
    import numpy as np
    logits = synth.normal_bf16(seed, case.name + ".logits", (case.batch, case.width, case.vocab), device=dev)
    draft_np = synth.rng(seed, case.name + ".draft").integers(0, case.vocab, (case.batch, case.width - 1))
    draft_np = draft_np.astype(np.int32)
    # make some drafts right: the first j_r follow the target's own predictions
    t = logits.float().argmax(dim=2).cpu().numpy().astype(np.int32)
    keep = np.random.default_rng(seed).integers(0, case.width, case.batch)
    for r in range(case.batch):
        draft_np[r, :keep[r]] = t[r, :keep[r]]
    ctx = torch.full((case.batch,), 100000, dtype=torch.int32, device=dev)
    out, cnt = dqd.spec_verify_greedy(logits, torch.from_numpy(draft_np).to(dev), ctx)
    reqs = sample_rows(case.batch, max_reqs, seed)
    lg = bits(logits[torch.as_tensor(reqs, device=dev)].contiguous())
    rout, rcnt, rctx = oracle.spec_verify_greedy(lg, draft_np[reqs], np.full(len(reqs), 100000, np.int32))
    assert np.array_equal(cnt.cpu().numpy()[reqs], rcnt)
    assert np.array_equal(ctx.cpu().numpy()[reqs], rctx)
    o = out.cpu().numpy()[reqs]
    k = np.arange(case.width)[None, :] < rcnt[:, None]
    assert np.array_equal(o[k], rout[k])


@pytest.mark.parametrize("case", WORKLOADS["verify_8b"].verifies, ids=lambda c: c.name)
def test_verify_accept(dev, dqd, case):
    check_verify(dqd, dev, case, WORKLOADS["verify_8b"].seed)


def check_rope(dqd, dev, case, seed, max_tokens=16):
    """The bench's RoPE + append call at full size: sampled tokens' rotated q
    and appended k, v against the oracle."""
    import numpy as np
    ctx = np.asarray(case.context, np.int32)
    table, nblk = synth.block_table(seed, case.name + ".table", ctx, True)
    rows = case.batch * case.width
    qkv = synth.normal_bf16(seed, case.name + ".qkv", (rows, (case.hq + 2 * case.hkv) * case.d), device=dev)
    kp = torch.zeros((nblk, case.hkv, 16, case.d), dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    q = dqd.rope_kv_append(qkv, case.batch, case.width, case.hq, case.hkv, kp, vp,
                           torch.from_numpy(table).to(dev), torch.from_numpy(ctx).to(dev), rope_base=case.rope_base)
    toks = sample_rows(rows, max_tokens, seed)
    kr = kp.view(-1, case.d)
    vr = vp.view(-1, case.d)
    for t in toks:
        b, i = divmod(int(t), case.width)
        one = bits(qkv[t:t + 1])
        rq, rk, rv, slot = oracle.rope_kv_append(one, 1, 1, case.hq, case.hkv, case.rope_base,
                                                 ctx[b:b + 1] - (case.width - 1 - i), table[b:b + 1], nblk)
        assert_close(f64(q[b, i]), rq[0, 0], what=f"{case.name} q token {t}")
        for g in range(case.hkv):
            row = int(slot[0, 0]) + 16 * g
            assert_close(f64(kr[row]), rk[0, 0, g], what=f"{case.name} k token {t}")
            assert np.array_equal(bits(vr[row]), one[0, (case.hq + case.hkv + g) * case.d:(case.hq + case.hkv + g + 1) * case.d])


# the standalone RoPE + append at the shapes of the 8B decode and verify steps
ROPE_CASES = [configs.RopeCase("rope_append_32_8", 1, 1, 32, 8, (8192,)),
              configs.RopeCase("rope_append_b64_w16", 64, 16, 32, 8, configs._ctx_uniform(3, 64, 512, 4096))]


@pytest.mark.parametrize("case", ROPE_CASES, ids=lambda c: c.name)
def test_rope_append(dev, dqd, case):
    check_rope(dqd, dev, case, 3)


def check_qkv_rope(dqd, dev, case, seed, max_tokens=12):
    """The bench's fused QKV + RoPE + append call at full size: bit for bit
    equal to the two-call chain (dq_gemm, rope_kv_append) on the same inputs,
    and sampled tokens against the oracle's float64 projection and rotation
    (rotated outputs bounded per pair: the rotation is an isometry)."""
    d, hq, hkv = case.d, case.hq, case.hkv
    n, k, m = (hq + 2 * hkv) * d, case.k, case.batch * case.width
    ctx = np.asarray(case.context, np.int32)
    table, nblk = synth.block_table(seed, case.name + ".table", ctx, True)
    x = synth.normal_bf16(seed, case.name + ".x", (m, k), device=dev)
    if case.wtype == oracle.W_INT4_G128:
        wq = synth.int4_weight(seed, case.name, n, k, device=dev)
        weight = dqd.Weight.int4(dqd.pack_int4_g128(wq.codes, wq.scales, wq.zeros))
        host = (wq.codes.cpu().numpy(), bits(wq.scales), wq.zeros.cpu().numpy())
    else:
        w = synth.normal_bf16(seed, case.name, (n, k), 0.02, device=dev)
        weight = dqd.Weight.bf16(w)
        host = (bits(w), None, None)
    t, c = torch.from_numpy(table).to(dev), torch.from_numpy(ctx).to(dev)
    kp = torch.zeros((nblk, hkv, 16, d), dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    kp2, vp2 = kp.clone(), vp.clone()
    q = dqd.dq_gemm_qkv_rope_append(weight, x, case.batch, case.width, hq, hkv, kp, vp, t, c,
                                    rope_base=case.rope_base)
    q2 = dqd.rope_kv_append(dqd.dq_gemm(weight, x), case.batch, case.width, hq, hkv, kp2, vp2, t, c,
                            rope_base=case.rope_base)
    for a, b_ in ((q, q2), (kp, kp2), (vp, vp2)):
        assert torch.equal(a.view(torch.int16), b_.view(torch.int16)), f"{case.name}: fused differs from the chain"
    toks = sample_rows(m, max_tokens, seed)
    y = oracle.dq_gemm(case.wtype, *host, bits(x[torch.as_tensor(toks, device=dev)])).reshape(len(toks), -1, d)
    kr, vr = kp.view(-1, d), vp.view(-1, d)
    for j, tk in enumerate(toks):
        b, i = divmod(int(tk), case.width)
        pos = float(ctx[b] - case.width + i)
        rq = oracle.rope(y[j, :hq], np.full(hq, pos), case.rope_base)
        rk = oracle.rope(y[j, hq:hq + hkv], np.full(hkv, pos), case.rope_base)
        got_q = f64(q[b, i]).reshape(-1, 2)
        slot = oracle.rope_kv_append(oracle.bf16_round(y[j:j + 1].reshape(1, -1)), 1, 1, hq, hkv,
                                     case.rope_base, ctx[b:b + 1] - (case.width - 1 - i), table[b:b + 1],
                                     nblk)[3][0, 0]
        got_k = np.stack([f64(kr[int(slot) + 16 * g]) for g in range(hkv)])
        got_v = np.stack([f64(vr[int(slot) + 16 * g]) for g in range(hkv)])
        for name, got, ref in (("q", got_q, rq), ("k", got_k, rk)):
            ref = ref.reshape(-1, 2)
            rms = float(np.sqrt(np.mean(ref ** 2)))
            bound = 1e-2 * (np.linalg.norm(ref, axis=1, keepdims=True) + rms)
            assert np.all(np.abs(got.reshape(-1, 2) - ref) <= bound), f"{case.name} {name} token {tk}"
        assert_close(got_v, y[j, hq + hkv:], what=f"{case.name} v token {tk}")


@pytest.mark.parametrize("wl", ["llama3_8b_b1", "verify_8b"])
def test_qkv_rope_append(dev, dqd, wl):
    cases = WORKLOADS[wl].qkv_ropes
    assert cases
    for case in cases:
        check_qkv_rope(dqd, dev, case, WORKLOADS[wl].seed)
