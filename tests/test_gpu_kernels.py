"""GPU parity of each hot-path kernel against the CPU oracle, through the C-ABI.

Inputs are seeded and synthetic; both sides consume the same bf16 bits.
Tolerances: the GPU accumulates in fp32 and the oracle in fp64, so GEMV
outputs agree to ~1e-6 relative; bf16-rounded outputs (attention, SwiGLU)
may differ by one bf16 unit where the two land on different sides of a
rounding boundary.  Column invariance (a row's bits do not depend on how
many rows are processed together) is checked bit for bit.
"""

import numpy as np
import pytest
import torch

from tests.gpu_util import rand_bf16, rand_f32, bf16_values, pack_reference

pytestmark = pytest.mark.gpu

MS = [1, 2, 7, 8, 9, 13, 16]


@pytest.fixture(scope="module")
def ops():
    import __graft_entry__ as g
    g.build()
    import self_speculative_decoding_gb300 as ssd
    return ssd.ops


def P(W):
    """Weights in the library's packed layout."""
    import self_speculative_decoding_gb300 as ssd
    return ssd.pack_weight(W)


@pytest.mark.parametrize("R,K", [(16, 32), (48, 704), (4096, 11008)])
def test_pack_layout(ops, R, K):
    W, Wb = rand_bf16((R, K), seed=R + K)
    got = P(W).cpu().view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, pack_reference(Wb))


def _bf16_close(got, ref, rel=1.0 / 64):
    """Equal up to one bf16 rounding step (plus fp32-vs-fp64 noise)."""
    scale = np.maximum(np.abs(ref), 1e-3)
    return np.max(np.abs(got - ref) / scale) <= rel


# ---------------------------------------------------------------- GEMV family

@pytest.mark.parametrize("R,K", [(64, 256), (48, 704), (256, 1024), (1024, 4096), (4096, 11008)])
@pytest.mark.parametrize("M", MS)
def test_linear_matches_oracle(ops, R, K, M):
    from oracle import ops as O
    W, Wb = rand_bf16((R, K), seed=R * 7 + K)
    act, actb = rand_bf16((M, K), seed=M + 1000, std=1.0)
    y = ops.linear(P(W), act).cpu().numpy()
    ref = O.linear(Wb, bf16_values(act))
    np.testing.assert_allclose(y, ref, rtol=1e-4, atol=1e-4 * np.sqrt(K) * 0.02)


@pytest.mark.parametrize("R,K", [(48, 704), (1024, 4096), (4096, 11008)])
def test_linear_column_invariance(ops, R, K):
    W, _ = rand_bf16((R, K), seed=3)
    W = P(W)
    act, _ = rand_bf16((16, K), seed=4, std=1.0)
    full = ops.linear(W, act)
    for M in (1, 5, 8, 9, 13):
        part = ops.linear(W, act[:M].contiguous())
        assert torch.equal(part, full[:M])
    for j in (0, 7, 8, 15):
        one = ops.linear(W, act[j:j + 1].contiguous())
        assert torch.equal(one[0], full[j])


@pytest.mark.parametrize("R,K", [(768, 256), (12288, 4096)])
@pytest.mark.parametrize("M", [1, 9, 16])
def test_rmsnorm_linear_matches_oracle(ops, R, K, M):
    from oracle import ops as O
    W, Wb = rand_bf16((R, K), seed=11)
    W = P(W)
    x, xd = rand_f32((M, K), seed=12, std=2.0)
    g, gd = rand_f32((K,), seed=13, std=0.1, mean=1.0)
    y = ops.rmsnorm_linear(W, x, g, 1e-5).cpu().numpy()
    ref = O.rmsnorm_linear(Wb, xd, gd, 1e-5)
    # a bf16 rounding flip of one input element moves y by ~ |W| * 2^-8 |h|
    assert np.max(np.abs(y - ref)) < 5e-3
    assert np.mean(np.abs(y - ref)) < 5e-5
    full = ops.rmsnorm_linear(W, x, g, 1e-5)
    one = ops.rmsnorm_linear(W, x[M - 1:M].contiguous(), g, 1e-5)
    assert torch.equal(one[0], full[M - 1])


@pytest.mark.parametrize("R,K", [(256, 704), (4096, 11008)])
@pytest.mark.parametrize("M", [1, 13])
def test_residual_linear_matches_oracle(ops, R, K, M):
    from oracle import ops as O
    W, Wb = rand_bf16((R, K), seed=21)
    act, _ = rand_bf16((M, K), seed=22, std=1.0)
    x, xd = rand_f32((M, R), seed=23)
    out = ops.residual_linear(P(W), act, x.clone()).cpu().numpy()
    ref = xd + O.linear(Wb, bf16_values(act))
    np.testing.assert_allclose(out, ref, rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("F,K", [(704, 256), (11008, 4096)])
@pytest.mark.parametrize("M", [1, 13])
def test_swiglu_matches_oracle(ops, F, K, M):
    from oracle import ops as O
    Wg, Wgb = rand_bf16((F, K), seed=31)
    Wu, Wub = rand_bf16((F, K), seed=32)
    Wg, Wu = P(Wg), P(Wu)
    x, xd = rand_f32((M, K), seed=33)
    g, gd = rand_f32((K,), seed=34, std=0.1, mean=1.0)
    u = bf16_values(ops.swiglu(Wg, Wu, x, g, 1e-5))
    ref = O.swiglu(Wgb, Wub, xd, gd, 1e-5)
    diff = np.abs(u - ref)
    assert np.mean(diff > 0) < 0.02                       # almost all bit-equal
    assert _bf16_close(u, ref, rel=1.0 / 32)
    one = ops.swiglu(Wg, Wu, x[:1].contiguous(), g, 1e-5)
    full = ops.swiglu(Wg, Wu, x, g, 1e-5)
    assert torch.equal(one[0], full[0])


# ---------------------------------------------------------------- attention

def _attn_case(H, Hkv, dh, pos0, M, max_seq, seed):
    rng = np.random.default_rng(seed)
    kc0 = torch.from_numpy(rng.standard_normal((Hkv, max_seq, dh)).astype(np.float32)).to(torch.bfloat16)
    vc0 = torch.from_numpy(rng.standard_normal((Hkv, max_seq, dh)).astype(np.float32)).to(torch.bfloat16)
    qkv, qkvd = rand_f32((M, (H + 2 * Hkv) * dh), seed=seed + 1, std=1.0)
    return kc0, vc0, qkv, qkvd


@pytest.mark.parametrize("H,Hkv,dh", [(4, 4, 64), (32, 32, 128), (16, 2, 128), (64, 8, 128)])
@pytest.mark.parametrize("pos0,M", [(0, 1), (5, 1), (60, 8), (63, 13), (200, 16), (700, 1),
                                    (1000, 13)])
def test_attention_matches_oracle(ops, H, Hkv, dh, pos0, M):
    from oracle import ops as O
    max_seq = 1024 + 64
    kc0, vc0, qkv, qkvd = _attn_case(H, Hkv, dh, pos0, M, max_seq, seed=pos0 * 31 + M)
    kc, vc = kc0.cuda(), vc0.cuda()
    out = bf16_values(ops.attention(qkv, pos0, kc, vc, H, Hkv, dh, 1e4))
    ref, Kr, Vr = O.attention(qkvd, pos0, kc0.to(torch.float64).numpy(),
                              vc0.to(torch.float64).numpy(), H, Hkv, dh, 1e4)
    # appended K/V: bf16 of the same rotated value, at most one rounding step apart
    kg = bf16_values(kc)[:, pos0:pos0 + M]
    vg = bf16_values(vc)[:, pos0:pos0 + M]
    np.testing.assert_array_equal(vg, Vr[:, pos0:pos0 + M])
    assert _bf16_close(kg, Kr[:, pos0:pos0 + M], rel=1.0 / 128)
    # untouched cache stays untouched
    assert torch.equal(kc[:, :pos0].cpu(), kc0[:, :pos0])
    # Outputs are bf16 on both sides and almost all bit-equal.  The rest
    # differ because ~0.1% of the stored K values are one bf16 step apart
    # (RoPE in fp32 on the GPU vs fp64 in the oracle), which moves a score by
    # ~2^-9 |q_i k_i| and an output by a few bf16 steps at most.
    assert np.mean(out != ref) < 0.02
    assert _bf16_close(out, ref, rel=1.0 / 32)
    assert np.mean(np.abs(out - ref)) < 1e-4


@pytest.mark.parametrize("H,Hkv,dh", [(32, 32, 128), (64, 8, 128), (4, 4, 64)])
def test_attention_row_invariance(ops, H, Hkv, dh):
    # M rows at once == the same rows one at a time (cache and outputs bitwise)
    pos0, M, max_seq = 121, 13, 256
    kc0, vc0, qkv, _ = _attn_case(H, Hkv, dh, pos0, M, max_seq, seed=5)
    ka, va = kc0.cuda(), vc0.cuda()
    full = ops.attention(qkv, pos0, ka, va, H, Hkv, dh, 1e4)
    kb, vb = kc0.cuda(), vc0.cuda()
    rows = [ops.attention(qkv[m:m + 1].contiguous(), pos0 + m, kb, vb, H, Hkv, dh, 1e4)
            for m in range(M)]
    assert torch.equal(torch.cat(rows), full)
    assert torch.equal(ka, kb) and torch.equal(va, vb)


# ---------------------------------------------------------------- LM head

@pytest.mark.parametrize("V,D", [(1024, 256), (32000, 4096)])
@pytest.mark.parametrize("M", [1, 13])
@pytest.mark.parametrize("T", [0.0, 0.6])
def test_lm_head_summary_matches_oracle(ops, V, D, M, T):
    from oracle import ops as O
    import self_speculative_decoding_gb300 as ssd
    W, Wb = rand_bf16((V, D), seed=41, std=0.02 * 10)
    W = P(W)
    x, xd = rand_f32((M, D), seed=42)
    g, gd = rand_f32((D,), seed=43, std=0.1, mean=1.0)
    seed, rnd, pos0 = 1234, 3, 77
    logits, stats = ops.lm_head(W, x, g, 1e-5, temperature=T, seed=seed, round=rnd, stream_id=0,
                                pos0=pos0)
    z = logits.cpu().numpy().astype(np.float64)
    ref_z = O.lm_head(Wb, xd, gd, 1e-5)
    assert np.max(np.abs(z - ref_z)) <= 5e-2
    rs = ssd.row_stats(stats)
    checked = 0
    for m in range(M):
        ref = O.row_summary(ref_z[m], T, seed, pos0 + m + 1, rnd, 0)
        assert abs(rs[m]["conf"] - ref["conf"]) <= 1e-3
        assert abs(rs[m]["lse"] - ref["lse"]) <= 5e-2
        if ref["gap"] > 0.1:
            assert rs[m]["top1"] == ref["top1"]
            checked += 1
        # the summary is consistent with the GPU's own logits
        assert rs[m]["top1"] == int(np.argmax(z[m]))
        if T > 0:
            assert abs(rs[m]["lse_t"] - ref["lse_t"]) <= 5e-2
            from oracle.philox import uniforms
            gum = -np.log(-np.log(uniforms(seed, pos0 + m + 1, rnd, 0, V)))
            sc = ref_z[m] / T + gum
            srt = np.sort(sc)
            if srt[-1] - srt[-2] > 0.1:
                assert rs[m]["sample"] == ref["sample"]
    assert checked >= 1
    # row invariance of the summary
    _, s1 = ops.lm_head(W, x[M - 1:M].contiguous(), g, 1e-5, temperature=T, seed=seed, round=rnd,
                        stream_id=0, pos0=pos0 + M - 1)
    assert torch.equal(s1[0], stats[M - 1])


# ---------------------------------------------------------------- RNG / accept

def test_philox_matches_oracle(ops):
    from oracle.philox import philox4x32_10
    rng = np.random.default_rng(9)
    ctr = rng.integers(0, 2 ** 32, size=(4096, 4), dtype=np.uint64).astype(np.uint32)
    key = 0x0123456789ABCDEF
    out = ops.philox(torch.from_numpy(ctr.view(np.int32)).cuda(), key).cpu().numpy().view(np.uint32)
    ref = philox4x32_10(tuple(ctr[:, i].astype(np.uint64) for i in range(4)),
                        (key & 0xFFFFFFFF, key >> 32))
    np.testing.assert_array_equal(out, np.stack([r.astype(np.uint32) for r in ref], axis=1))


@pytest.mark.parametrize("case", range(12))
def test_stochastic_accept_matches_oracle(ops, case):
    from oracle import ops as O
    rng = np.random.default_rng(100 + case)
    V, d, T, seed = 2000, 1 + case % 6, 0.6, 1234 + case
    base = rng.standard_normal(V) * 3
    P = np.stack([base + rng.standard_normal(V) * 0.5 for _ in range(d + 1)]).astype(np.float32)
    Q = np.stack([base + rng.standard_normal(V) * 0.5 for _ in range(d)]).astype(np.float32)
    drafts = [int(np.argmax(Q[j] + rng.gumbel(size=V))) for j in range(d)]
    n, rnd = 500 + case, 7
    em, nem = ops.accept_stochastic(torch.from_numpy(P).cuda(), torch.from_numpy(Q).cuda(),
                                    torch.tensor(drafts, dtype=torch.int32).cuda(), T, seed, rnd, n)
    got = em.cpu().numpy()[: int(nem.item())].tolist()
    a, ref = O.accept_stochastic(P.astype(np.float64), Q.astype(np.float64), drafts, T, seed, rnd, n)
    margins = O.accept_margins(P.astype(np.float64), Q.astype(np.float64), drafts, T, seed, rnd, n)
    # compare decisions up to the first near-boundary one
    k = 0
    while k < min(len(margins), a + 1) and margins[k] > 0.05:
        k += 1
    assert got[:min(k, a)] == ref[:min(k, a)]
    if k > a:   # every decision up to the emitted correction was clear-cut
        assert len(got) == len(ref)
        if O.resample_gap(P.astype(np.float64), Q.astype(np.float64), a, T, seed, rnd, n) > 0.1:
            assert got[-1] == ref[-1]
