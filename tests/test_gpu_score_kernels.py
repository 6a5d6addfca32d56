"""GPU parity of the batched candidate-mask scoring kernels (SWIFT §4.1.2)
through the C-ABI (ssd_op_linear_rows, ssd_op_score_attention).

* The many-row projection equals the plain product W act (fp64 oracle on the
  same bf16 bits) for every epilogue: store, residual add through a row map
  (rows not named stay bit-identical), SwiGLU (one bf16 step), argmax
  (exact wherever the top-2 gap exceeds 1e-3).  Sizes span several row and
  output tiles with ragged tails.
* A row's result does not depend on how many rows are processed together
  (bit for bit), across token-tile widths from 16 to 256 columns.
* The window attention equals oracle.ops.score_attention within bf16
  rounding of its operands (P and the output are bf16), on both forms: the
  tensor-core one (dh 128, windows of a multiple of 8 rows) and the
  mma.sync one (the other shapes).
"""

import numpy as np
import pytest
import torch

from tests.gpu_util import rand_bf16, rand_f32, bf16_values

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    import __graft_entry__ as g
    g.build()
    import self_speculative_decoding_gb300 as ssd
    return ssd.ops


def P(W):
    import self_speculative_decoding_gb300 as ssd
    return ssd.pack_weight(W)


SHAPES = [(16, 32, 1), (272, 96, 37), (64, 1024, 128), (528, 704, 300), (1024, 4096, 513)]


@pytest.mark.parametrize("R,K,T", SHAPES)
def test_rows_store(ops, R, K, T):
    from oracle import ops as O
    W, Wb = rand_bf16((R, K), seed=R + K)
    act, _ = rand_bf16((T, K), seed=T, std=1.0)
    y = ops.linear_rows(P(W), act).cpu().numpy()
    ref = O.linear(Wb, bf16_values(act))
    np.testing.assert_allclose(y, ref, rtol=1e-4, atol=2e-6 * np.sqrt(K))


@pytest.mark.parametrize("R,K,T", SHAPES[1:])
def test_rows_residual_through_map(ops, R, K, T):
    from oracle import ops as O
    W, Wb = rand_bf16((R, K), seed=5)
    act, _ = rand_bf16((T, K), seed=6, std=1.0)
    rows = 2 * T + 3
    x0, x0n = rand_f32((rows, R), seed=7)
    rng = np.random.default_rng(8)
    rmap = np.sort(rng.choice(rows, size=T, replace=False)).astype(np.int32)
    x = x0.clone()
    ops.linear_rows(P(W), act, epi="resid", out=x, rowmap=torch.from_numpy(rmap).cuda())
    got = x.cpu().numpy()
    ref = x0n.copy()
    ref[rmap] += O.linear(Wb, bf16_values(act))
    np.testing.assert_allclose(got[rmap], ref[rmap], rtol=1e-4, atol=1e-5 * np.sqrt(K))
    others = np.setdiff1d(np.arange(rows), rmap)
    np.testing.assert_array_equal(got[others], x0.cpu().numpy()[others])


@pytest.mark.parametrize("F,K,T", [(48, 64, 5), (704, 256, 130), (1376, 512, 257)])
def test_rows_swiglu(ops, F, K, T):
    from oracle import ops as O
    Wg, Wgb = rand_bf16((F, K), seed=1)
    Wu, Wub = rand_bf16((F, K), seed=2)
    act, _ = rand_bf16((T, K), seed=3, std=1.0)
    u = ops.linear_rows(P(Wg), act, epi="swiglu", W1=P(Wu))
    got = bf16_values(u)
    ref = O.silu_product(Wgb, Wub, bf16_values(act))
    scale = np.maximum(np.abs(ref), 1e-4)
    assert np.max(np.abs(got - ref) / scale) <= 1.0 / 64


@pytest.mark.parametrize("V,K,T", [(1024, 256, 33), (4000, 512, 160)])
def test_rows_argmax(ops, V, K, T):
    from oracle import ops as O
    W, Wb = rand_bf16((V, K), seed=9)
    act, _ = rand_bf16((T, K), seed=10, std=1.0)
    idx = ops.linear_rows(P(W), act, epi="argmax").cpu().numpy()
    z = O.linear(Wb, bf16_values(act))
    for t in range(T):
        s = np.sort(z[t])
        if s[-1] - s[-2] > 1e-3:
            assert idx[t] == int(np.argmax(z[t])), t
        else:
            assert z[t][idx[t]] >= s[-1] - 1e-3


# The 13B scoring projections at the launch shape of a layer that 9 of the 16
# candidates keep (288 window rows): qkv 15360 x 5120 (store), o_proj
# 5120 x 5120 and down 5120 x 13824 (residual through a row map).  The oracle
# computes a seeded sample of 96 output features against every window row.
T13 = 288


def _sample(n, k, seed):
    return np.sort(np.random.default_rng(seed).choice(n, size=k, replace=False))


@pytest.mark.parametrize("epi,R,K", [("store", 15360, 5120), ("resid", 5120, 5120),
                                     ("resid", 5120, 13824)])
def test_rows_13b_shapes_sampled(ops, epi, R, K):
    from oracle import ops as O
    W, Wb = rand_bf16((R, K), seed=R + 3 * K)
    act, _ = rand_bf16((T13, K), seed=31, std=1.0)
    feats = _sample(R, 96, R + K)
    ref = O.linear(Wb[feats], bf16_values(act))           # [T13, 96]
    if epi == "store":
        y = ops.linear_rows(P(W), act).cpu().numpy()
        np.testing.assert_allclose(y[:, feats], ref, rtol=1e-4, atol=2e-6 * np.sqrt(K))
        return
    rows = 2 * T13 + 3
    x0, x0n = rand_f32((rows, R), seed=32)
    rmap = _sample(rows, T13, 33).astype(np.int32)
    x = x0.clone()
    ops.linear_rows(P(W), act, epi="resid", out=x, rowmap=torch.from_numpy(rmap).cuda())
    got = x.cpu().numpy()
    want = x0n[rmap][:, feats] + ref
    np.testing.assert_allclose(got[rmap][:, feats], want, rtol=1e-4, atol=1e-5 * np.sqrt(K))
    others = np.setdiff1d(np.arange(rows), rmap)
    np.testing.assert_array_equal(got[others], x0.cpu().numpy()[others])


@pytest.mark.parametrize("R,K", [(528, 704), (1600, 512), (16384, 256)])
def test_rows_count_invariance(ops, R, K):
    # token tiles of different widths (16 .. 256 columns) for different T; the
    # number of accumulators depends on the matrix only
    W, _ = rand_bf16((R, K), seed=11)
    Wp = P(W)
    act, _ = rand_bf16((513, K), seed=12, std=1.0)
    full = ops.linear_rows(Wp, act)
    for T in (1, 17, 128, 129, 257, 300):
        part = ops.linear_rows(Wp, act[:T].contiguous())
        assert torch.equal(part, full[:T]), T
    one = ops.linear_rows(Wp, act[200:201].contiguous())
    assert torch.equal(one[0], full[200])


@pytest.mark.parametrize("H,Hkv,dh,N,split,cand", [
    (4, 2, 64, 8, 20, [0, 2]),
    (2, 2, 128, 33, 70, [1]),
    (8, 1, 64, 70, 130, [3, 0, 2]),
    (4, 4, 128, 32, 2040, [0, 1, 2, 3]),
    # tensor-core form (dh 128, N a multiple of 8): several candidate groups,
    # candidates out of order, a partial last prefix block, a prefix shorter
    # than one block, GQA
    (8, 8, 128, 32, 300, [5, 1, 3, 0, 2, 7, 9, 8, 4]),
    (4, 2, 128, 16, 100, [2, 0, 3, 1, 4, 5, 7, 6, 8, 9, 10, 11, 12, 13, 14, 15]),
    (8, 2, 128, 64, 129, [1, 0, 2, 3]),
    (4, 1, 128, 8, 1, list(range(31, -1, -1))),
])
def test_score_attention(ops, H, Hkv, dh, N, split, cand):
    from oracle import ops as O
    max_seq = ((split + 63) // 64) * 64 + 64
    nk = max(cand) + 1
    Kc, _ = rand_bf16((Hkv, max_seq, dh), seed=1, std=1.0)
    Vc, _ = rand_bf16((Hkv, max_seq, dh), seed=2, std=1.0)
    WK, _ = rand_bf16((nk * N, Hkv, dh), seed=3, std=1.0)
    WV, _ = rand_bf16((nk * N, Hkv, dh), seed=4, std=1.0)
    q, _ = rand_bf16((len(cand) * N, H, dh), seed=5, std=0.3)
    cd = torch.tensor(cand, dtype=torch.int32, device="cuda")
    out = ops.score_attention(q, cd, N, split, Kc, Vc, WK, WV, H, Hkv, dh)
    got = bf16_values(out)
    ref = O.score_attention(bf16_values(q), cand, N, split, bf16_values(Kc), bf16_values(Vc),
                            bf16_values(WK), bf16_values(WV), H, Hkv)
    assert np.max(np.abs(got - ref)) <= 2e-2, np.max(np.abs(got - ref))
