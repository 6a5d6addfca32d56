"""Pins for the per-kernel references of oracle.ops (the functions the GPU
kernel tests compare against), each checked against something other than
itself: exact integer arithmetic, closed forms of softmax and SiLU, and the
special cases of attention that fix its slicing, causality and cache writes.

A transposed operand, a wrong slice of the packed q/k/v row, a sign error in
SiLU, a key visible to an earlier row or a K/V row written at the wrong
position each fails one of these.
"""

import math

import numpy as np
import torch

from oracle import ops as O
from oracle.numerics import bf16_round


def _bits(vals) -> np.ndarray:
    """bf16 bit patterns of values that bf16 represents exactly."""
    t = torch.tensor(np.asarray(vals, dtype=np.float32)).to(torch.bfloat16)
    assert torch.equal(t.to(torch.float32), torch.tensor(np.asarray(vals, dtype=np.float32)))
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def test_linear_is_the_exact_integer_product():
    rng = np.random.default_rng(0)
    R, K, M = 16, 48, 5
    W = rng.integers(-4, 5, size=(R, K))
    act = rng.integers(-3, 4, size=(M, K))
    got = O.linear(_bits(W), act.astype(np.float64))
    # brute force with Python integers
    for m in range(M):
        for r in range(R):
            assert got[m, r] == sum(int(W[r, k]) * int(act[m, k]) for k in range(K))


def test_silu_product_closed_forms():
    # gate rows pick one activation each, up rows pick another: u = bf16(silu(a_i) a_j)
    xs = [0.0, 1.0, -1.0, 2.0, -2.0, 8.0, -8.0, 0.5]
    K = len(xs)
    Wg = np.eye(K)
    Wu = np.roll(np.eye(K), 1, axis=1)          # up row i picks a_{i+1}
    act = np.array([xs], dtype=np.float64)
    u = O.silu_product(_bits(Wg), _bits(Wu), act)[0]
    for i, x in enumerate(xs):
        y = xs[(i + 1) % K]
        exact = x / (1.0 + math.exp(-x)) * y
        assert abs(u[i] - exact) <= 2.0 ** -8 * abs(exact) + 1e-300, (x, y, u[i], exact)
    # silu(x) - silu(-x) = x: with up picking a constant 1
    Wu1 = np.zeros((2, 2))
    Wu1[:, 1] = 1.0
    for x in (0.25, 1.5, 3.0):
        act2 = np.array([[x, 1.0], [-x, 1.0]])
        Wg1 = np.array([[1.0, 0.0], [1.0, 0.0]])
        a = O.silu_product(_bits(Wg1), _bits(Wu1), act2)[:, 0]
        assert abs((a[0] - a[1]) - x) <= 2.0 ** -7 * (abs(a[0]) + abs(a[1]))
    # silu(0) = 0 exactly; large arguments approach the identity
    z = O.silu_product(_bits(np.eye(2)), _bits(np.eye(2)), np.array([[0.0, 64.0]]))[0]
    assert z[0] == 0.0 and z[1] == 64.0 * 64.0


def test_rmsnorm_linear_of_a_constant_row():
    # rmsnorm(c, g) = sign(c) g (up to eps); identity weights return bf16 of it
    K = 32
    g = np.linspace(0.5, 2.0, K)
    for c in (3.0, -0.25):
        y = O.rmsnorm_linear(_bits(np.eye(K)), np.full((1, K), c), g, 1e-5)[0]
        want = bf16_round(np.sign(c) * g / math.sqrt(1.0 + 1e-5 / c ** 2))
        np.testing.assert_array_equal(y, want)


def test_row_summary_closed_form():
    z = np.array([0.0, math.log(3.0), -1e9])
    s = O.row_summary(z)
    assert s["top1"] == 1 and s["top2"] == 0
    assert abs(s["conf"] - 0.75) < 1e-12
    assert abs(s["lse"] - math.log(4.0)) < 1e-12
    assert abs(s["gap"] - math.log(3.0)) < 1e-12


def _qkv_row(q, k, v):
    return np.concatenate([q.ravel(), k.ravel(), v.ravel()])


def test_attention_single_key_returns_its_value():
    H, Hkv, dh, max_seq = 4, 2, 8, 4
    rng = np.random.default_rng(1)
    q = rng.standard_normal((H, dh))
    k = rng.standard_normal((Hkv, dh))
    v = rng.standard_normal((Hkv, dh))
    K0 = np.zeros((Hkv, max_seq, dh))
    out, K1, V1 = O.attention(_qkv_row(q, k, v)[None], 0, K0, K0.copy(), H, Hkv, dh, 10000.0)
    # one visible key: every head returns its KV head's value, rounded to bf16
    for h in range(H):
        np.testing.assert_array_equal(out[0, h * dh:(h + 1) * dh], bf16_round(v[h // (H // Hkv)]))
    # position 0: RoPE is the identity, the cache row holds bf16(k), bf16(v)
    np.testing.assert_array_equal(K1[:, 0], bf16_round(k))
    np.testing.assert_array_equal(V1[:, 0], bf16_round(v))
    assert not np.any(K1[:, 1:]) and not np.any(V1[:, 1:])


def test_attention_is_causal_and_uniform_for_a_zero_query():
    # two rows at positions 0 and 1 with zero queries: row 0 sees only key 0,
    # row 1 averages values 0 and 1 with equal weights
    H = Hkv = 2
    dh, max_seq = 8, 4
    rng = np.random.default_rng(2)
    q = np.zeros((H, dh))
    rows = []
    vs = []
    for _ in range(2):
        k = rng.standard_normal((Hkv, dh))
        v = rng.standard_normal((Hkv, dh))
        vs.append(bf16_round(v))
        rows.append(_qkv_row(q, k, v))
    K0 = np.zeros((Hkv, max_seq, dh))
    out, K1, _ = O.attention(np.stack(rows), 0, K0, K0.copy(), H, Hkv, dh, 10000.0)
    for h in range(H):
        np.testing.assert_array_equal(out[0, h * dh:(h + 1) * dh], vs[0][h])
        np.testing.assert_allclose(out[1, h * dh:(h + 1) * dh],
                                   bf16_round(0.5 * (vs[0][h] + vs[1][h])), rtol=0, atol=0)
    # position 1's key is stored rotated: same norm per rotated pair, not the raw key
    k1 = rows[1][H * dh:(H + Hkv) * dh].reshape(Hkv, dh)
    half = dh // 2
    for kv in range(Hkv):
        a, b = K1[kv, 1, :half], K1[kv, 1, half:]
        ra, rb = k1[kv, :half], k1[kv, half:]
        np.testing.assert_allclose(a * a + b * b, ra * ra + rb * rb, rtol=2e-2)
        assert not np.allclose(K1[kv, 1], bf16_round(k1[kv]))
