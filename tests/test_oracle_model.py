"""Pins for the oracle's decoder forward.

The independent check is a second formulation of the same decoder built
from library routines (torch.nn.functional.rms_norm, scaled_dot_product_attention
with a causal mask, silu; RoPE as multiplication by unit complex numbers via
torch.polar) over whole sequences at once, in float64.  A dropped term, a
wrong sign in the rotation, a transposed projection or an off-by-one in the
causal mask in either formulation makes them disagree.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from synthetic import TINY, make_weights, weights_to_numpy, make_prompt, shrink
from oracle.model import OracleModel, softmax
from oracle.numerics import widen


def _torch_reference_logits(shape, wn, tokens, bf16):
    """Whole-sequence forward with torch library ops (fp64)."""
    def rnd(t):
        return t.to(torch.bfloat16).to(torch.float64) if bf16 else t

    def W(a):
        return torch.from_numpy(widen(a))

    H, Hkv, dh, D = shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.d_model
    T = len(tokens)
    x = W(wn["tok_embed"])[torch.as_tensor(tokens, dtype=torch.long)]
    i = torch.arange(dh // 2, dtype=torch.float64)
    inv = shape.rope_theta ** (-2.0 * i / dh)
    ang = torch.arange(T, dtype=torch.float64)[:, None] * inv[None, :]
    rot = torch.polar(torch.ones_like(ang), ang)            # [T, dh/2]

    def rope(v):                                             # v [T, heads, dh]
        c = torch.complex(v[..., : dh // 2], v[..., dh // 2:]) * rot[:, None, :]
        return torch.cat([c.real, c.imag], dim=-1)

    for lw in wn["layers"]:
        h = rnd(F.rms_norm(x, (D,), W(lw["attn_norm"]), eps=shape.norm_eps))
        qkv = h @ W(lw["wqkv"]).T
        q = rope(qkv[:, : H * dh].reshape(T, H, dh))
        k = rnd(rope(qkv[:, H * dh:(H + Hkv) * dh].reshape(T, Hkv, dh)))
        v = rnd(qkv[:, (H + Hkv) * dh:].reshape(T, Hkv, dh))
        rep = H // Hkv
        k = k.repeat_interleave(rep, dim=1)
        v = v.repeat_interleave(rep, dim=1)
        a = F.scaled_dot_product_attention(q.transpose(0, 1)[None], k.transpose(0, 1)[None],
                                           v.transpose(0, 1)[None], is_causal=True)
        a = rnd(a[0].transpose(0, 1).reshape(T, H * dh))
        x = x + a @ W(lw["wo"]).T
        h2 = rnd(F.rms_norm(x, (D,), W(lw["mlp_norm"]), eps=shape.norm_eps))
        u = rnd(F.silu(h2 @ W(lw["w_gate"]).T) * (h2 @ W(lw["w_up"]).T))
        x = x + u @ W(lw["w_down"]).T
    hf = rnd(F.rms_norm(x, (D,), W(wn["final_norm"]), eps=shape.norm_eps))
    return (hf @ W(wn["lm_head"]).T).numpy()


def _oracle_logits(model, tokens):
    kv = model.new_cache(len(tokens) + 4)
    X = model.embed_rows(tokens)
    X = model.run_layers(X, range(len(tokens)), kv, range(model.s.n_layers))
    return model.lm_head(X)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("gqa", [False, True])
def test_forward_matches_library_formulation(dtype, gqa):
    w = TINY if not gqa else shrink(TINY, n_heads=8, n_kv_heads=2, head_dim=32)
    wn = weights_to_numpy(make_weights(w, dtype=dtype, random_gains=True))
    model = OracleModel(w.shape, wn)
    toks = make_prompt(w, 12)
    got = _oracle_logits(model, toks)
    ref = _torch_reference_logits(w.shape, wn, toks, dtype == "bf16")
    if dtype == "fp32":
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-10)
    else:
        # bf16 rounding points may land on different sides of a rounding
        # boundary when the two formulations differ in the last fp64 bits.
        assert np.max(np.abs(got - ref)) < 2e-3
        assert np.mean(np.abs(got - ref)) < 1e-5


def test_rmsnorm_of_constant_vector():
    model = OracleModel(TINY.shape, weights_to_numpy(make_weights(TINY)))
    g = np.linspace(0.5, 1.5, 256)
    for c in (1e-3, 0.7, -3.0):
        got = model.rmsnorm(np.full(256, c), g)
        np.testing.assert_allclose(got, c / np.sqrt(c * c + TINY.shape.norm_eps) * g, rtol=1e-14)


def test_rope_identity_at_zero_and_relative_property():
    model = OracleModel(TINY.shape, weights_to_numpy(make_weights(TINY)))
    rng = np.random.default_rng(0)
    q = rng.standard_normal((3, 64))
    k = rng.standard_normal((3, 64))
    np.testing.assert_array_equal(model.rope(q, 0), q)
    # norms of each rotated pair are preserved
    r = model.rope(q, 37)
    np.testing.assert_allclose(r[:, :32] ** 2 + r[:, 32:] ** 2, q[:, :32] ** 2 + q[:, 32:] ** 2,
                               rtol=1e-12)
    # the score depends only on the position difference
    s1 = np.sum(model.rope(q, 5) * model.rope(k, 2), axis=1)
    s2 = np.sum(model.rope(q, 105) * model.rope(k, 102), axis=1)
    np.testing.assert_allclose(s1, s2, rtol=1e-9)


def test_attention_single_key_returns_value():
    w = TINY
    model = OracleModel(w.shape, weights_to_numpy(make_weights(w)))
    kv = model.new_cache(4)
    rng = np.random.default_rng(3)
    kv.K[0][:, 0] = rng.standard_normal((4, 64))
    kv.V[0][:, 0] = rng.standard_normal((4, 64))
    q = rng.standard_normal((4, 64)) * 10
    out = model.attention_row(q, kv, 0, 0)
    np.testing.assert_array_equal(out, kv.V[0][:, 0].reshape(-1))


def test_attention_matches_scipy_softmax():
    from scipy.special import softmax as sp_softmax
    w = shrink(TINY, n_heads=4, n_kv_heads=2)
    model = OracleModel(w.shape, weights_to_numpy(make_weights(w)))
    kv = model.new_cache(16)
    rng = np.random.default_rng(4)
    for l in range(1):
        kv.K[l][:] = rng.standard_normal(kv.K[l].shape)
        kv.V[l][:] = rng.standard_normal(kv.V[l].shape)
    q = rng.standard_normal((4, 64))
    pos = 9
    out = model.attention_row(q, kv, 0, pos).reshape(4, 64)
    for h in range(4):
        K = kv.K[0][h // 2, : pos + 1]
        V = kv.V[0][h // 2, : pos + 1]
        p = sp_softmax(K @ q[h] / 8.0)
        np.testing.assert_allclose(out[h], p @ V, rtol=1e-12, atol=1e-14)


def test_rows_are_independent_of_batching():
    # batched rows give bit-identical results to one row at a time
    w = TINY
    wn = weights_to_numpy(make_weights(w, dtype="bf16", random_gains=True))
    model = OracleModel(w.shape, wn)
    toks = make_prompt(w, 10)
    full = _oracle_logits(model, toks)
    kv = model.new_cache(16)
    rows = []
    for p, t in enumerate(toks):
        X = model.run_layers(model.embed_rows([t]), [p], kv, range(4))
        rows.append(model.lm_head(X)[0])
    np.testing.assert_array_equal(np.stack(rows), full)


def test_causality():
    w = TINY
    model = OracleModel(w.shape, weights_to_numpy(make_weights(w)))
    toks = make_prompt(w, 10)
    a = _oracle_logits(model, toks)
    toks2 = toks.copy()
    toks2[7] = (toks2[7] + 1) % w.shape.vocab
    b = _oracle_logits(model, toks2)
    np.testing.assert_array_equal(a[:7], b[:7])
    assert np.max(np.abs(a[7:] - b[7:])) > 0


def test_softmax_helper():
    z = np.array([1.0, 2.0, 3.0, -np.inf])
    p = softmax(z)
    e = np.exp([1.0, 2.0, 3.0])
    np.testing.assert_allclose(p[:3], e / e.sum(), rtol=1e-15)
    assert p[3] == 0.0
