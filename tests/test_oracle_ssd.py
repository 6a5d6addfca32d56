"""Pins for the oracle's draft / verify / accept loop.

What the pages fix and these tests check:
* greedy self-speculative output equals greedy autoregressive output token
  for token (lossless: SWIFT §1 and §6, LayerSkip blog §3);
* the KV the verify reuses equals a fresh full-model recompute (LayerSkip
  blog §3.2);
* each verify yields between 1 and d+1 tokens (LayerSkip blog §3.3);
* at temperature > 0 the emitted tokens follow the target distribution:
  checked by exact enumeration at a tiny vocabulary, and by a chi-square test
  of the sampled path.
"""

from dataclasses import replace
from itertools import product

import numpy as np
import pytest

from synthetic import TINY, make_weights, weights_to_numpy, make_prompt, shrink
from synthetic.configs import Policy
from oracle import OracleModel, prefill, ar_generate, ssd_generate
from oracle.model import softmax
from oracle.speculative import acceptance_ratio, residual_distribution, accept_stochastic
from oracle.philox import gumbel_argmax, uniform


def _model(dtype="fp32", lm_head_scale=10.0, w=TINY):
    return OracleModel(w.shape, weights_to_numpy(
        make_weights(w, dtype=dtype, lm_head_scale=lm_head_scale, random_gains=True)))


POLICIES = [
    Policy(mode="skip", skip=(2,), d_max=4, tau=0.5),
    Policy(mode="skip", skip=(2,), d_max=4, tau=None),
    Policy(mode="skip", skip=(2,), d_max=4, tau=0.2),
    Policy(mode="skip", skip=(1, 2), d_max=3, tau=0.05),
    Policy(mode="skip", skip=(0, 3), d_max=5, tau=None),
    Policy(mode="skip", skip=(), d_max=4, tau=None),
    Policy(mode="exit", exit_layer=0, d_max=6, tau=None),
    Policy(mode="exit", exit_layer=1, d_max=4, tau=0.1),
    Policy(mode="exit", exit_layer=3, d_max=3, tau=None),
]


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("pi", range(len(POLICIES)))
def test_greedy_ssd_equals_ar(dtype, pi):
    pol = POLICIES[pi]
    m = _model(dtype)
    prompt = make_prompt(TINY)
    st_ar = prefill(m, prompt, pol, 128)
    ar_generate(m, st_ar, pol, 40)
    st = prefill(m, prompt, pol, 128)
    stats = ssd_generate(m, st, pol, 40)
    assert st.tokens == st_ar.tokens
    for r in stats.records:
        assert 1 <= len(r.emitted) <= r.d + 1
        assert r.d <= pol.d_max


def test_kv_reuse_equals_fresh_recompute():
    pol = Policy(mode="skip", skip=(1, 2), d_max=4, tau=0.05)
    m = _model("bf16")
    st = prefill(m, make_prompt(TINY), pol, 128)
    stats = ssd_generate(m, st, pol, 30)
    assert any(r.accepted < r.d for r in stats.records)   # rollbacks happened
    n = st.n
    fresh = m.new_cache(128)
    m.run_layers(m.embed_rows(st.tokens[: n - 1]), range(n - 1), fresh, range(4))
    for l in range(4):
        np.testing.assert_array_equal(st.kv.K[l][:, : n - 1], fresh.K[l][:, : n - 1])
        np.testing.assert_array_equal(st.kv.V[l][:, : n - 1], fresh.V[l][:, : n - 1])


@pytest.mark.parametrize("pol", [Policy(mode="skip", skip=(), d_max=4, tau=None),
                                 Policy(mode="exit", exit_layer=3, d_max=5, tau=None)])
def test_full_model_draft_accepts_everything(pol):
    m = _model("bf16")
    st = prefill(m, make_prompt(TINY), pol, 128)
    stats = ssd_generate(m, st, pol, 36)
    assert stats.alpha == 1.0
    for r in stats.records:
        assert r.d == pol.d_max and r.accepted == pol.d_max
        assert len(r.emitted) == pol.d_max + 1


def test_tau_above_one_reduces_to_ar_steps():
    pol = Policy(mode="skip", skip=(2,), d_max=4, tau=1.5)
    m = _model("fp32")
    st = prefill(m, make_prompt(TINY), pol, 128)
    stats = ssd_generate(m, st, pol, 10)
    assert stats.rounds == 10
    assert all(r.d == 0 and len(r.emitted) == 1 and r.stop_conf is not None
               for r in stats.records)


def test_tau_zero_always_drafts_dmax():
    pol = Policy(mode="skip", skip=(2,), d_max=3, tau=0.0)
    m = _model("fp32")
    st = prefill(m, make_prompt(TINY), pol, 128)
    stats = ssd_generate(m, st, pol, 20)
    assert all(r.d == 3 and r.extra_pass for r in stats.records)


def test_confidence_is_top1_probability():
    pol = Policy(mode="skip", skip=(2,), d_max=4, tau=0.2)
    m = _model("fp32")
    st = prefill(m, make_prompt(TINY), pol, 128)
    stats = ssd_generate(m, st, pol, 20)
    for r in stats.records:
        for c, z in zip(r.conf, r.draft_logits):
            assert c == pytest.approx(np.max(softmax(z)), rel=1e-12)
            assert c >= pol.tau
        if r.stop_conf is not None:
            assert r.stop_conf < pol.tau


# ---------------------------------------------------------------------------
# stochastic acceptance: exactness by enumeration at a tiny vocabulary


def _tiny_vocab_model():
    w = shrink(TINY, n_layers=2, vocab=6)
    return OracleModel(w.shape, weights_to_numpy(
        make_weights(w, lm_head_scale=40.0, random_gains=True))), w


def _last_logits(m, toks, layers):
    kv = m.new_cache(len(toks) + 1)
    X = m.run_layers(m.embed_rows(toks), range(len(toks)), kv, layers)
    return m.lm_head(X[-1:])[0]


def test_stochastic_acceptance_is_exact_by_enumeration():
    m, w = _tiny_vocab_model()
    V, T = w.shape.vocab, 1.0
    full = lambda c: softmax(_last_logits(m, c, range(2)) / T)
    draft = lambda c: softmax(_last_logits(m, c, range(1)) / T)   # exit at layer 0
    ctx = [int(t) for t in make_prompt(w, 5)]

    def first_token_law(c):
        p0, q0 = full(c), draft(c)
        law = np.zeros(V)
        for y0 in range(V):
            a0 = acceptance_ratio(p0, q0, y0)
            law[y0] += q0[y0] * a0
            law += q0[y0] * (1.0 - a0) * residual_distribution(p0, q0)
        return law

    # joint law of the first two emitted tokens of SSD with d = 2
    p0, q0 = full(ctx), draft(ctx)
    res0 = residual_distribution(p0, q0)
    joint = np.zeros((V, V))
    for y0, y1 in product(range(V), repeat=2):
        q1 = draft(ctx + [y0])
        p1 = full(ctx + [y0])
        pr = q0[y0] * q1[y1]
        a0 = acceptance_ratio(p0, q0, y0)
        a1 = acceptance_ratio(p1, q1, y1)
        joint[y0, y1] += pr * a0 * a1
        joint[y0, :] += pr * a0 * (1.0 - a1) * residual_distribution(p1, q1)
        for r in range(V):
            joint[r, :] += pr * (1.0 - a0) * res0[r] * first_token_law(ctx + [r])
    ar = np.stack([p0[t] * full(ctx + [t]) for t in range(V)])
    assert np.abs(joint.sum() - 1.0) < 1e-12
    np.testing.assert_allclose(joint, ar, rtol=0, atol=1e-12)
    # the draft really differs from the target here
    assert np.max(np.abs(p0 - q0)) > 0.05


def test_sampled_acceptance_path_follows_target():
    # The Philox-driven path (draft sampling, acceptance uniform, residual
    # sampling) reproduces p0 for the first emitted token.
    from scipy.stats import chisquare
    rng = np.random.default_rng(5)
    V, T, seed = 5, 1.0, 77
    Z0 = rng.standard_normal(V) * 2
    Q0 = rng.standard_normal(V) * 2
    Q1 = rng.standard_normal((V, V)) * 2
    P1 = rng.standard_normal((V, V)) * 2
    P2 = rng.standard_normal((V, V, V)) * 2
    counts = np.zeros(V)
    n_rounds = 30000
    for rnd in range(n_rounds):
        y0 = gumbel_argmax(Q0 / T, seed, 10, rnd, 0)
        y1 = gumbel_argmax(Q1[y0] / T, seed, 11, rnd, 0)
        P = np.stack([Z0, P1[y0], P2[y0, y1]])
        a, em = accept_stochastic(
            P, [Q0, Q1[y0]], [y0, y1], T,
            draw_u=lambda j: uniform(seed, 10 + j, rnd, 1),
            draw_tok=lambda j, logw: gumbel_argmax(logw, seed, 10 + j, rnd, 2))
        assert 1 <= len(em) <= 3
        counts[em[0]] += 1
    p0 = softmax(Z0 / T)
    assert chisquare(counts, n_rounds * p0).pvalue > 1e-3


def test_stochastic_exit_mode_runs():
    pol = Policy(mode="exit", exit_layer=1, d_max=5, tau=None, temperature=0.6, seed=1234)
    m = _model("bf16", lm_head_scale=4.0)
    st = prefill(m, make_prompt(TINY), pol, 128)
    stats = ssd_generate(m, st, pol, 30)
    assert st.n == 16 + 1 + 30
    assert all(0 <= t < TINY.shape.vocab for t in st.tokens)
    assert 0.0 < stats.alpha < 1.0
