"""The oracle's sampled acceptance, end to end: the law of the emitted tokens.

LayerSkip blog §3.3 (layerskip_ssd): each draft y_j is accepted with
probability min(1, p_j(y_j) / q_j(y_j)); the first rejected draft is replaced
by a sample of norm(max(0, p_j - q_j)); when all d drafts are accepted a bonus
token is sampled from p_d, the full model's distribution after the last
draft.  Speculative sampling then emits exactly the target's sequence law:
the first three emitted tokens follow p(x1) p(x2 | x1) p(x3 | x1, x2).

These tests run ``oracle.speculative.accept_stochastic`` itself, with the
Philox draws the oracle's rounds use, over whole sequences built from
several rounds (a round that emits fewer than three tokens is followed by
the next one from the extended context), and compare the frequencies of
(x1, x2, x3) with the product law by a chi-square test.  The target and
draft "models" are fixed logit tables indexed by the context, so every case
is cheap and exact.  Cases:

* a draft unlike the target (rejections and residual draws at depth 0 and 1,
  bonus draws when both drafts pass);
* a draft equal to the target (every draft accepted: the third token is
  always the bonus drawn from p_d);
* a draft equal to the target at even context lengths only (depth 0 always
  accepted in rounds that start there, so depth 1 decides).

Planted mistakes must fail: the bonus drawn from p_{d-1} instead of p_d, and
the depth-1 acceptance and residual computed from the depth-0 row.
"""

from __future__ import annotations

from functools import lru_cache

import numpy as np
import pytest
from scipy.stats import chisquare

from oracle.model import softmax
from oracle.philox import (STREAM_ACCEPT, STREAM_DRAFT, STREAM_RESAMPLE, gumbel_argmax_u,
                           uniforms_table)
from oracle.speculative import accept_stochastic

V = 4          # vocabulary
D = 2          # drafts per round
K = 3          # emitted tokens whose joint law is checked
T = 0.8        # temperature
SEED = 4321
MAX_ROUNDS = K  # every round emits at least one token


@lru_cache(maxsize=None)
def _logits(table_seed: int, prefix) -> np.ndarray:
    """Deterministic logits for a context (a tuple of token ids)."""
    key = table_seed
    for t in prefix:
        key = key * (V + 1) + t + 1
    return np.random.default_rng(key).standard_normal(V) * 1.5


def target(prefix):
    return _logits(11, prefix)


def draft_unlike(prefix):
    return _logits(29, prefix)


def draft_equal(prefix):
    return target(prefix)


def draft_even(prefix):
    return target(prefix) if len(prefix) % 2 == 0 else _logits(29, prefix)


def _product_law() -> np.ndarray:
    law = np.zeros((V,) * K)
    for idx in np.ndindex(*law.shape):
        pr = 1.0
        for i in range(K):
            pr *= softmax(target(idx[:i]) / T)[idx[i]]
        law[idx] = pr
    return law


def _sample(draft, n_seq: int, accept=accept_stochastic, mutate_P=None):
    """Emitted-sequence counts [V]*K and the number of rounds run.

    Sequence s, round r: drafts at positions (context length + j) sampled by
    Gumbel-max on stream 0, the acceptance uniform of draft j on stream 1,
    the residual / bonus draw of depth j on stream 2, all with round counter
    s * MAX_ROUNDS + r -- the oracle's own counter layout."""
    rnd = (np.arange(n_seq)[:, None] * MAX_ROUNDS + np.arange(MAX_ROUNDS)[None, :])
    # positions are context lengths 0..K-1 plus the depth 0..D
    pos = np.arange(K + D + 1)
    Ud = uniforms_table(SEED, pos[None, None, :], rnd[:, :, None], STREAM_DRAFT, V)
    Ua = uniforms_table(SEED, pos[None, None, :], rnd[:, :, None], STREAM_ACCEPT, 1)[..., 0]
    Ur = uniforms_table(SEED, pos[None, None, :], rnd[:, :, None], STREAM_RESAMPLE, V)
    counts = np.zeros((V,) * K)
    rounds = 0
    for s in range(n_seq):
        ctx: tuple = ()
        r = 0
        while len(ctx) < K:
            n = len(ctx)
            ys, Qs = [], []
            for j in range(D):
                z = draft(ctx + tuple(ys))
                ys.append(gumbel_argmax_u(z / T, Ud[s, r, n + j]))
                Qs.append(z)
            P = np.stack([target(ctx + tuple(ys[:j])) for j in range(D + 1)])
            if mutate_P is not None:
                P = mutate_P(P)
            a, em = accept(P, Qs, ys, T,
                           draw_u=lambda j: Ua[s, r, n + j],
                           draw_tok=lambda j, logw: gumbel_argmax_u(logw, Ur[s, r, n + j]))
            assert 0 <= a <= D and len(em) == a + 1 and em[:a] == ys[:a]
            ctx = ctx + tuple(int(t) for t in em)
            r += 1
        counts[ctx[:K]] += 1
        rounds += r
    return counts, rounds


def _pvalue(counts: np.ndarray) -> float:
    law = _product_law()
    return chisquare(counts.reshape(-1), counts.sum() * law.reshape(-1)).pvalue


@pytest.mark.parametrize("draft", [draft_unlike, draft_equal, draft_even],
                         ids=["unlike", "equal", "equal-at-even-lengths"])
def test_emitted_sequence_follows_the_target_law(draft):
    counts, rounds = _sample(draft, 60000)
    assert rounds >= 60000
    assert _pvalue(counts) > 1e-4


def test_cases_reach_every_branch():
    # the cases above really exercise rejections at depth 0 and 1, residual
    # draws and bonus draws
    seen = set()

    def spy(P, Q, ys, T_, draw_u, draw_tok):
        a, em = accept_stochastic(P, Q, ys, T_, draw_u, draw_tok)
        seen.add(a)
        return a, em

    _sample(draft_unlike, 3000, accept=spy)
    assert seen == {0, 1, 2}
    seen.clear()
    _sample(draft_equal, 500, accept=spy)
    assert seen == {2}
    seen.clear()
    _sample(draft_even, 3000, accept=spy)
    assert {1, 2} <= seen


def test_bonus_from_the_previous_row_fails():
    # planted: the bonus token drawn from p_{d-1} instead of p_d
    def bonus_from_previous(P):
        P = P.copy()
        P[D] = P[D - 1]
        return P

    counts, _ = _sample(draft_equal, 20000, mutate_P=bonus_from_previous)
    assert _pvalue(counts) < 1e-6


def test_depth_one_from_the_first_row_fails():
    # planted: depth 1 accepted and resampled against the depth-0 target row
    def first_row(P):
        P = P.copy()
        P[1] = P[0]
        return P

    counts, _ = _sample(draft_unlike, 20000, mutate_P=first_row)
    assert _pvalue(counts) < 1e-6
