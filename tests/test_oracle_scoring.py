"""Pins for the oracle's matchness scoring (SWIFT §4.1, §4.1.2, D.2)."""

import numpy as np
import pytest

from synthetic import TINY, make_weights, weights_to_numpy, make_prompt, shrink
from synthetic.configs import Policy
from oracle import OracleModel, prefill, ar_generate, score_masks, score_masks_bruteforce


def _setup(n_gen=12, lm_head_scale=10.0):
    w = shrink(TINY, n_layers=6)
    m = OracleModel(w.shape, weights_to_numpy(
        make_weights(w, dtype="bf16", lm_head_scale=lm_head_scale, random_gains=True)))
    pol = Policy(mode="skip", skip=(), d_max=4)
    st = prefill(m, make_prompt(w, 10), pol, 64)
    ar_generate(m, st, pol, n_gen)       # the window holds full-model greedy tokens
    return m, st


def test_empty_mask_scores_one_on_greedy_window():
    m, st = _setup()
    scores, best, _ = score_masks(m, st.tokens, st.kv, [(), (1, 2)], N=8)
    assert scores[0] == 1.0
    assert best == 0


def test_batched_scoring_equals_bruteforce_count():
    m, st = _setup()
    masks = [(1,), (2, 4), (0, 5), (1, 2, 3), (3,)]
    N = 8
    scores, best, _ = score_masks(m, st.tokens, st.kv, masks, N=N)
    counts = score_masks_bruteforce(m, st.tokens, st.kv, masks, N=N)
    np.testing.assert_array_equal(np.round(scores * N).astype(np.int64), counts)
    assert best == int(np.argmax(counts))
    # the masks are not all equally good, so the test discriminates
    assert len(set(counts.tolist())) > 1


def test_best_mask_ties_go_to_lowest_index():
    m, st = _setup()
    scores, best, _ = score_masks(m, st.tokens, st.kv, [(1, 2), (), ()], N=8)
    assert scores[1] == scores[2] == 1.0
    assert best == 1


def test_scoring_does_not_touch_the_shared_cache():
    m, st = _setup()
    before = [k.copy() for k in st.kv.K]
    score_masks(m, st.tokens, st.kv, [(1,), (2,)], N=8)
    for a, b in zip(before, st.kv.K):
        np.testing.assert_array_equal(a, b)
