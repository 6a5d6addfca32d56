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


def test_score_attention_equals_model_attention_on_forked_caches():
    """oracle.ops.score_attention equals the decoder's own attention row when
    candidate k's window keys are written into a copy of the shared cache at
    positions split + w (the per-candidate fork of oracle.scoring)."""
    from oracle.ops import score_attention
    from oracle.model import OracleModel, KVCache
    from types import SimpleNamespace
    rng = np.random.default_rng(7)
    H, Hkv, dh, N, split, max_seq = 4, 2, 16, 5, 9, 32
    K = rng.standard_normal((Hkv, max_seq, dh))
    V = rng.standard_normal((Hkv, max_seq, dh))
    rows = 3 * N
    WK = rng.standard_normal((rows, Hkv, dh))
    WV = rng.standard_normal((rows, Hkv, dh))
    cand = [2, 0]
    q = rng.standard_normal((len(cand) * N, H, dh))
    got = score_attention(q, cand, N, split, K, V, WK, WV, H, Hkv)
    m = OracleModel.__new__(OracleModel)
    m.s = SimpleNamespace(n_heads=H, n_kv_heads=Hkv, head_dim=dh)
    from oracle.numerics import bf16_round
    for j, k in enumerate(cand):
        kv = KVCache.__new__(KVCache)
        kv.K, kv.V = [K.copy()], [V.copy()]
        for w in range(N):
            kv.K[0][:, split + w] = WK[k * N + w]
            kv.V[0][:, split + w] = WV[k * N + w]
        for i in range(N):
            ref = bf16_round(m.attention_row(q[j * N + i], kv, 0, split + i))
            np.testing.assert_array_equal(got[j * N + i], ref)
