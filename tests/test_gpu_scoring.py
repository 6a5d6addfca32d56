"""GPU parity of candidate-mask scoring (SWIFT §4.1.2) through ssd_score_masks.

* GPU and oracle score the same candidate skip sets on the same committed
  context (the oracle's own greedy tokens, fed to the GPU as a prompt); per
  candidate the match counts may differ only at window rows where the
  oracle's top-1/top-2 gap is <= 0.1.
* The empty candidate reproduces the full model, so on the library's own
  greedy window it scores 1.0, except at rows with a near tie (the batched
  scoring forward sums in its own fixed order, not the decode GEMV's).
* Scoring reads the shared KV cache but never writes it.
"""

import numpy as np
import pytest
import torch

from synthetic import TINY, make_weights, weights_to_numpy, make_prompt, make_masks
from synthetic.configs import Policy, ModelShape, Workload
from tests.gpu_util import to_device_weights

pytestmark = pytest.mark.gpu

SMALL = Workload(name="small-score", shape=ModelShape(
    n_layers=8, d_model=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn_dim=704, vocab=1024),
    scaled_layers=(3, 5), scale=0.1, mask_layers=tuple(range(2, 8)), mask_drop=3, n_masks=6)


@pytest.fixture(scope="module")
def ssd():
    import __graft_entry__ as g
    g.build()
    import self_speculative_decoding_gb300 as m
    return m


def _near_tie(z, thr=0.1):
    s = np.sort(z)
    return s[-1] - s[-2] <= thr


@pytest.mark.parametrize("N", [8, 20, 33])
def test_scoring_matches_oracle(ssd, N):
    from oracle import OracleModel, prefill, ar_generate, score_masks
    w = SMALL
    wts = make_weights(w, dtype="bf16", lm_head_scale=10.0, random_gains=True)
    pol = Policy(mode="skip", skip=(), d_max=4)
    m = OracleModel(w.shape, weights_to_numpy(wts))
    st = prefill(m, make_prompt(w, 12), pol, 256)
    ar_generate(m, st, pol, N + 4)
    seq = st.tokens
    masks = [()] + make_masks(w)
    ref, ref_best, logits = score_masks(m, seq, st.kv, masks, N)

    ctx = ssd.SSDContext(w.shape, to_device_weights(wts), max_seq=256, max_score_rows=512)
    ctx.set_policy(pol)
    ctx.prefill(seq)
    ctx.rewind(len(seq))            # the committed context is exactly the oracle's
    got, best = ctx.score_masks(masks, N)
    targets = np.asarray(seq[len(seq) - N:])
    for k in range(len(masks)):
        ties = sum(_near_tie(z) for z in logits[k])
        assert abs(round(got[k] * N) - round(ref[k] * N)) <= ties, (k, got[k], ref[k], ties)
        if ties == 0:
            assert round(got[k] * N) == round(ref[k] * N)
    assert 0 <= best < len(masks)
    assert got[best] == np.max(got)
    ctx.close()


@pytest.mark.parametrize("w", [TINY, SMALL])
def test_empty_mask_scores_one_on_own_greedy_window(ssd, w):
    from oracle import OracleModel, prefill, score_masks
    wts = make_weights(w, dtype="bf16", random_gains=True)
    ctx = ssd.SSDContext(w.shape, to_device_weights(wts), max_seq=256, max_score_rows=256)
    pol = Policy(mode="skip", skip=(), d_max=4)
    ctx.set_policy(pol)
    ctx.prefill(make_prompt(w, 10))
    ctx.decode_ar(40)
    scores, best = ctx.score_masks([(), (1,), (0, 2)], 32)
    # the full model predicts its own greedy tokens; the batched pass sums in
    # another order than the decode, so a miss is allowed only at a row whose
    # (oracle) top-1/top-2 gap is <= 0.1
    seq = ctx.tokens()
    m = OracleModel(w.shape, weights_to_numpy(wts))
    st = prefill(m, seq, pol, 256)
    _, _, logits = score_masks(m, seq, st.kv, [()], 32)
    ties = sum(_near_tie(z) for z in logits[0])
    assert round(scores[0] * 32) >= 32 - ties
    if ties == 0:
        assert scores[0] == 1.0 and best == 0
    ctx.close()


def test_scoring_leaves_the_shared_cache_untouched(ssd):
    w = SMALL
    wts = make_weights(w, dtype="bf16", lm_head_scale=10.0, random_gains=True)
    ctx = ssd.SSDContext(w.shape, to_device_weights(wts), max_seq=256, max_score_rows=256)
    pol = Policy(mode="skip", skip=(3, 5), d_max=4, tau=None)
    ctx.set_policy(pol)
    prompt = make_prompt(w, 12)
    ctx.prefill(prompt)
    ctx.decode_ar(30)
    n = len(ctx.tokens())
    ref, _ = ctx.decode_ar(20)
    ctx.rewind(n)
    ctx.score_masks(make_masks(w), 24)
    after, _ = ctx.generate(20)
    assert after == ref
    ctx.close()


def test_scoring_capacity_errors(ssd):
    from self_speculative_decoding_gb300 import SSDError
    w = TINY
    wts = make_weights(w, dtype="bf16")
    ctx = ssd.SSDContext(w.shape, to_device_weights(wts), max_seq=128, max_score_rows=64)
    ctx.set_policy(Policy(mode="skip", skip=(), d_max=4))
    ctx.prefill(make_prompt(w, 10))
    with pytest.raises(SSDError, match="CAPACITY"):
        ctx.score_masks([()] * 3, 32)            # K * N > max_score_rows
    with pytest.raises(SSDError, match="CAPACITY"):
        ctx.score_masks([()], 20)                # window longer than the context
    ctx.close()


def test_scoring_together_equals_alone(ssd):
    # candidates that agree on the first layers share those rows; every step is
    # row-count invariant, so a candidate's matchness is bit-identical whether
    # it is scored with others (shared prefixes, duplicates) or alone
    w = SMALL
    wts = make_weights(w, dtype="bf16", lm_head_scale=10.0, random_gains=True)
    ctx = ssd.SSDContext(w.shape, to_device_weights(wts), max_seq=256, max_score_rows=512)
    ctx.set_policy(Policy(mode="skip", skip=(), d_max=4))
    ctx.prefill(make_prompt(w, 12))
    ctx.decode_ar(40)
    masks = [(), (5,), (2, 5), (2, 6), (2, 5), (6, 7), (2, 3, 4)] + make_masks(w)
    together, best = ctx.score_masks(masks, 24)
    alone = [ctx.score_masks([m], 24)[0][0] for m in masks]
    assert list(together) == alone
    assert best == int(np.argmax(together))
    ctx.close()
