"""GPU lossy early exit (ssd_decode_lossy; LayerSkip blog §3, inference mode
one) and AdaInfer exit features (ssd_layer_features; EE-structure page,
steps 1-2) against the oracle.

* Lossy greedy tokens equal the oracle's lossy tokens up to the oracle's
  first near tie (top-1/top-2 logit gap <= 0.1).
* With a draft that runs every sublayer, lossy decoding is the library's own
  autoregressive decoding, bit for bit, and leaves no lossy mark.
* After lossy steps that drop layers, the lossless entry points refuse
  (STATE) until the context is rewound to before them or prefilled again.
* Features per layer match the oracle: top prob and gap within 1e-3 x head
  (the confidence tolerance; an LM head sharpened by `head` multiplies the
  logit deviation that bf16 rounding boundaries cause, as in the round
  parity tests), top-1 exact where the oracle's logit gap exceeds 0.1; the
  step commits what decode_ar commits.
"""

import math

import numpy as np
import pytest

from synthetic import TINY, make_weights, weights_to_numpy, make_prompt
from synthetic.configs import Policy, ModelShape, Workload
from tests.gpu_util import to_device_weights

pytestmark = pytest.mark.gpu

SMALL = Workload(name="small-lossy", shape=ModelShape(
    n_layers=6, d_model=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn_dim=704, vocab=1024),
    scaled_layers=(2, 4), scale=0.1)


@pytest.fixture(scope="module")
def ssd():
    import __graft_entry__ as g
    g.build()
    import self_speculative_decoding_gb300 as m
    return m


def _wts(w, head=10.0):
    return make_weights(w, dtype="bf16", lm_head_scale=head, random_gains=True)


@pytest.mark.parametrize("w,pol", [
    (TINY, Policy(mode="exit", exit_layer=1, d_max=3)),
    (SMALL, Policy(mode="skip", skip=(2, 4), d_max=3)),
    (SMALL, Policy(mode="skip", skip_attn=(1,), skip_mlp=(3, 4), d_max=3)),
])
def test_lossy_matches_oracle(ssd, w, pol):
    from oracle import OracleModel, prefill
    from oracle.adaptive import lossy_step
    wts = _wts(w)
    prompt = make_prompt(w, 12)
    ctx = ssd.SSDContext(w.shape, to_device_weights(wts), max_seq=128)
    ctx.set_policy(pol)
    ctx.prefill(prompt)
    got, st = ctx.decode_lossy(24)
    assert st["emitted"] == 24
    m = OracleModel(w.shape, weights_to_numpy(wts))
    ost = prefill(m, prompt, pol, 128)
    assert ctx.tokens()[:len(prompt) + 1] == ost.tokens
    for i in range(24):
        z = lossy_step(m, ost, pol)
        s = np.sort(z)
        if s[-1] - s[-2] <= 0.1:
            break
        assert got[i] == ost.tokens[-1], i
    ctx.close()


@pytest.mark.parametrize("pol", [Policy(mode="skip", skip=(), d_max=3),
                                 Policy(mode="exit", exit_layer=5, d_max=3)])
def test_lossy_with_every_layer_is_ar(ssd, pol):
    w = SMALL
    ctx = ssd.SSDContext(w.shape, to_device_weights(_wts(w)), max_seq=128)
    ctx.set_policy(pol)
    prompt = make_prompt(w, 10)
    ctx.prefill(prompt)
    a, _ = ctx.decode_ar(20)
    ctx.prefill(prompt)
    b, _ = ctx.decode_lossy(20)
    assert a == b
    ctx.generate(4)              # no lossy mark: lossless decoding continues
    ctx.close()


def test_lossy_mark_guards_lossless_calls(ssd):
    from self_speculative_decoding_gb300 import SSDError
    w = SMALL
    ctx = ssd.SSDContext(w.shape, to_device_weights(_wts(w)), max_seq=128, max_score_rows=64)
    pol = Policy(mode="skip", skip=(2, 4), d_max=3)
    ctx.set_policy(pol)
    prompt = make_prompt(w, 10)
    ctx.prefill(prompt)
    ctx.decode_ar(5)
    n = len(ctx.tokens())
    ctx.decode_lossy(6)
    for call in (lambda: ctx.generate(2), lambda: ctx.decode_ar(2),
                 lambda: ctx.score_masks([(), (1,)], 4), lambda: ctx.layer_features()):
        with pytest.raises(SSDError, match="STATE"):
            call()
    ctx.decode_lossy(2)          # lossy decoding may go on
    ctx.rewind(n + 1)            # position n is still lossy: still refused
    with pytest.raises(SSDError, match="STATE"):
        ctx.decode_ar(1)
    ctx.rewind(n)                # back to before the first lossy position
    ref, _ = ctx.decode_ar(4)
    ctx.prefill(prompt)
    ctx.decode_ar(5)
    again, _ = ctx.decode_ar(4)
    assert ref == again
    ctx.close()


@pytest.mark.parametrize("w,min_layer,head", [(TINY, 0, 1.0), (TINY, 0, 10.0), (SMALL, 2, 1.0),
                                              (SMALL, 2, 10.0)])
def test_layer_features_match_oracle(ssd, w, min_layer, head):
    from oracle import OracleModel, prefill
    from oracle.adaptive import layer_features
    wts = _wts(w, head)
    tol = 1e-3 * head
    pol = Policy(mode="skip", skip=(), d_max=3)
    prompt = make_prompt(w, 12)
    ctx = ssd.SSDContext(w.shape, to_device_weights(wts), max_seq=128)
    ctx.set_policy(pol)
    ctx.prefill(prompt)
    seq = ctx.tokens()
    top1, p1, gap = ctx.layer_features(min_layer)
    after = ctx.tokens()
    # the step commits what an autoregressive step commits
    ctx.prefill(prompt)
    ar, _ = ctx.decode_ar(1)
    assert after[-1] == ar[0] and after[:-1] == seq
    m = OracleModel(w.shape, weights_to_numpy(wts))
    ost = prefill(m, prompt, pol, 128)
    assert ost.tokens == seq
    f = layer_features(m, ost, pol, min_layer)
    L = w.shape.n_layers
    assert len(top1) == L - min_layer
    for i in range(L - min_layer):
        assert abs(p1[i] - f.top_prob[i]) <= tol, (i, p1[i], f.top_prob[i])
        assert abs(gap[i] - f.gap[i]) <= 2 * tol, (i, gap[i], f.gap[i])
        p2 = f.top_prob[i] - f.gap[i]
        if p2 <= 0 or math.log(f.top_prob[i] / p2) > 0.1:
            assert top1[i] == f.top1[i], i
    ctx.close()


def test_layer_features_arguments(ssd):
    from self_speculative_decoding_gb300 import SSDError
    w = TINY
    ctx = ssd.SSDContext(w.shape, to_device_weights(_wts(w)), max_seq=64)
    ctx.set_policy(Policy(mode="skip", skip=(), d_max=2))
    ctx.prefill(make_prompt(w, 8))
    with pytest.raises(SSDError, match="INVALID_ARG"):
        ctx.layer_features(w.shape.n_layers)
    with pytest.raises(SSDError, match="INVALID_ARG"):
        ctx.layer_features(-1)
    ctx.close()
