"""Pins for sub-layer skip policies in the oracle (SWIFT Fig. 10: the
attention and the MLP sublayer of a layer are skipped separately).

* Dropping both sublayers of the layers in S is the whole-layer skip S:
  identical drafts, confidences and verify logits.
* A sublayer whose residual branch is zero contributes nothing: with W_o of
  layer l zeroed, dropping l's attention drafts exactly what keeping it
  does; dropping l's MLP instead does not (which catches swapped sublayers);
  the same holds with W_down zeroed and the roles exchanged.
* Greedy self-speculative output with sub-layer policies equals greedy
  autoregressive output (losslessness).
* s0, the first layer the verify recomputes, is the first layer with any
  dropped sublayer.
"""

import numpy as np
import pytest

from synthetic import TINY, make_weights, weights_to_numpy, make_prompt
from synthetic.configs import Policy
from oracle import OracleModel, prefill, ar_generate, ssd_generate
from oracle.speculative import ssd_round


def _model(zero=None, dtype="fp32"):
    wn = weights_to_numpy(make_weights(TINY, dtype=dtype, lm_head_scale=10.0, random_gains=True))
    if zero is not None:
        layer, name = zero
        wn["layers"][layer][name] = np.zeros_like(wn["layers"][layer][name])
    return OracleModel(TINY.shape, wn)


def _first_rounds(m, pol, n_rounds=3):
    st = prefill(m, make_prompt(TINY), pol, 128)
    return [ssd_round(m, st, pol) for _ in range(n_rounds)]


def test_both_sublayers_equal_whole_layer_skip():
    m = _model()
    whole = Policy(mode="skip", skip=(1, 2), d_max=4, tau=None)
    parts = Policy(mode="skip", skip_attn=(1, 2), skip_mlp=(1, 2), d_max=4, tau=None)
    for a, b in zip(_first_rounds(m, whole), _first_rounds(m, parts)):
        assert a.draft == b.draft and a.emitted == b.emitted
        assert np.array_equal(np.stack(a.draft_logits), np.stack(b.draft_logits))
        assert np.array_equal(a.verify_logits, b.verify_logits)


@pytest.mark.parametrize("zeroed,neutral,active", [
    ("wo", "skip_attn", "skip_mlp"),
    ("w_down", "skip_mlp", "skip_attn"),
])
def test_dropping_a_zero_branch_changes_nothing(zeroed, neutral, active):
    layer = 2
    m = _model(zero=(layer, zeroed))
    full = Policy(mode="skip", skip=(), d_max=3, tau=None)

    def pol(extra):
        # the same s0 for every policy compared: layer 3's MLP is also dropped
        kw = {"skip_attn": (), "skip_mlp": (3,)}
        if extra:
            kw[extra] = tuple(sorted(set(kw[extra]) | {layer}))
        return Policy(mode="skip", d_max=3, tau=None, **kw)

    base, drop_neutral, drop_active = pol(None), pol(neutral), pol(active)
    ra = _first_rounds(m, base, 1)[0]
    rn = _first_rounds(m, drop_neutral, 1)[0]
    rx = _first_rounds(m, drop_active, 1)[0]
    za, zn, zx = (np.stack(r.draft_logits) for r in (ra, rn, rx))
    assert np.allclose(za, zn, rtol=0, atol=1e-9)
    assert np.max(np.abs(za - zx)) > 1e-3
    assert full.first_recomputed(4) == 4


POLICIES = [
    Policy(mode="skip", skip_attn=(2,), d_max=4, tau=None),
    Policy(mode="skip", skip_mlp=(1,), d_max=4, tau=0.1),
    Policy(mode="skip", skip=(3,), skip_attn=(1,), skip_mlp=(2,), d_max=5, tau=None),
    Policy(mode="skip", skip_attn=(0, 2), skip_mlp=(1, 3), d_max=3, tau=None),
]


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("pi", range(len(POLICIES)))
def test_greedy_sublayer_ssd_equals_ar(dtype, pi):
    pol = POLICIES[pi]
    m = _model(dtype=dtype)
    prompt = make_prompt(TINY)
    st_ar = prefill(m, prompt, pol, 128)
    ar_generate(m, st_ar, pol, 30)
    st = prefill(m, prompt, pol, 128)
    stats = ssd_generate(m, st, pol, 30)
    assert st.tokens == st_ar.tokens
    assert any(r.d > 0 for r in stats.records)


def test_first_recomputed_layer():
    assert Policy(mode="skip", skip_mlp=(5, 9)).first_recomputed(12) == 5
    assert Policy(mode="skip", skip=(7,), skip_attn=(3,)).first_recomputed(12) == 3
    assert Policy(mode="skip", skip_attn=(2,)).sublayers(2) == (False, True)
    assert Policy(mode="skip", skip_mlp=(2,)).sublayers(2) == (True, False)
    assert Policy(mode="skip", skip=(2,), skip_mlp=(2,)).sublayers(2) == (False, False)
    assert Policy(mode="skip", skip_mlp=(2,)).draft_layers(4) == (0, 1, 2, 3)
