"""Planted mistakes in the oracle (on the CPU) must be caught by its pins.

Each case monkeypatches one plausible slip into the oracle and checks that
the corresponding independent check then fails.
"""

import numpy as np
import pytest

from synthetic import TINY, make_weights, weights_to_numpy, make_prompt, shrink
from synthetic.configs import Policy
from oracle import OracleModel, prefill, ar_generate, ssd_generate
from oracle import speculative as spec_mod
from oracle.model import softmax

from tests.test_oracle_model import _torch_reference_logits, _oracle_logits


def _disagrees_with_library(model_patch, monkeypatch):
    w = shrink(TINY, n_heads=8, n_kv_heads=2, head_dim=32)
    wn = weights_to_numpy(make_weights(w, dtype="fp32", random_gains=True))
    m = OracleModel(w.shape, wn)
    model_patch(m, monkeypatch)
    toks = make_prompt(w, 12)
    got = _oracle_logits(m, toks)
    ref = _torch_reference_logits(w.shape, wn, toks, False)
    return np.max(np.abs(got - ref)) > 1e-6


def test_rope_sign_slip_is_caught(monkeypatch):
    def patch(m, mp):
        orig = m.rope
        mp.setattr(m, "rope", lambda v, pos: orig(v, -pos))
    assert _disagrees_with_library(patch, monkeypatch)


def test_dropped_norm_gain_is_caught(monkeypatch):
    def patch(m, mp):
        mp.setattr(m, "rmsnorm", lambda x, g: x / np.sqrt(np.mean(x * x) + 1e-5))
    assert _disagrees_with_library(patch, monkeypatch)


def test_off_by_one_causal_mask_is_caught(monkeypatch):
    def patch(m, mp):
        orig = m.attention_row
        mp.setattr(m, "attention_row", lambda q, kv, l, pos: orig(q, kv, l, max(pos - 1, 0)))
    assert _disagrees_with_library(patch, monkeypatch)


def test_wrong_kv_group_is_caught(monkeypatch):
    def patch(m, mp):
        s = m.s

        def attn(q, kv, layer, pos):
            out = np.empty((s.n_heads, s.head_dim))
            for h in range(s.n_heads):
                kvh = h % s.n_kv_heads            # interleaved instead of grouped
                sc = kv.K[layer][kvh, : pos + 1] @ q[h] / np.sqrt(s.head_dim)
                p = softmax(sc)
                out[h] = p @ kv.V[layer][kvh, : pos + 1]
            return out.reshape(-1)
        mp.setattr(m, "attention_row", attn)
    assert _disagrees_with_library(patch, monkeypatch)


def test_accepting_one_token_too_many_breaks_losslessness(monkeypatch):
    pol = Policy(mode="skip", skip=(1, 2), d_max=4, tau=None)
    w = TINY
    m = OracleModel(w.shape, weights_to_numpy(make_weights(w, lm_head_scale=10.0)))
    prompt = make_prompt(w)
    st_ar = prefill(m, prompt, pol, 128)
    ar_generate(m, st_ar, pol, 30)

    orig_round = spec_mod.ssd_round

    def sloppy_round(model, st, policy):
        n0 = st.n
        rec = orig_round(model, st, policy)
        if rec.accepted < rec.d:       # keep the first rejected draft as if accepted
            del st.tokens[n0:]
            st.tokens.extend(rec.draft[: rec.accepted + 1])
        return rec
    monkeypatch.setattr(spec_mod, "ssd_round", sloppy_round)
    st = prefill(m, prompt, pol, 128)
    spec_mod.ssd_generate(m, st, pol, 30)
    assert st.tokens != st_ar.tokens


def test_residual_without_clamp_breaks_exactness(monkeypatch):
    # replacing norm(max(0, p - q)) by norm(|p - q|) must break the enumeration identity
    from tests import test_oracle_ssd as t
    monkeypatch.setattr(t, "residual_distribution",
                        lambda p, q: np.abs(p - q) / np.sum(np.abs(p - q)))
    with pytest.raises(AssertionError):
        t.test_stochastic_acceptance_is_exact_by_enumeration()
