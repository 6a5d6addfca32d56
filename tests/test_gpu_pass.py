"""The persistent pass kernel computes exactly what one kernel per step computes.

Each decode pass (draft step, extra pass, verify pass, autoregressive step)
runs either as one persistent launch or as one kernel per step; both use the
same device code and the same partitions.  For skip and exit policies, MHA
and GQA shapes, greedy and sampled decoding, the same prefill and rounds give
identical drafts, draft confidences, verify logits (bitwise), emitted tokens
and autoregressive tokens on both paths.
"""

import numpy as np
import pytest

from synthetic import TINY, make_weights, make_prompt
from synthetic.configs import Policy, ModelShape, Workload
from tests.gpu_util import to_device_weights

pytestmark = pytest.mark.gpu

SMALL_GQA = Workload(name="small-gqa", shape=ModelShape(
    n_layers=6, d_model=512, n_heads=8, n_kv_heads=2, head_dim=64, ffn_dim=1408, vocab=2048),
    scaled_layers=(2, 3), scale=0.1)
MID = Workload(name="mid-dh128", shape=ModelShape(
    n_layers=4, d_model=1024, n_heads=8, n_kv_heads=8, head_dim=128, ffn_dim=2816, vocab=4096),
    scaled_layers=(1, 2), scale=0.1)

CASES = [
    (TINY, Policy(mode="skip", skip=(2,), d_max=4, tau=None)),
    (TINY, Policy(mode="exit", exit_layer=1, d_max=6, tau=None, temperature=0.6, seed=7)),
    (SMALL_GQA, Policy(mode="skip", skip=(2, 3), d_max=8, tau=0.1)),
    (MID, Policy(mode="skip", skip=(1, 2), d_max=5, tau=None, temperature=0.8, seed=3)),
    (MID, Policy(mode="exit", exit_layer=0, d_max=3, tau=0.05)),
    (SMALL_GQA, Policy(mode="skip", skip_attn=(2,), skip_mlp=(3, 4), d_max=6, tau=None)),
]


@pytest.fixture(scope="module")
def ssd():
    import __graft_entry__ as g
    g.build()
    import self_speculative_decoding_gb300 as m
    return m


def _run(ctx, pol, prompt, rounds):
    ctx.set_policy(pol)
    first = ctx.prefill(prompt)
    out = []
    for _ in range(rounds):
        drafts, conf = ctx.draft()
        logits = ctx.verify(want_logits=True)
        emitted = ctx.accept()
        out.append((drafts, conf, logits, emitted))
    ar, _ = ctx.decode_ar(12)
    gen, _ = ctx.generate(24)
    return first, out, ar, gen


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_pass_kernel_matches_kernel_per_step(ssd, ci):
    w, pol = CASES[ci]
    wts = make_weights(w, dtype="bf16", lm_head_scale=10.0, random_gains=True)
    ctx = ssd.SSDContext(w.shape, to_device_weights(wts), max_seq=256)
    ctx.set_policy(pol)
    assert ctx.set_pass_kernel(True), "the persistent pass kernel is not in use"
    prompt = make_prompt(w, 20)
    a = _run(ctx, pol, prompt, 6)
    assert not ctx.set_pass_kernel(False)
    b = _run(ctx, pol, prompt, 6)
    assert a[0] == b[0]
    for (d1, c1, l1, e1), (d2, c2, l2, e2) in zip(a[1], b[1]):
        assert d1 == d2 and e1 == e2
        assert np.array_equal(np.asarray(c1, np.float32), np.asarray(c2, np.float32))
        assert np.array_equal(l1, l2)
    assert a[2] == b[2] and a[3] == b[3]
    ctx.close()


def test_pass_kernel_survives_policy_changes(ssd):
    w = TINY
    wts = make_weights(w, dtype="bf16", lm_head_scale=10.0, random_gains=True)
    ctx = ssd.SSDContext(w.shape, to_device_weights(wts), max_seq=256)
    prompt = make_prompt(w, 16)
    outs = []
    for pol in (Policy(mode="skip", skip=(1,), d_max=3, tau=None),
                Policy(mode="exit", exit_layer=2, d_max=5, tau=None),
                Policy(mode="skip", skip=(1,), d_max=3, tau=None)):
        ctx.set_policy(pol)
        ctx.prefill(prompt)
        outs.append(ctx.generate(20)[0])
    assert outs[0] == outs[2] == outs[1]   # greedy output does not depend on the policy
    ctx.close()
