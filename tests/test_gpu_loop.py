"""ssd_generate's device loop (one graph launch: conditional nodes decide the
draft loop's stop, the extra pass, the verify width and the next round on the
device) against the host-driven loop through the context C-ABI.

* Same tokens, same committed context and the same counts (rounds, drafted,
  accepted, emitted, draft steps, siblings verified and taken) for greedy and
  sampled decoding, skip / sub-layer / exit policies, dynamic verification and
  verify passes wider than the activation stage.
* Generation continues across calls exactly as in one call.
"""

import pytest

from synthetic import TINY, make_weights, make_prompt
from synthetic.configs import Policy, ModelShape, Workload
from tests.gpu_util import to_device_weights

pytestmark = pytest.mark.gpu

WIDE = Workload(name="wide-d4096", shape=ModelShape(
    n_layers=3, d_model=4096, n_heads=32, n_kv_heads=8, head_dim=128, ffn_dim=2048, vocab=4096),
    scaled_layers=(1,), scale=0.1)

CASES = [
    (TINY, Policy(mode="skip", skip=(2,), d_max=4, tau=None)),
    (TINY, Policy(mode="skip", skip=(1, 2), d_max=7, tau=0.2)),
    (TINY, Policy(mode="exit", exit_layer=1, d_max=12, tau=None)),
    (TINY, Policy(mode="skip", skip_attn=(1,), skip_mlp=(2,), d_max=5, tau=None)),
    (TINY, Policy(mode="skip", skip=(2,), d_max=4, tau=None, tree_tau=1.0, tree_max=4)),
    (TINY, Policy(mode="skip", skip=(2,), d_max=6, tau=None, temperature=0.8, seed=7)),
    (TINY, Policy(mode="skip", skip=(0,), d_max=0, tau=None)),
    (WIDE, Policy(mode="skip", skip=(1,), d_max=8, tau=None)),
    (WIDE, Policy(mode="exit", exit_layer=0, d_max=7, tau=None, tree_tau=1.0, tree_max=8)),
]

KEYS = ("rounds", "drafted", "accepted", "emitted", "draft_steps", "side_rows", "side_accepted")


@pytest.fixture(scope="module")
def ssd():
    import __graft_entry__ as g
    g.build()
    import self_speculative_decoding_gb300 as m
    return m


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_device_loop_equals_host_loop(ssd, ci):
    w, pol = CASES[ci]
    wts = make_weights(w, dtype="bf16", lm_head_scale=10.0, random_gains=True)
    ctx = ssd.SSDContext(w.shape, to_device_weights(wts), max_seq=256)
    ctx.set_policy(pol)
    prompt = make_prompt(w, 20)
    res = {}
    for loop in (False, True):
        active = ctx.set_device_loop(loop)
        if loop:
            assert active, ctx.last_error()
        ctx.prefill(prompt)
        toks, st = ctx.generate(60)
        res[loop] = (toks, ctx.tokens(), {k: st[k] for k in KEYS})
        if active:
            assert st["draft_ms"] == 0.0 and st["kernel_launches"] > 0
    assert res[True] == res[False]
    ctx.close()


def test_device_loop_continues_across_calls(ssd):
    w, pol = CASES[1]
    wts = make_weights(w, dtype="bf16", lm_head_scale=10.0, random_gains=True)
    ctx = ssd.SSDContext(w.shape, to_device_weights(wts), max_seq=256)
    ctx.set_policy(pol)
    assert ctx.set_device_loop(True), ctx.last_error()
    prompt = make_prompt(w, 20)
    ctx.prefill(prompt)
    full, _ = ctx.generate(50)
    ctx.prefill(prompt)
    a, _ = ctx.generate(1)
    b, _ = ctx.generate(22)
    c, _ = ctx.generate(27)
    assert a + b + c == full
    ctx.close()


def test_device_loop_in_several_launches(ssd):
    # more than one launch's worth of tokens (512 per launch): the rounds
    # continue across launches exactly as in the host-driven loop
    w, pol = CASES[0]
    wts = make_weights(w, dtype="bf16", lm_head_scale=10.0, random_gains=True)
    ctx = ssd.SSDContext(w.shape, to_device_weights(wts), max_seq=1280)
    ctx.set_policy(pol)
    prompt = make_prompt(w, 20)
    res = {}
    for loop in (False, True):
        assert ctx.set_device_loop(loop) == loop, ctx.last_error()
        ctx.prefill(prompt)
        toks, st = ctx.generate(1100)
        res[loop] = (toks, ctx.tokens(), {k: st[k] for k in KEYS})
    assert res[True] == res[False]
    ctx.close()
