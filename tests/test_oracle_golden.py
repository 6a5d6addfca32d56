"""The oracle still reproduces its stored tiny-workload fixture (regression)."""

import json
import os

from synthetic import TINY, make_weights, weights_to_numpy, make_prompt
from oracle import OracleModel, prefill, ar_generate

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_greedy_fixture():
    with open(os.path.join(HERE, "golden", "tiny_fp32_greedy.json")) as f:
        g = json.load(f)
    m = OracleModel(TINY.shape, weights_to_numpy(make_weights(TINY)))
    prompt = make_prompt(TINY)
    assert [int(t) for t in prompt] == g["prompt"]
    st = prefill(m, prompt, TINY.policy, 128)
    ar_generate(m, st, TINY.policy, TINY.gen_len - 1)
    assert st.tokens[len(prompt):] == g["ar_greedy_tokens"]
    # the literal tiny policy (tau 0.5) never drafts on random weights: top-1
    # probability over 1024 near-uniform logits is far below the threshold
    assert g["ssd_drafted"] == 0 and g["ssd_greedy_tokens"] == g["ar_greedy_tokens"]


def test_tiny_sharp_tree_fixture():
    # dynamic verification (siblings from the draft's second choice) on the
    # sharpened tiny model: the stored run is reproduced, takes siblings, and
    # its tokens are the autoregressive greedy tokens
    from dataclasses import replace
    from synthetic.configs import TINY_SHARP
    from oracle import ssd_generate
    with open(os.path.join(HERE, "golden", "tiny_sharp_tree.json")) as f:
        g = json.load(f)
    w = TINY_SHARP
    pol = replace(w.policy, tree_tau=g["policy"]["tree_tau"], tree_max=g["policy"]["tree_max"])
    m = OracleModel(w.shape, weights_to_numpy(make_weights(w)))
    prompt = make_prompt(w)
    assert [int(t) for t in prompt] == g["prompt"]
    st = prefill(m, prompt, pol, 128)
    stats = ssd_generate(m, st, pol, w.gen_len - 1)
    assert st.tokens[len(prompt):] == g["tokens"]
    assert (stats.rounds, stats.drafted, stats.accepted, stats.side_rows, stats.side_accepted) == \
        (g["rounds"], g["drafted"], g["accepted"], g["side_rows"], g["side_accepted"])
    assert [len(r.emitted) for r in stats.records] == g["emitted_per_round"]
    assert g["side_accepted"] > 0
    ar = prefill(m, prompt, pol, 128)
    ar_generate(m, ar, pol, w.gen_len - 1)
    assert ar.tokens == st.tokens
