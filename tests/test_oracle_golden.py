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
