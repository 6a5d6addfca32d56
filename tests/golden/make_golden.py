"""Writes the oracle's regression fixtures for the tiny fp32 workload.

Calls only ``oracle`` and ``synthetic``: the stored values are the oracle's
own output on seeded inputs, kept so that a later change to the oracle's
arithmetic shows up as a diff.  Run from the repository root:

    python tests/golden/make_golden.py
"""

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from dataclasses import replace  # noqa: E402

from synthetic import TINY, make_weights, weights_to_numpy, make_prompt  # noqa: E402
from synthetic.configs import TINY_SHARP  # noqa: E402
from oracle import OracleModel, prefill, ar_generate, ssd_generate  # noqa: E402

# dynamic verification on the sharpened tiny model: every kept draft sends
# the draft's second choice as a sibling, at most 4 per round
TREE_POLICY = replace(TINY_SHARP.policy, tree_tau=1.0, tree_max=4)


def main():
    m = OracleModel(TINY.shape, weights_to_numpy(make_weights(TINY)))
    prompt = make_prompt(TINY)
    st = prefill(m, prompt, TINY.policy, 128)
    ar_generate(m, st, TINY.policy, TINY.gen_len - 1)
    st2 = prefill(m, prompt, TINY.policy, 128)
    stats = ssd_generate(m, st2, TINY.policy, TINY.gen_len - 1)
    out = {
        "workload": TINY.name,
        "prompt": [int(t) for t in prompt],
        "ar_greedy_tokens": st.tokens[len(prompt):],
        "ssd_greedy_tokens": st2.tokens[len(prompt):],
        "ssd_rounds": stats.rounds,
        "ssd_drafted": stats.drafted,
        "ssd_accepted": stats.accepted,
    }
    with open(os.path.join(HERE, "tiny_fp32_greedy.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")

    w = TINY_SHARP
    m = OracleModel(w.shape, weights_to_numpy(make_weights(w)))
    prompt = make_prompt(w)
    st = prefill(m, prompt, TREE_POLICY, 128)
    stats = ssd_generate(m, st, TREE_POLICY, w.gen_len - 1)
    out = {
        "workload": w.name,
        "policy": {"skip": list(TREE_POLICY.skip), "d_max": TREE_POLICY.d_max,
                   "tree_tau": TREE_POLICY.tree_tau, "tree_max": TREE_POLICY.tree_max},
        "prompt": [int(t) for t in prompt],
        "tokens": st.tokens[len(prompt):],
        "rounds": stats.rounds,
        "drafted": stats.drafted,
        "accepted": stats.accepted,
        "side_rows": stats.side_rows,
        "side_accepted": stats.side_accepted,
        "emitted_per_round": [len(r.emitted) for r in stats.records],
    }
    with open(os.path.join(HERE, "tiny_sharp_tree.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
