"""The debug build of the library (-DSSD_DEBUG_CHECKS): device-side bounds
checks on token ids, K/V positions and pass row counts, and a canary after
every workspace of a context.

The tiny and the small grouped-query models decode (prefill, self-speculative
generation with skip and exit drafting, dynamic verification, autoregressive
decoding, a rewind) in a child process that loads the debug build; no bounds
check may fire (any would surface as an error of the next call) and every
canary must still hold its pattern.  The outputs must also equal those of
the release build, which the parent process computes.
"""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import torch
from synthetic import TINY, make_prompt, make_weights
from synthetic.configs import Policy
from tests.gpu_util import to_device_weights
from tests.test_gpu_model import SMALL_GQA
import self_speculative_decoding_gb300 as ssd

out = {}
for w, pols in ((TINY, [Policy(mode="skip", skip=(2,), d_max=4, tau=None),
                        Policy(mode="exit", exit_layer=1, d_max=6, tau=None),
                        Policy(mode="skip", skip=(2,), d_max=4, tau=None, tree_tau=1.0, tree_max=3)]),
                (SMALL_GQA, [Policy(mode="skip", skip=(2, 3), d_max=8, tau=None),
                             Policy(mode="exit", exit_layer=2, d_max=6, temperature=0.6, seed=3)])):
    wts = make_weights(w, dtype="bf16", lm_head_scale=10.0, random_gains=True)
    ctx = ssd.SSDContext(w.shape, to_device_weights(wts), max_seq=192)
    for i, pol in enumerate(pols):
        ctx.set_policy(pol)
        prompt = make_prompt(w, 20)
        first = ctx.prefill(prompt)
        toks, _ = ctx.generate(50)
        ctx.rewind(len(prompt) + 10)
        more, _ = ctx.generate(20)
        ctx.prefill(prompt)
        ar, _ = ctx.decode_ar(30)
        out[f"{w.name}/{i}"] = [first, toks, more, ar]
    checked, bad = ctx.debug_canaries()
    out[f"{w.name}/canaries"] = [checked, bad]
    ctx.close()
print("RESULT " + json.dumps(out))
"""


def _run(env_lib):
    env = dict(os.environ)
    if env_lib:
        env["SSD_LIBSSD"] = env_lib
    else:
        env.pop("SSD_LIBSSD", None)
    p = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True,
                       text=True, timeout=900)
    assert p.returncode == 0, p.stdout[-2000:] + p.stderr[-4000:]
    line = next(l for l in p.stdout.splitlines() if l.startswith("RESULT "))
    return json.loads(line[len("RESULT "):])


def test_debug_build_runs_clean_and_matches_release():
    import __graft_entry__ as g
    g.build()
    from self_speculative_decoding_gb300 import build as b
    dbg = b.build_variant("debug", ["-DSSD_DEBUG_CHECKS=1"])
    got = _run(dbg)
    ref = _run(None)
    for name in ("tiny-L4-d256", "small-gqa"):
        checked, bad = got[f"{name}/canaries"]
        assert checked > 20 and bad == 0, (name, checked, bad)
        assert ref[f"{name}/canaries"] == [0, 0]      # the release build has none
    for k in ref:
        if not k.endswith("canaries"):
            assert got[k] == ref[k], k
