"""Failure detection without faulting the GPU.

* The device's bounded waits (an mbarrier wait and a global-counter wait,
  the two kinds the kernels use) are made to run out against conditions
  nothing fulfils: both give up and report, and the call returns promptly.
* An injected allocation failure in ssd_create (host-side fault injection)
  gives SSD_ERR_OOM at every position, and a context created afterwards
  works.
* Calls in the wrong state and over capacity fail with their status and
  leave the context usable (see also test_gpu_model's state tests).
* The statistics carry the device time of draft, verify and AR passes (the
  inputs of SWIFT's cost coefficient c).
"""

import time

import pytest
import torch

from synthetic import TINY, make_weights, make_prompt
from synthetic.configs import Policy
from tests.gpu_util import to_device_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssd():
    import __graft_entry__ as g
    g.build()
    import self_speculative_decoding_gb300 as m
    return m


def test_bounded_device_waits_give_up_and_report(ssd):
    t0 = time.perf_counter()
    assert ssd.ops.wait_selftest(4096) == 3
    assert time.perf_counter() - t0 < 5.0
    assert ssd.ops.wait_selftest(1) == 3
    # the context is still healthy afterwards
    x = torch.ones(16, device="cuda")
    torch.cuda.synchronize()
    assert float(x.sum()) == 16.0


@pytest.mark.parametrize("n", [0, 1, 5, 12, 20])
def test_injected_allocation_failure(ssd, n):
    from self_speculative_decoding_gb300 import SSDError, _abi
    wts = to_device_weights(make_weights(TINY, dtype="bf16"))
    _abi.lib().ssd_debug_fail_alloc(n)
    with pytest.raises(SSDError, match="OOM"):
        ssd.SSDContext(TINY.shape, wts, max_seq=128, max_score_rows=32)
    _abi.lib().ssd_debug_fail_alloc(-1)
    ctx = ssd.SSDContext(TINY.shape, wts, max_seq=128, max_score_rows=32)
    ctx.set_policy(Policy(mode="skip", skip=(2,), d_max=3))
    ctx.prefill(make_prompt(TINY, 8))
    toks, _ = ctx.generate(10)
    assert len(toks) == 10
    ctx.close()


def test_misaligned_weight_refused(ssd):
    # every weight pointer must be 16-byte aligned (vector loads, bulk copies)
    from self_speculative_decoding_gb300 import SSDError
    wts = to_device_weights(make_weights(TINY, dtype="bf16"))
    g = wts["layers"][1]["mlp_norm"]
    buf = torch.zeros(g.numel() + 4, dtype=torch.float32, device="cuda")
    buf[1:1 + g.numel()] = g
    wts["layers"][1]["mlp_norm"] = buf[1:1 + g.numel()]          # 4 bytes off
    with pytest.raises(SSDError, match="INVALID_ARG"):
        ssd.SSDContext(TINY.shape, wts, max_seq=128)


def test_pass_timing_statistics(ssd):
    wts = to_device_weights(make_weights(TINY, dtype="bf16", lm_head_scale=10.0))
    ctx = ssd.SSDContext(TINY.shape, wts, max_seq=128)
    ctx.set_policy(Policy(mode="skip", skip=(2,), d_max=3, tau=None))
    ctx.set_device_loop(False)   # per-pass device times come from the host-driven loop
    ctx.prefill(make_prompt(TINY, 8))
    _, st = ctx.generate(20)
    assert st["draft_steps"] > 0 and st["draft_ms"] > 0 and st["verify_ms"] > 0
    ctx.rewind(9)
    _, ar = ctx.decode_ar(20)
    assert ar["ar_ms"] > 0
    ctx.close()
