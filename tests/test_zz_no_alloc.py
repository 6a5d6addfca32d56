"""ssd_op_linear_noalloc: the projection GEMV for callers that cannot allocate.

Callers whose device memory is already fully owned by their own allocator, or
whose latency-critical step must not allocate, call this entry point instead
of ssd_op_linear: it takes its scratch from a fixed array the library reserves
on the GPU.  Its output must agree with the allocating entry point's on two
calls in a row (the second call reuses the array the first left behind).
"""

import ctypes as C

import numpy as np
import pytest
import torch

from tests.gpu_util import rand_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from self_speculative_decoding_gb300 import _abi
    return _abi.lib()


@pytest.mark.parametrize("R,K,M", [(4096, 4096, 1), (8192, 11008, 13), (48, 704, 3)])
def test_noalloc_linear_matches_allocating_entry_point(lib, R, K, M):
    import self_speculative_decoding_gb300 as ssd
    W, _ = rand_bf16((R, K), seed=R + K + M)
    Wp = ssd.pack_weight(W)
    act, _ = rand_bf16((M, K), seed=M, std=1.0)
    ref = ssd.ops.linear(Wp, act)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        y = torch.full((M, R), float("nan"), dtype=torch.float32, device="cuda")
        st = lib.ssd_op_linear_noalloc(Wp.data_ptr(), R, K, act.data_ptr(), M, y.data_ptr(),
                                       stream)
        assert st == 0, lib.ssd_op_linear_noalloc_last_error()
        torch.cuda.synchronize()
        np.testing.assert_allclose(y.cpu().numpy(), ref.cpu().numpy(), rtol=1e-4,
                                   atol=1e-4 * np.sqrt(K) * 0.02)


def test_noalloc_linear_rejects_shapes_beyond_its_scratch(lib):
    W = torch.zeros(8208, 32, dtype=torch.bfloat16, device="cuda")
    act = torch.zeros(1, 32, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(1, 8208, dtype=torch.float32, device="cuda")
    st = lib.ssd_op_linear_noalloc(W.data_ptr(), 8208, 32, act.data_ptr(), 1, y.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert st == 3  # SSD_ERR_CAPACITY
    assert b"8192" in lib.ssd_op_linear_noalloc_last_error()
