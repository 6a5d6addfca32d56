"""ssd_op_linear_noalloc: the projection GEMV for callers that cannot allocate.

Callers whose device memory is already fully owned by their own allocator, or
whose latency-critical step must not allocate, call this entry point instead
of ssd_op_linear: it takes its scratch from a fixed array the library reserves
on the GPU.  Both entry points run the same kernel with the same partition and
the same summation order, so their outputs must be bit-identical, on two calls
in a row and after a call of another shape has left its own partial sums and
counters in the shared array.
"""

import pytest
import torch

from tests.gpu_util import rand_bf16

pytestmark = pytest.mark.gpu

# (R, K, M).  48 x 704 and 6368 x 1024 split row groups across CTAs and so use
# the fixed array; 6368 rows (398 row groups, two partial segments each, about
# 0.8 MiB) is the largest scratch use under the 8192-row limit, since 8192 rows
# and 4096 rows are partitioned into whole row groups per CTA.
SHAPES = [(4096, 4096, 1), (8192, 11008, 13), (48, 704, 3), (6368, 1024, 5)]


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from self_speculative_decoding_gb300 import _abi
    return _abi.lib()


def _case(ssd, R, K, M):
    W, _ = rand_bf16((R, K), seed=R + K + M)
    Wp = ssd.pack_weight(W)
    act, _ = rand_bf16((M, K), seed=M, std=1.0)
    return Wp, act, ssd.ops.linear(Wp, act)


def _noalloc(lib, Wp, act):
    R, K = Wp.shape
    M = act.shape[0]
    y = torch.full((M, R), float("nan"), dtype=torch.float32, device="cuda")
    st = lib.ssd_op_linear_noalloc(Wp.data_ptr(), R, K, act.data_ptr(), M, y.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.ssd_op_linear_noalloc_last_error()
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("R,K,M", SHAPES)
def test_noalloc_linear_matches_allocating_entry_point(lib, R, K, M):
    import self_speculative_decoding_gb300 as ssd
    Wp, act, ref = _case(ssd, R, K, M)
    for _ in range(2):
        assert torch.equal(_noalloc(lib, Wp, act), ref)


def test_noalloc_linear_after_a_call_of_another_shape(lib):
    # every call reuses the one array: a call must not depend on what a call
    # with a different partition left in it
    import self_speculative_decoding_gb300 as ssd
    cases = [_case(ssd, *s) for s in SHAPES]
    for order in ([2, 3, 2], [3, 2, 3], [0, 3, 1, 2]):
        for i in order:
            Wp, act, ref = cases[i]
            assert torch.equal(_noalloc(lib, Wp, act), ref), SHAPES[i]


def test_noalloc_linear_rejects_shapes_beyond_its_scratch(lib):
    W = torch.zeros(8208, 32, dtype=torch.bfloat16, device="cuda")
    act = torch.zeros(1, 32, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(1, 8208, dtype=torch.float32, device="cuda")
    st = lib.ssd_op_linear_noalloc(W.data_ptr(), 8208, 32, act.data_ptr(), 1, y.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert st == 3  # SSD_ERR_CAPACITY
    assert b"8192" in lib.ssd_op_linear_noalloc_last_error()
