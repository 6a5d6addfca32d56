"""The C-ABI library builds, loads, and exports every function the headers declare."""

import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in ("ssd.h", "ssd_ops.h"):
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(ssd_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from self_speculative_decoding_gb300 import build as b
    b.build()
    from self_speculative_decoding_gb300 import _abi
    return _abi.load()


def test_headers_declare_the_boundary():
    names = _declared()
    for must in ("ssd_create", "ssd_destroy", "ssd_set_policy", "ssd_prefill", "ssd_draft",
                 "ssd_verify", "ssd_accept", "ssd_score_masks", "ssd_generate", "ssd_decode_ar",
                 "ssd_last_error"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    from self_speculative_decoding_gb300 import _abi
    assert set(_declared()) <= set(_abi.EXPORTED)


def test_null_context_is_an_error_not_a_crash(lib):
    assert lib.ssd_destroy(None) == 0
    assert lib.ssd_set_policy(None, None) == 1
    assert lib.ssd_generate(None, 4, None, None) == 1
    assert lib.ssd_last_error(None) == b"null context"


def test_op_argument_checks_need_no_gpu(lib):
    # invalid sizes are rejected on the host before any launch
    assert lib.ssd_op_linear(None, 16, 32, None, 1, None, None) == 1
    assert lib.ssd_op_attention(None, 0, 0, None, None, 64, 4, 4, 64, 1e4, None, None) == 1
    assert b"M" in lib.ssd_ops_last_error() or b"sizes" in lib.ssd_ops_last_error()
