"""ctypes declarations of the libssd C-ABI (include/ssd.h, include/ssd_ops.h).

Argument marshalling only: every step of the decoding path runs in the
library's CUDA kernels.  Importing this module loads the in-tree
``libssd.so`` and raises if it is missing — there is no fallback path.
"""

from __future__ import annotations

import ctypes as C
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libssd.so")

SSD_OK = 0
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "STATE", 3: "CAPACITY", 4: "OOM", 5: "CUDA",
                6: "TIMEOUT"}
SSD_MODE_SKIP = 0
SSD_MODE_EXIT = 1
SSD_DTYPE_BF16 = 0
SSD_DTYPE_FP32 = 1


class SsdConfig(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("d_model", C.c_int32), ("n_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn_dim", C.c_int32),
                ("vocab", C.c_int32), ("rope_theta", C.c_float), ("norm_eps", C.c_float),
                ("max_seq", C.c_int32), ("max_draft", C.c_int32), ("max_score_rows", C.c_int32),
                ("dtype", C.c_int32)]


class SsdLayerWeights(C.Structure):
    _fields_ = [("attn_norm", C.c_void_p), ("wqkv", C.c_void_p), ("wo", C.c_void_p),
                ("mlp_norm", C.c_void_p), ("w_gate", C.c_void_p), ("w_up", C.c_void_p),
                ("w_down", C.c_void_p)]


class SsdWeights(C.Structure):
    _fields_ = [("tok_embed", C.c_void_p), ("final_norm", C.c_void_p), ("lm_head", C.c_void_p),
                ("layers", C.POINTER(SsdLayerWeights))]


class SsdPolicy(C.Structure):
    _fields_ = [("mode", C.c_int32), ("skip_mask", C.c_uint64 * 4), ("exit_layer", C.c_int32),
                ("d_max", C.c_int32), ("tau", C.c_float), ("temperature", C.c_float),
                ("seed", C.c_uint64), ("skip_attn_mask", C.c_uint64 * 4),
                ("skip_mlp_mask", C.c_uint64 * 4), ("tree_tau", C.c_float),
                ("tree_max", C.c_int32)]


class SsdSwiftParams(C.Structure):
    _fields_ = [("skip_count", C.c_int32), ("lo_layer", C.c_int32), ("window", C.c_int32),
                ("candidates", C.c_int32), ("max_steps", C.c_int32), ("patience", C.c_int32),
                ("target", C.c_float), ("seed", C.c_uint64)]


class SsdSwiftReport(C.Structure):
    _fields_ = [("steps", C.c_int32), ("stopped_by", C.c_int32), ("final_mask", C.c_uint64 * 4),
                ("rounds", C.c_int64), ("drafted", C.c_int64), ("accepted", C.c_int64),
                ("emitted", C.c_int64), ("opt_seconds", C.c_double), ("total_seconds", C.c_double)]


class SsdStats(C.Structure):
    _fields_ = [("rounds", C.c_int64), ("drafted", C.c_int64), ("accepted", C.c_int64),
                ("emitted", C.c_int64), ("draft_steps", C.c_int64),
                ("kernel_launches", C.c_int64), ("bytes_streamed", C.c_double),
                ("draft_ms", C.c_double), ("verify_ms", C.c_double), ("ar_ms", C.c_double),
                ("side_rows", C.c_int64), ("side_accepted", C.c_int64)]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_}


class SsdKernelTimes(C.Structure):
    _fields_ = [("ms", C.c_double * 8), ("bytes", C.c_double * 8), ("launches", C.c_int64 * 8)]

    CLASSES = ("qkv", "attention", "o_proj", "gate_up", "down", "lm_head", "control",
               "attention+o_proj")

    def as_dict(self) -> dict:
        return {name: {"ms": self.ms[i], "bytes": self.bytes[i], "launches": self.launches[i]}
                for i, name in enumerate(self.CLASSES)}


class SsdRowStats(C.Structure):
    _fields_ = [("top1", C.c_int32), ("top2", C.c_int32), ("sample", C.c_int32),
                ("pad", C.c_int32), ("z1", C.c_float), ("z2", C.c_float), ("lse", C.c_float),
                ("conf", C.c_float), ("lse_t", C.c_float), ("pad2", C.c_float * 3)]


assert C.sizeof(SsdRowStats) == 48

_P = C.c_void_p
_I = C.c_int32
_SIGS = {
    "ssd_pack_weight": [_P, _P, _I, _I, _P],
    "ssd_create": [C.POINTER(SsdConfig), C.POINTER(SsdWeights), _P, C.POINTER(_P)],
    "ssd_destroy": [_P],
    "ssd_set_policy": [_P, C.POINTER(SsdPolicy)],
    "ssd_prefill": [_P, C.POINTER(_I), _I, C.POINTER(_I)],
    "ssd_draft": [_P, C.POINTER(_I), C.POINTER(C.c_float), C.POINTER(_I)],
    "ssd_verify": [_P, C.POINTER(C.c_float)],
    "ssd_accept": [_P, C.POINTER(_I), C.POINTER(_I)],
    "ssd_generate": [_P, _I, C.POINTER(_I), C.POINTER(SsdStats)],
    "ssd_decode_ar": [_P, _I, C.POINTER(_I), C.POINTER(SsdStats)],
    "ssd_score_masks": [_P, C.POINTER(C.c_uint64), _I, _I, C.POINTER(C.c_float), C.POINTER(_I)],
    "ssd_decode_lossy": [_P, _I, C.POINTER(_I), C.POINTER(SsdStats)],
    "ssd_layer_features": [_P, _I, C.POINTER(_I), C.POINTER(C.c_float), C.POINTER(C.c_float)],
    "ssd_rewind": [_P, _I],
    "ssd_get_tokens": [_P, C.POINTER(_I), _I, C.POINTER(_I)],
    "ssd_set_timeout_ms": [_P, _I],
    "ssd_set_device_loop": [_P, _I, C.POINTER(C.c_int32)],
    "ssd_debug_fail_alloc": [_I],
    "ssd_swift_generate": [_P, C.POINTER(SsdSwiftParams), _I, _P, _P, _P, _P, _I,
                           C.POINTER(SsdSwiftReport)],
    "ssd_profile_decode": [_P, _I, C.POINTER(SsdKernelTimes)],
    "ssd_profile_kernels": [_P, _I, C.POINTER(SsdKernelTimes)],
    "ssd_debug_canaries": [_P, C.POINTER(C.c_int32), C.POINTER(C.c_int32)],
    "ssd_last_error": [_P],
    "ssd_op_linear": [_P, _I, _I, _P, _I, _P, _P],
    "ssd_op_rmsnorm_linear": [_P, _I, _I, _P, _P, C.c_float, _I, _P, _P],
    "ssd_op_residual_linear": [_P, _I, _I, _P, _I, _P, _P],
    "ssd_op_swiglu": [_P, _P, _I, _I, _P, _P, C.c_float, _I, _P, _P],
    "ssd_op_attention": [_P, _I, _I, _P, _P, _I, _I, _I, _I, C.c_float, _P, _P],
    "ssd_op_lm_head": [_P, _I, _I, _P, _P, C.c_float, _I, C.c_float, C.c_uint64, _I, _I, _I, _P,
                       _P, _P],
    "ssd_op_accept_stochastic": [_P, _P, _P, _I, _I, C.c_float, C.c_uint64, _I, _I, _P, _P, _P],
    "ssd_op_philox": [_P, _I, C.c_uint64, _P, _P],
    "ssd_ops_last_error": [],
    "ssd_op_linear_noalloc": [_P, _I, _I, _P, _I, _P, _P],
    "ssd_op_wait_selftest": [_I, C.POINTER(C.c_int32), _P],
    "ssd_op_linear_rows": [_P, _P, _I, _I, _P, _I, _I, _P, _P, _P],
    "ssd_op_score_attention": [_P, _P, _I, _I, _I, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P],
    "ssd_op_linear_noalloc_last_error": [],
}

EXPORTED = tuple(_SIGS)


def load(path: Optional[str] = None) -> C.CDLL:
    """The library at ``path``; default: $SSD_LIBSSD if set (another build of
    the library, e.g. the debug build), else the in-tree libssd.so."""
    path = path or os.environ.get("SSD_LIBSSD") or LIB_PATH
    if not os.path.exists(path):
        raise ImportError(
            f"libssd.so not found at {path}: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    lib = C.CDLL(path)
    for name, args in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = C.c_char_p if name.endswith("last_error") else C.c_int
    return lib


_lib = None


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        _lib = load()
    return _lib


class SSDError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status
