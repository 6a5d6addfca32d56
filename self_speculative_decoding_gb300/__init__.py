"""Layer-skipping self-speculative decoding on one GB300 (sm_103a).

Python binding of the libssd C-ABI.  PyTorch only provides device memory and
streams; every step of the path (embedding, the fused RMSNorm + projections,
attention with KV append, the LM head with its row summary, drafting,
verification, acceptance and rollback) runs in the library's CUDA kernels.
The functions here marshal arguments and raise on error; there is no CPU or
PyTorch fallback.
"""

from __future__ import annotations

import ctypes as C
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

from . import _abi
from ._abi import (SSDError, SsdConfig, SsdLayerWeights, SsdPolicy, SsdRowStats, SsdStats,
                   SsdSwiftParams, SsdSwiftReport, SsdWeights, SSD_MODE_EXIT, SSD_MODE_SKIP)

__all__ = ["SSDContext", "SSDError", "ops", "pack_weight", "pack_weights", "policy_struct",
           "stream_handle"]

MATRICES = ("wqkv", "wo", "w_gate", "w_up", "w_down")


def pack_weight(W: torch.Tensor) -> torch.Tensor:
    """Row-major bf16 [R, K] CUDA matrix -> the library's packed layout (a new
    tensor of the same shape and size)."""
    if W.dtype != torch.bfloat16 or W.dim() != 2:
        raise ValueError("pack_weight expects a 2-D bf16 tensor")
    out = torch.empty_like(W)
    st = _lib().ssd_pack_weight(_ptr(W), _ptr(out), W.shape[0], W.shape[1], stream_handle())
    if st != _abi.SSD_OK:
        raise SSDError(st, _lib().ssd_ops_last_error().decode())
    return out


def pack_weights(wts: Dict, release: bool = False) -> Dict:
    """A copy of a weight dict with every projection matrix packed.  With
    ``release`` the row-major matrices are dropped from ``wts`` as they are
    packed, so that peak memory is the model plus one matrix."""
    out = {k: v for k, v in wts.items() if k not in ("layers", "lm_head")}
    out["lm_head"] = pack_weight(wts["lm_head"])
    if release:
        wts["lm_head"] = None
    out["layers"] = []
    for lw in wts["layers"]:
        nl = {k: v for k, v in lw.items() if k not in MATRICES}
        for k in MATRICES:
            nl[k] = pack_weight(lw[k])
            if release:
                lw[k] = None
        out["layers"].append(nl)
    out["packed"] = True
    return out


def _lib():
    return _abi.lib()


def stream_handle(stream: Optional[torch.cuda.Stream] = None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def policy_struct(policy) -> SsdPolicy:
    """Marshals a policy (attributes mode, skip, skip_attn, skip_mlp,
    exit_layer, d_max, tau, temperature, seed, tree_tau, tree_max — e.g.
    ``synthetic.Policy``) into ``ssd_policy``."""
    p = SsdPolicy()
    p.mode = SSD_MODE_SKIP if policy.mode == "skip" else SSD_MODE_EXIT
    for field, mask in (("skip", p.skip_mask), ("skip_attn", p.skip_attn_mask),
                        ("skip_mlp", p.skip_mlp_mask)):
        for l in getattr(policy, field, ()):
            mask[l // 64] |= 1 << (l % 64)
    p.exit_layer = int(getattr(policy, "exit_layer", -1))
    p.d_max = int(policy.d_max)
    tau = getattr(policy, "tau", None)
    p.tau = -1.0 if tau is None else float(tau)
    p.temperature = float(getattr(policy, "temperature", 0.0))
    p.seed = int(getattr(policy, "seed", 0)) & ((1 << 64) - 1)
    tree_tau = getattr(policy, "tree_tau", None)
    p.tree_tau = 0.0 if tree_tau is None else float(tree_tau)
    p.tree_max = int(getattr(policy, "tree_max", 0))
    return p


class SSDContext:
    """One model on one GPU: owns the library context (KV cache, workspaces,
    graphs); borrows the weight tensors, which must outlive it."""

    def __init__(self, shape, weights: Dict, max_seq: int, max_draft: int = 15,
                 max_score_rows: int = 0, stream: Optional[torch.cuda.Stream] = None):
        self.shape = shape
        # fp32 models: every matrix fp32 and row-major (not packed); bf16
        # models: projection matrices bf16 in the packed layout
        self.fp32 = all(lw[k].dtype == torch.float32 for lw in weights["layers"] for k in MATRICES)
        if self.fp32:
            if weights["tok_embed"].dtype != torch.float32 or weights["lm_head"].dtype != torch.float32:
                raise ValueError("an fp32 model needs fp32 tok_embed and lm_head")
        elif not weights.get("packed"):
            raise ValueError("bf16 weights must be packed with pack_weights() first")
        self._weights = weights  # keep the tensors alive
        cfg = SsdConfig(shape.n_layers, shape.d_model, shape.n_heads, shape.n_kv_heads,
                        shape.head_dim, shape.ffn_dim, shape.vocab, shape.rope_theta,
                        shape.norm_eps, max_seq, max_draft, max_score_rows,
                        _abi.SSD_DTYPE_FP32 if self.fp32 else _abi.SSD_DTYPE_BF16)
        self._layers = (SsdLayerWeights * shape.n_layers)()
        for i, lw in enumerate(weights["layers"]):
            for k in MATRICES:
                if lw[k].dtype != (torch.float32 if self.fp32 else torch.bfloat16):
                    raise ValueError(f"layer {i} {k}: every matrix must have the model's dtype")
            self._layers[i] = SsdLayerWeights(_ptr(lw["attn_norm"]), _ptr(lw["wqkv"]),
                                              _ptr(lw["wo"]), _ptr(lw["mlp_norm"]),
                                              _ptr(lw["w_gate"]), _ptr(lw["w_up"]),
                                              _ptr(lw["w_down"]))
        w = SsdWeights(_ptr(weights["tok_embed"]), _ptr(weights["final_norm"]),
                       _ptr(weights["lm_head"]), self._layers)
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        h = C.c_void_p()
        st = _lib().ssd_create(C.byref(cfg), C.byref(w), stream_handle(self.stream), C.byref(h))
        if st != _abi.SSD_OK:
            raise SSDError(st, "ssd_create failed")
        self._h = h
        self.max_seq = max_seq
        self.d_max = 0
        self.vocab = shape.vocab

    # ------------------------------------------------------------------
    def _check(self, st: int):
        if st != _abi.SSD_OK:
            raise SSDError(st, _lib().ssd_last_error(self._h).decode())

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib().ssd_destroy(self._h)
            self._h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------------
    def set_policy(self, policy):
        self._check(_lib().ssd_set_policy(self._h, C.byref(policy_struct(policy))))
        self.d_max = int(policy.d_max)

    def prefill(self, tokens: Sequence[int]) -> int:
        arr = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        first = C.c_int32()
        self._check(_lib().ssd_prefill(self._h, arr.ctypes.data_as(C.POINTER(C.c_int32)),
                                       len(arr), C.byref(first)))
        return int(first.value)

    def draft(self) -> Tuple[List[int], List[float]]:
        out = (C.c_int32 * max(self.d_max, 1))()
        conf = (C.c_float * (self.d_max + 1))()
        d = C.c_int32()
        self._check(_lib().ssd_draft(self._h, out, conf, C.byref(d)))
        n_steps = min(d.value + 1, self.d_max) if self.d_max else 0
        return [out[i] for i in range(d.value)], [conf[i] for i in range(n_steps)]

    def verify(self, want_logits: bool = True, d: Optional[int] = None) -> Optional[np.ndarray]:
        if not want_logits:
            self._check(_lib().ssd_verify(self._h, None))
            return None
        buf = np.zeros(((self.d_max + 1), self.vocab), dtype=np.float32)
        self._check(_lib().ssd_verify(self._h, buf.ctypes.data_as(C.POINTER(C.c_float))))
        return buf if d is None else buf[: d + 1]

    def accept(self) -> List[int]:
        out = (C.c_int32 * (self.d_max + 1))()
        n = C.c_int32()
        self._check(_lib().ssd_accept(self._h, out, C.byref(n)))
        return [out[i] for i in range(n.value)]

    def generate(self, n_tokens: int, want_tokens: bool = True):
        out = np.zeros(max(n_tokens, 1), dtype=np.int32)
        stats = SsdStats()
        ptr = out.ctypes.data_as(C.POINTER(C.c_int32)) if want_tokens else None
        self._check(_lib().ssd_generate(self._h, n_tokens, ptr, C.byref(stats)))
        return (out[:n_tokens].tolist() if want_tokens else None), stats.as_dict()

    def decode_ar(self, n_tokens: int, want_tokens: bool = True):
        out = np.zeros(max(n_tokens, 1), dtype=np.int32)
        stats = SsdStats()
        ptr = out.ctypes.data_as(C.POINTER(C.c_int32)) if want_tokens else None
        self._check(_lib().ssd_decode_ar(self._h, n_tokens, ptr, C.byref(stats)))
        return (out[:n_tokens].tolist() if want_tokens else None), stats.as_dict()

    def decode_lossy(self, n_tokens: int, want_tokens: bool = True):
        """Lossy early exit (ssd_decode_lossy): the draft layers alone decide."""
        out = np.zeros(max(n_tokens, 1), dtype=np.int32)
        stats = SsdStats()
        ptr = out.ctypes.data_as(C.POINTER(C.c_int32)) if want_tokens else None
        self._check(_lib().ssd_decode_lossy(self._h, n_tokens, ptr, C.byref(stats)))
        return (out[:n_tokens].tolist() if want_tokens else None), stats.as_dict()

    def layer_features(self, min_layer: int = 0):
        """AdaInfer exit features of one AR step (ssd_layer_features):
        (top1, top_prob, gap) lists over layers min_layer .. L-1."""
        nl = self.shape.n_layers - min_layer
        t = np.zeros(max(nl, 1), dtype=np.int32)
        p = np.zeros(max(nl, 1), dtype=np.float32)
        g = np.zeros(max(nl, 1), dtype=np.float32)
        self._check(_lib().ssd_layer_features(self._h, min_layer,
                                              t.ctypes.data_as(C.POINTER(C.c_int32)),
                                              p.ctypes.data_as(C.POINTER(C.c_float)),
                                              g.ctypes.data_as(C.POINTER(C.c_float))))
        return t[:nl].tolist(), p[:nl].tolist(), g[:nl].tolist()

    def score_masks(self, masks: Sequence[Sequence[int]], N: int):
        K = len(masks)
        words = np.zeros((K, 4), dtype=np.uint64)
        for k, m in enumerate(masks):
            for l in m:
                words[k, l // 64] |= np.uint64(1 << (l % 64))
        scores = np.zeros(K, dtype=np.float32)
        best = C.c_int32()
        self._check(_lib().ssd_score_masks(self._h, words.ctypes.data_as(C.POINTER(C.c_uint64)),
                                           K, N, scores.ctypes.data_as(C.POINTER(C.c_float)),
                                           C.byref(best)))
        return scores, int(best.value)

    def rewind(self, n: int):
        self._check(_lib().ssd_rewind(self._h, n))

    def tokens(self) -> List[int]:
        n = C.c_int32()
        self._check(_lib().ssd_get_tokens(self._h, None, 0, C.byref(n)))
        buf = (C.c_int32 * max(n.value, 1))()
        self._check(_lib().ssd_get_tokens(self._h, buf, n.value, C.byref(n)))
        return [buf[i] for i in range(n.value)]

    def profile_decode(self, n_steps: int) -> dict:
        """Per-kernel-class device time (CUDA events on the context stream)."""
        out = _abi.SsdKernelTimes()
        self._check(_lib().ssd_profile_decode(self._h, n_steps, C.byref(out)))
        return out.as_dict()

    def debug_canaries(self) -> Tuple[int, int]:
        """(canaries checked, canary bytes overwritten); (0, 0) in release
        builds (ssd_debug_canaries)."""
        n, bad = C.c_int32(0), C.c_int32(0)
        self._check(_lib().ssd_debug_canaries(self._h, C.byref(n), C.byref(bad)))
        return n.value, bad.value

    def profile_kernels(self, reps: int = 5) -> dict:
        """Per-kernel-class device time with each class's launches of one
        autoregressive step captured as a graph and replayed (ssd.h:
        ssd_profile_kernels); launches = per step."""
        out = _abi.SsdKernelTimes()
        self._check(_lib().ssd_profile_kernels(self._h, reps, C.byref(out)))
        return out.as_dict()

    def set_timeout_ms(self, ms: int):
        self._check(_lib().ssd_set_timeout_ms(self._h, ms))

    def swift_generate(self, params, n_tokens: int, trace_cap: int = 0):
        """SWIFT layer-set optimisation while generating n_tokens (ssd.h:
        ssd_swift_generate).  ``params`` has the fields of ssd_swift_params
        (e.g. a ``types.SimpleNamespace``).  Returns (tokens,
        report dict, trace) with trace = (candidate masks [steps][K] as
        layer tuples, scores [steps][K], winners [steps]) for the first
        ``trace_cap`` steps."""
        p = SsdSwiftParams()
        for f, _ in SsdSwiftParams._fields_:
            setattr(p, f, getattr(params, f))
        K = int(params.candidates)
        out = np.zeros(max(n_tokens, 1), dtype=np.int32)
        tm = np.zeros((max(trace_cap, 1), K, 4), dtype=np.uint64)
        tsc = np.zeros((max(trace_cap, 1), K), dtype=np.float32)
        tb = np.zeros(max(trace_cap, 1), dtype=np.int32)
        rep = SsdSwiftReport()
        self._check(_lib().ssd_swift_generate(
            self._h, C.byref(p), n_tokens, out.ctypes.data, tm.ctypes.data, tsc.ctypes.data,
            tb.ctypes.data, trace_cap, C.byref(rep)))
        steps = min(rep.steps, trace_cap)
        L = self.shape.n_layers

        def layers(m):
            return tuple(l for l in range(L) if (int(m[l // 64]) >> (l % 64)) & 1)

        trace = ([[layers(tm[s, k]) for k in range(K)] for s in range(steps)],
                 tsc[:steps].tolist(), tb[:steps].tolist())
        report = {f: getattr(rep, f) for f, _ in SsdSwiftReport._fields_ if f != "final_mask"}
        report["final"] = layers(rep.final_mask)
        return out[:n_tokens].tolist(), report, trace

    def last_error(self) -> str:
        """The context's last error message (ssd_last_error)."""
        return _lib().ssd_last_error(self._h).decode()

    def set_device_loop(self, enable: bool) -> bool:
        """generate() as one graph launch with device-side control (True,
        the default where supported) or driven from the host (False; stats
        then carry per-pass device times).  Returns whether the device loop
        is in use.  Both produce the same tokens and counts."""
        active = C.c_int32(0)
        self._check(_lib().ssd_set_device_loop(self._h, 1 if enable else 0, C.byref(active)))
        return bool(active.value)


class _Ops:
    """Kernel-level entry points on torch CUDA tensors (ssd_ops.h)."""

    @staticmethod
    def _check(st: int):
        if st != _abi.SSD_OK:
            raise SSDError(st, _lib().ssd_ops_last_error().decode())

    def linear(self, W: torch.Tensor, act: torch.Tensor) -> torch.Tensor:
        R, K = W.shape
        M = act.shape[0]
        y = torch.empty(M, R, dtype=torch.float32, device=W.device)
        self._check(_lib().ssd_op_linear(_ptr(W), R, K, _ptr(act), M, _ptr(y), stream_handle()))
        return y

    def rmsnorm_linear(self, W, x, gain, eps) -> torch.Tensor:
        R, K = W.shape
        M = x.shape[0]
        y = torch.empty(M, R, dtype=torch.float32, device=W.device)
        self._check(_lib().ssd_op_rmsnorm_linear(_ptr(W), R, K, _ptr(x), _ptr(gain), eps, M,
                                                 _ptr(y), stream_handle()))
        return y

    def residual_linear(self, W, act, x) -> torch.Tensor:
        R, K = W.shape
        M = act.shape[0]
        self._check(_lib().ssd_op_residual_linear(_ptr(W), R, K, _ptr(act), M, _ptr(x),
                                                  stream_handle()))
        return x

    def swiglu(self, Wg, Wu, x, gain, eps) -> torch.Tensor:
        F, K = Wg.shape
        M = x.shape[0]
        u = torch.empty(M, F, dtype=torch.bfloat16, device=Wg.device)
        self._check(_lib().ssd_op_swiglu(_ptr(Wg), _ptr(Wu), F, K, _ptr(x), _ptr(gain), eps, M,
                                         _ptr(u), stream_handle()))
        return u

    def attention(self, qkv, pos0, k_cache, v_cache, H, Hkv, dh, theta) -> torch.Tensor:
        M = qkv.shape[0]
        max_seq = k_cache.shape[1]
        out = torch.empty(M, H * dh, dtype=torch.bfloat16, device=qkv.device)
        self._check(_lib().ssd_op_attention(_ptr(qkv), M, pos0, _ptr(k_cache), _ptr(v_cache),
                                            max_seq, H, Hkv, dh, theta, _ptr(out),
                                            stream_handle()))
        return out

    def lm_head(self, W, x, gain, eps, temperature=0.0, seed=0, round=0, stream_id=0, pos0=0,
                want_logits=True):
        V, D = W.shape
        M = x.shape[0]
        logits = torch.empty(M, V, dtype=torch.float32, device=W.device) if want_logits else None
        stats = torch.zeros(M, 12, dtype=torch.int32, device=W.device)
        self._check(_lib().ssd_op_lm_head(_ptr(W), V, D, _ptr(x), _ptr(gain), eps, M,
                                          temperature, seed, round, stream_id, pos0,
                                          _ptr(logits), _ptr(stats), stream_handle()))
        return logits, stats

    def accept_stochastic(self, P, Q, drafts, T, seed, round, n):
        d = drafts.shape[0]
        V = P.shape[1]
        emitted = torch.zeros(d + 1, dtype=torch.int32, device=P.device)
        n_em = torch.zeros(1, dtype=torch.int32, device=P.device)
        self._check(_lib().ssd_op_accept_stochastic(_ptr(P), _ptr(Q) if d else None,
                                                    _ptr(drafts) if d else None, d, V, T, seed,
                                                    round, n, _ptr(emitted), _ptr(n_em),
                                                    stream_handle()))
        return emitted, n_em

    LINEAR_ROWS_EPI = {"store": 0, "resid": 1, "swiglu": 2, "argmax": 3}

    def linear_rows(self, W, act, epi="store", W1=None, out=None, rowmap=None):
        """Many-row projection (ssd_op_linear_rows).  epi "store" -> fp32
        [T, R]; "resid" adds into out (fp32) at rows rowmap (or 0..T-1);
        "swiglu" -> bf16 [T, R] with W1 the up matrix; "argmax" -> int32 [T]."""
        R, K = W.shape
        T = act.shape[0]
        e = self.LINEAR_ROWS_EPI[epi]
        if out is None:
            if epi == "store":
                out = torch.empty(T, R, dtype=torch.float32, device=W.device)
            elif epi == "swiglu":
                out = torch.empty(T, R, dtype=torch.bfloat16, device=W.device)
            elif epi == "argmax":
                out = torch.empty(T, dtype=torch.int32, device=W.device)
            else:
                raise ValueError("epi 'resid' needs out")
        self._check(_lib().ssd_op_linear_rows(_ptr(W), _ptr(W1), R, K, _ptr(act), T, e, _ptr(out),
                                              _ptr(rowmap), stream_handle()))
        return out

    def score_attention(self, q, cand, N, split, k_cache, v_cache, wk, wv, H, Hkv, dh):
        """Window attention of candidate-mask scoring (ssd_op_score_attention);
        q bf16 [len(cand) N, H, dh]; returns bf16 [len(cand) N, H dh]."""
        nc = cand.shape[0]
        out = torch.empty(nc * N, H * dh, dtype=torch.bfloat16, device=q.device)
        self._check(_lib().ssd_op_score_attention(_ptr(q), _ptr(cand), nc, N, split,
                                                  _ptr(k_cache), _ptr(v_cache), k_cache.shape[1],
                                                  _ptr(wk), _ptr(wv), wk.shape[0], H, Hkv, dh,
                                                  _ptr(out),
                                                  stream_handle()))
        return out

    def wait_selftest(self, polls: int = 4096) -> int:
        """Device bounded waits made to run out (ssd_op_wait_selftest);
        returns the code (3 = both waits gave up and reported)."""
        code = C.c_int32(-1)
        self._check(_lib().ssd_op_wait_selftest(polls, C.byref(code), stream_handle()))
        return code.value

    def philox(self, ctr: torch.Tensor, key: int) -> torch.Tensor:
        out = torch.empty_like(ctr)
        self._check(_lib().ssd_op_philox(_ptr(ctr), ctr.shape[0], key, _ptr(out),
                                         stream_handle()))
        return out


ops = _Ops()


def row_stats(stats: torch.Tensor) -> List[dict]:
    """Decodes an [M, 12] int32 tensor of ssd_row_stats records."""
    s = stats.cpu()
    ints = s[:, :4].numpy()
    flts = s.view(torch.float32)[:, 4:9].numpy()
    return [{"top1": int(i[0]), "top2": int(i[1]), "sample": int(i[2]), "z1": float(f[0]),
             "z2": float(f[1]), "lse": float(f[2]), "conf": float(f[3]), "lse_t": float(f[4])}
            for i, f in zip(ints, flts)]
