"""Isolated throughput of the decoder's weight-streaming kernels.

Times one kernel class of a Llama-style decoder layer through the op entry
points of libssd (ssd_ops.h) with CUDA events, over several weight copies
used in rotation so that every launch streams its matrix from HBM (the
copies together exceed twice the 129 MB L2).  Prints one JSON line per
kernel: rows processed, algorithmic bytes per launch (the weights, plus the
K/V read for attention), mean microseconds per launch and GB/s.

    python -m self_speculative_decoding_gb300.kernel_bench \
        [--kernel qkv,o_proj,gate_up,down,lm_head,attention,gate_up_rows,...,score_attn]
        [--model 7b|13b|70b] \
        [--rows M] [--iters N] [--context L] [--lib path/to/libssd.so]

``score_attn`` times the window attention of candidate-mask scoring for
--rows / 32 candidates of 32 window positions over a shared prefix of
--context positions.

``--lib`` times another build of the library (e.g. one compiled with a
different ring geometry by build.build_variant).
"""

from __future__ import annotations

import argparse
import ctypes as C
import json
import math
import os
import sys

import torch

from . import _abi

MODELS = {
    # D, H, Hkv, dh, F, V
    "7b": (4096, 32, 32, 128, 11008, 32000),
    "13b": (5120, 40, 40, 128, 13824, 32000),
    "70b": (8192, 64, 8, 128, 28672, 32000),
}
KERNELS = ("qkv", "o_proj", "gate_up", "down", "lm_head", "attention")
# many-row projections (tcgen05 GEMM) of the batched scoring forward
ROW_KERNELS = ("qkv_rows", "o_proj_rows", "gate_up_rows", "down_rows", "lm_head_rows")


def _packed(lib, R, K, n, st):
    out = []
    for _ in range(n):
        W = (torch.randn(R, K, device="cuda") * 0.02).to(torch.bfloat16)
        P = torch.empty_like(W)
        if lib.ssd_pack_weight(W.data_ptr(), P.data_ptr(), R, K, st) != 0:
            raise RuntimeError(lib.ssd_ops_last_error().decode())
        out.append(P)
        del W
    return out


def _copies(nbytes: int) -> int:
    return max(2, math.ceil(300e6 / nbytes) + 1)


def bench_kernel(lib, name: str, model: str, M: int, iters: int, context: int) -> dict:
    D, H, Hkv, dh, F, V = MODELS[model]
    st = torch.cuda.current_stream().cuda_stream
    eps = C.c_float(1e-5)
    x = torch.randn(M, D, device="cuda")
    gain = torch.ones(D, device="cuda")
    calls = []
    if name == "qkv":
        R = (H + 2 * Hkv) * dh
        Ws = _packed(lib, R, D, _copies(R * D * 2), st)
        y = torch.empty(M, R, device="cuda")
        nbytes = R * D * 2
        calls = [lambda W=W: lib.ssd_op_rmsnorm_linear(W.data_ptr(), R, D, x.data_ptr(),
                                                       gain.data_ptr(), eps, M, y.data_ptr(), st)
                 for W in Ws]
    elif name in ("o_proj", "down"):
        K = H * dh if name == "o_proj" else F
        Ws = _packed(lib, D, K, _copies(D * K * 2), st)
        act = (torch.randn(M, K, device="cuda") * 0.1).to(torch.bfloat16)
        nbytes = D * K * 2
        calls = [lambda W=W: lib.ssd_op_residual_linear(W.data_ptr(), D, K, act.data_ptr(), M,
                                                        x.data_ptr(), st)
                 for W in Ws]
    elif name == "gate_up":
        n = _copies(2 * F * D * 2)
        Wg = _packed(lib, F, D, n, st)
        Wu = _packed(lib, F, D, n, st)
        u = torch.empty(M, F, dtype=torch.bfloat16, device="cuda")
        nbytes = 2 * F * D * 2
        calls = [lambda g=g, w=w: lib.ssd_op_swiglu(g.data_ptr(), w.data_ptr(), F, D,
                                                    x.data_ptr(), gain.data_ptr(), eps, M,
                                                    u.data_ptr(), st)
                 for g, w in zip(Wg, Wu[::-1])]
    elif name == "lm_head":
        Ws = _packed(lib, V, D, _copies(V * D * 2), st)
        stats = torch.zeros(M, 12, dtype=torch.int32, device="cuda")
        nbytes = V * D * 2
        calls = [lambda W=W: lib.ssd_op_lm_head(W.data_ptr(), V, D, x.data_ptr(),
                                                gain.data_ptr(), eps, M, C.c_float(0.0), 0, 0,
                                                0, 0, None, stats.data_ptr(), st)
                 for W in Ws]
    elif name == "attention":
        max_seq = ((context + M + 63) // 64) * 64
        n = _copies(2 * Hkv * max_seq * dh * 2)
        kc = [(torch.randn(Hkv, max_seq, dh, device="cuda") * 0.5).to(torch.bfloat16)
              for _ in range(n)]
        vc = [(torch.randn(Hkv, max_seq, dh, device="cuda") * 0.5).to(torch.bfloat16)
              for _ in range(n)]
        qkv = torch.randn(M, (H + 2 * Hkv) * dh, device="cuda")
        out = torch.empty(M, H * dh, dtype=torch.bfloat16, device="cuda")
        nbytes = 2 * Hkv * (context + M) * dh * 2
        calls = [lambda k=k, v=v: lib.ssd_op_attention(qkv.data_ptr(), M, context, k.data_ptr(),
                                                       v.data_ptr(), max_seq, H, Hkv, dh,
                                                       C.c_float(1e4), out.data_ptr(), st)
                 for k, v in zip(kc, vc)]
    elif name in ROW_KERNELS:
        # activations pre-packed (rows padded to 16), as the scoring forward keeps them
        K = {"o_proj_rows": H * dh, "down_rows": F}.get(name, D)
        R = {"qkv_rows": (H + 2 * Hkv) * dh, "gate_up_rows": F, "lm_head_rows": V}.get(name, D)
        epi = {"qkv_rows": 0, "o_proj_rows": 1, "down_rows": 1, "gate_up_rows": 2,
               "lm_head_rows": 3}[name]
        Tp = (M + 15) // 16 * 16
        a_rm = (torch.randn(Tp, K, device="cuda") * 0.1).to(torch.bfloat16)
        act = torch.empty_like(a_rm)
        lib.ssd_pack_weight(a_rm.data_ptr(), act.data_ptr(), Tp, K, st)
        nmat = 2 if epi == 2 else 1
        n = _copies(nmat * R * K * 2)
        Ws = _packed(lib, R, K, n, st)
        W1 = _packed(lib, R, K, n, st) if epi == 2 else [None] * n
        if epi == 2:
            out = torch.empty(M, R, dtype=torch.bfloat16, device="cuda")
        elif epi == 3:
            out = torch.empty(M, dtype=torch.int32, device="cuda")
        else:
            out = torch.zeros(M, R, device="cuda")
        nbytes = nmat * R * K * 2
        flop = 2.0 * M * nmat * R * K
        calls = [lambda W=W, U=U: lib.ssd_op_linear_rows(
                     W.data_ptr(), U.data_ptr() if U is not None else None, R, K, act.data_ptr(),
                     M, epi | 16, out.data_ptr(), None, st)
                 for W, U in zip(Ws, W1)]
    elif name == "score_attn":
        N = 32
        nc = max(1, M // N)
        split = context
        max_seq = ((split + N + 63) // 64) * 64
        n = _copies(2 * Hkv * max_seq * dh * 2)
        kc = [(torch.randn(Hkv, max_seq, dh, device="cuda") * 0.5).to(torch.bfloat16)
              for _ in range(n)]
        vc = [(torch.randn(Hkv, max_seq, dh, device="cuda") * 0.5).to(torch.bfloat16)
              for _ in range(n)]
        q = (torch.randn(nc * N, H, dh, device="cuda") * 0.5).to(torch.bfloat16)
        wk = (torch.randn(nc * N, Hkv, dh, device="cuda") * 0.5).to(torch.bfloat16)
        wv = (torch.randn(nc * N, Hkv, dh, device="cuda") * 0.5).to(torch.bfloat16)
        cand = torch.arange(nc, dtype=torch.int32, device="cuda")
        out = torch.empty(nc * N, H * dh, dtype=torch.bfloat16, device="cuda")
        nbytes = 2 * Hkv * split * dh * 2
        flop = 4.0 * nc * N * H * (split + (N + 1) / 2) * dh
        calls = [lambda k=k, v=v: lib.ssd_op_score_attention(
                     q.data_ptr(), cand.data_ptr(), nc, N, split, k.data_ptr(), v.data_ptr(),
                     max_seq, wk.data_ptr(), wv.data_ptr(), nc * N, H, Hkv, dh, out.data_ptr(), st)
                 for k, v in zip(kc, vc)]
    else:
        raise ValueError(f"unknown kernel {name}")
    for i in range(3):
        if calls[i % len(calls)]() != 0:
            raise RuntimeError(lib.ssd_ops_last_error().decode())
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(iters):
        calls[i % len(calls)]()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / iters
    r = {"kernel": name, "model": model, "rows": M, "bytes": nbytes, "us": round(us, 2),
         "GBps": round(nbytes / us / 1e3, 1)}
    if name in ROW_KERNELS or name == "score_attn":
        r["TFLOPs"] = round(flop / us / 1e6, 1)
    return r


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--kernel", default=",".join(KERNELS))
    ap.add_argument("--model", default="7b", choices=sorted(MODELS))
    ap.add_argument("--rows", type=int, default=1)
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--context", type=int, default=512)
    ap.add_argument("--lib", default=None)
    a = ap.parse_args(argv)
    lib = _abi.load(a.lib) if a.lib else _abi.lib()
    torch.manual_seed(0)
    for k in a.kernel.split(","):
        print(json.dumps(bench_kernel(lib, k, a.model, a.rows, a.iters, a.context)), flush=True)
        torch.cuda.empty_cache()


if __name__ == "__main__":
    sys.exit(main())
