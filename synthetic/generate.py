"""Seeded generators: weights, prompts, candidate skip masks.

Weights are drawn N(0, 0.02) per tensor from a torch generator seeded from
(workload seed, tensor index), so that any single tensor can be regenerated
on its own.  The attention-output and MLP-down projections of the workload's
``scaled_layers`` are multiplied by ``scale`` (so that skipping those layers
drafts well), then everything is rounded to the workload dtype.

Layout of the returned dict (the layout the CUDA library consumes; the
oracle slices the same arrays):

    tok_embed  [V, D]            lm_head [V, D]          final_norm [D] fp32
    layers[l]: attn_norm [D] fp32, wqkv [(H + 2 Hkv) dh, D] (q rows, k rows,
               v rows), wo [D, H dh], mlp_norm [D] fp32, w_gate [F, D],
               w_up [F, D], w_down [D, F]
"""

from __future__ import annotations

from typing import Dict, List

import numpy as np
import torch

from .configs import Workload

_M64 = (1 << 64) - 1


def splitmix64(x: int) -> int:
    """One step of Steele/Lea/Flood's SplitMix64 finaliser on ``x + golden``."""
    x = (x + 0x9E3779B97F4A7C15) & _M64
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def _tensor_seed(weight_seed: int, index: int) -> int:
    return splitmix64(((weight_seed & 0xFFFFFFFF) << 32) + index) & ((1 << 63) - 1)


def _normal(shape, seed: int, device, std: float, scale: float, dtype) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    t.mul_(std * scale)
    return t.to(dtype)


def make_weights(w: Workload, device="cpu", dtype: str | None = None,
                 random_gains: bool | None = None, lm_head_scale: float | None = None) -> Dict:
    """Seeded synthetic weights for workload ``w`` on ``device``.

    ``dtype`` overrides the workload dtype ("bf16" or "fp32").
    ``random_gains`` draws the RMSNorm gains 1 + N(0, 0.1) instead of ones
    (parity cases use it so that a dropped gain is caught).
    ``lm_head_scale`` multiplies the LM head (parity cases use a sharper head
    so that greedy sequences have fewer near-ties).  Both default to the
    workload's own setting.
    """
    if random_gains is None:
        random_gains = w.random_gains
    if lm_head_scale is None:
        lm_head_scale = w.lm_head_scale
    s = w.shape
    dt = dtype or s.dtype
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    D, F, V = s.d_model, s.ffn_dim, s.vocab
    seed = w.weight_seed

    def gain(index: int) -> torch.Tensor:
        if not random_gains:
            return torch.ones(D, dtype=torch.float32, device=device)
        return 1.0 + _normal((D,), _tensor_seed(seed, index), device, 0.1, 1.0, torch.float32)

    out: Dict = {
        "tok_embed": _normal((V, D), _tensor_seed(seed, 0), device, 0.02, 1.0, tdt),
        "lm_head": _normal((V, D), _tensor_seed(seed, 1), device, 0.02, lm_head_scale, tdt),
        "final_norm": gain(2),
    }
    layers: List[Dict] = []
    scaled = set(w.scaled_layers)
    for l in range(s.n_layers):
        base = 16 + 16 * l
        sc = w.scale if l in scaled else 1.0
        layers.append({
            "attn_norm": gain(base + 0),
            "wqkv": _normal((s.qkv_rows, D), _tensor_seed(seed, base + 1), device, 0.02, 1.0, tdt),
            "wo": _normal((D, s.attn_dim), _tensor_seed(seed, base + 2), device, 0.02, sc, tdt),
            "mlp_norm": gain(base + 3),
            "w_gate": _normal((F, D), _tensor_seed(seed, base + 4), device, 0.02, 1.0, tdt),
            "w_up": _normal((F, D), _tensor_seed(seed, base + 5), device, 0.02, 1.0, tdt),
            "w_down": _normal((D, F), _tensor_seed(seed, base + 6), device, 0.02, sc, tdt),
        })
    out["layers"] = layers
    out["dtype"] = dt
    return out


def _to_numpy(t: torch.Tensor) -> np.ndarray:
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def weights_to_numpy(wts: Dict) -> Dict:
    """Host copies: bf16 tensors become uint16 arrays of their bit patterns."""
    out = {k: _to_numpy(v) for k, v in wts.items() if k not in ("layers", "dtype")}
    out["layers"] = [{k: _to_numpy(v) for k, v in lw.items()} for lw in wts["layers"]]
    out["dtype"] = wts["dtype"]
    return out


def make_prompt(w: Workload, length: int | None = None, seed: int | None = None) -> np.ndarray:
    """Uniform-random token ids (int32)."""
    rng = np.random.default_rng(w.prompt_seed if seed is None else seed)
    n = w.prompt_len if length is None else length
    return rng.integers(0, w.shape.vocab, size=n, dtype=np.int64).astype(np.int32)


def make_masks(w: Workload, n_masks: int | None = None) -> List[tuple]:
    """Candidate skip sets: each drops ``mask_drop`` of ``mask_layers``.

    Mask k is a partial Fisher-Yates shuffle of ``mask_layers`` driven by a
    SplitMix64 stream seeded with ``mask_seed + k``.
    """
    K = w.n_masks if n_masks is None else n_masks
    masks = []
    for k in range(K):
        cand = list(w.mask_layers)
        state = (w.mask_seed + k) & _M64
        for i in range(w.mask_drop):
            state = (state + 0x9E3779B97F4A7C15) & _M64
            r = splitmix64(state)
            j = i + r % (len(cand) - i)
            cand[i], cand[j] = cand[j], cand[i]
        masks.append(tuple(sorted(cand[: w.mask_drop])))
    return masks
