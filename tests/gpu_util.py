"""Helpers for the GPU parity tests: seeded inputs on both sides."""

import numpy as np
import torch


def rand_bf16(shape, seed, std=0.02):
    """A seeded bf16 tensor on cuda:0 and its bit pattern (uint16) on the host."""
    rng = np.random.default_rng(seed)
    t = torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32)).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.cuda(), bits


def rand_f32(shape, seed, std=1.0, mean=0.0):
    rng = np.random.default_rng(seed)
    a = (mean + rng.standard_normal(shape) * std).astype(np.float32)
    return torch.from_numpy(a).cuda(), a.astype(np.float64)


def bf16_values(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def to_device_weights(wts):
    """Device copies of a weight dict, projection matrices packed for the library."""
    import self_speculative_decoding_gb300 as ssd
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in wts.items()
           if k != "layers"}
    dev["layers"] = [{k: v.cuda() for k, v in lw.items()} for lw in wts["layers"]]
    return ssd.pack_weights(dev)


def pack_reference(bits: np.ndarray) -> np.ndarray:
    """The packed unit layout, written out with numpy index arithmetic:
    16 x 32 tiles ordered (row group, K block), each 8-row half row-major with
    the 16-byte chunks of row g at positions c ^ ((g >> 1) & 3)."""
    R, K = bits.shape
    u = bits.reshape(R // 16, 2, 8, K // 32, 4, 8)        # vr, h, g, kb, c, e
    u = u.transpose(0, 3, 1, 2, 4, 5).copy()               # vr, kb, h, g, c, e
    out = np.empty_like(u)
    for g in range(8):
        for c in range(4):
            out[:, :, :, g, c ^ ((g >> 1) & 3), :] = u[:, :, :, g, c, :]
    return out.reshape(R, K)


def top_gap(z) -> float:
    """Top-1 minus top-2 of a logit vector."""
    s = np.sort(np.asarray(z, dtype=np.float64))
    return float(s[-1] - s[-2])


def oracle_prompt(m, w, pol, accept, length=None, max_seq=256, tries=400):
    """A seeded prompt chosen on the oracle's values alone: the workload's own
    prompt seed first, then seeds 1000, 1001, ...; the first prompt for which
    accept(prompt, oracle state after the prefill) holds.  Parity tests use it
    to start from a prompt whose first decisions are not near ties, so that a
    comparison never has to be skipped."""
    from oracle import prefill
    from synthetic import make_prompt
    for i in range(tries):
        seed = w.prompt_seed if i == 0 else 1000 + i
        prompt = make_prompt(w, length, seed=seed)
        if accept(prompt, prefill(m, prompt, pol, max_seq)):
            return prompt
    raise AssertionError("no seeded prompt passes the oracle-side selection")
