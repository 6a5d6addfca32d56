"""Model shapes, draft policies and the five synthetic workloads.

The workloads stand in for the trained checkpoints and datasets the pages
measure on (LLaMA-2 7B/13B/70B on CNN/DM, GSM8K, HumanEval, ...), none of
which exist here: every weight is drawn N(0, 0.02) from a seed and every
prompt is uniform-random token ids.
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional, Tuple


@dataclass(frozen=True)
class ModelShape:
    """A Llama-style decoder: RMSNorm, rotate-half RoPE, (GQA) attention, SwiGLU."""

    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rope_theta: float = 1.0e4
    norm_eps: float = 1.0e-5
    # "bf16": bf16 weights, bf16 rounding at GEMM inputs and on stored K/V.
    # "fp32": fp32 weights and no rounding anywhere (the tiny oracle case).
    dtype: str = "bf16"

    @property
    def qkv_rows(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def attn_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def layer_params(self) -> int:
        d, f = self.d_model, self.ffn_dim
        return self.qkv_rows * d + d * self.attn_dim + 3 * d * f

    def total_params(self) -> int:
        return self.n_layers * self.layer_params() + 2 * self.vocab * self.d_model


@dataclass(frozen=True)
class Policy:
    """Draft policy: which layers the draft runs and when it stops.

    mode "skip": the draft runs every layer not in ``skip`` (SWIFT / Self-SD);
    ``skip_attn`` / ``skip_mlp`` additionally drop only the attention or only
    the MLP sublayer of the listed layers (SWIFT Fig. 10 skips the two
    sublayers separately).  A layer in ``skip`` drops both.
    mode "exit": the draft runs layers 0..exit_layer and applies the shared
    final norm + LM head to that hidden state (LayerSkip).
    ``tau`` is the top-1 confidence threshold of the early stop (None: no
    stop); ``temperature`` 0 means greedy drafting and acceptance.
    ``tree_tau`` (None: off) turns on dynamic verification: a kept draft
    whose top-1 confidence is below it also sends the draft's second choice
    to the verify as a sibling candidate, at most ``tree_max`` per round.
    """

    mode: str = "skip"
    skip: Tuple[int, ...] = ()
    exit_layer: int = -1
    d_max: int = 4
    tau: Optional[float] = None
    temperature: float = 0.0
    seed: int = 0
    skip_attn: Tuple[int, ...] = ()
    skip_mlp: Tuple[int, ...] = ()
    tree_tau: Optional[float] = None
    tree_max: int = 0

    def sublayers(self, layer: int) -> Tuple[bool, bool]:
        """(attention runs, MLP runs) for ``layer`` in the draft (skip mode)."""
        whole = layer in self.skip
        return (not whole and layer not in self.skip_attn,
                not whole and layer not in self.skip_mlp)

    def draft_layers(self, n_layers: int) -> Tuple[int, ...]:
        """Layers the draft runs at least one sublayer of."""
        if self.mode == "skip":
            return tuple(l for l in range(n_layers) if any(self.sublayers(l)))
        return tuple(range(self.exit_layer + 1))

    def first_recomputed(self, n_layers: int) -> int:
        """s0: the first layer the verify pass recomputes."""
        if self.mode == "skip":
            dropped = set(self.skip) | set(self.skip_attn) | set(self.skip_mlp)
            return min(dropped) if dropped else n_layers
        return self.exit_layer + 1


@dataclass(frozen=True)
class Workload:
    name: str
    shape: ModelShape
    weight_seed: int = 0
    # layers whose attention-output and MLP-down projections are scaled
    scaled_layers: Tuple[int, ...] = ()
    scale: float = 1.0
    prompt_len: int = 16
    prompt_seed: int = 1
    gen_len: int = 64
    policy: Policy = field(default_factory=Policy)
    # candidate-mask scoring (SWIFT layer-set optimisation)
    n_masks: int = 0
    window: int = 0
    mask_seed: int = 0
    mask_layers: Tuple[int, ...] = ()
    mask_drop: int = 0
    # greedy tokens generated after the prompt before scoring, so that the
    # scoring window holds full-model greedy tokens
    pre_generate: int = 0
    # weight options (make_weights defaults): LM head multiplier, RMSNorm
    # gains 1 + N(0, 0.1) instead of ones
    lm_head_scale: float = 1.0
    random_gains: bool = False


def _odd(lo: int, hi: int) -> Tuple[int, ...]:
    return tuple(l for l in range(lo, hi + 1) if l % 2 == 1)


TINY = Workload(
    name="tiny-L4-d256",
    shape=ModelShape(n_layers=4, d_model=256, n_heads=4, n_kv_heads=4, head_dim=64,
                     ffn_dim=704, vocab=1024, dtype="fp32"),
    weight_seed=0,
    scaled_layers=(2,),
    scale=0.1,
    prompt_len=16,
    prompt_seed=1,
    gen_len=64,
    policy=Policy(mode="skip", skip=(2,), d_max=4, tau=0.5),
)

_LLAMA7B = ModelShape(n_layers=32, d_model=4096, n_heads=32, n_kv_heads=32, head_dim=128,
                      ffn_dim=11008, vocab=32000)

LLAMA7B_SWIFT = Workload(
    name="llama2-7b-swift-skip",
    shape=_LLAMA7B,
    scaled_layers=_odd(9, 31),
    scale=0.1,
    prompt_len=512,
    gen_len=256,
    policy=Policy(mode="skip", skip=_odd(9, 31), d_max=8, tau=0.8),
)

LLAMA7B_SUBLAYER = Workload(
    # sub-layer drafting on the 7B shape (SWIFT Fig. 10): the draft drops the
    # attention sublayer of the odd layers 9..31 and the MLP sublayer of the
    # even layers 10..30 (as many sublayers as the whole-layer c1 set)
    name="llama2-7b-swift-sublayer",
    shape=_LLAMA7B,
    scaled_layers=_odd(9, 31),
    scale=0.1,
    prompt_len=512,
    gen_len=256,
    policy=Policy(mode="skip", skip_attn=_odd(9, 31),
                  skip_mlp=tuple(l for l in range(10, 31) if l % 2 == 0), d_max=8, tau=None),
)

LLAMA7B_LAYERSKIP = Workload(
    name="llama2-7b-layerskip-exit8",
    shape=_LLAMA7B,
    scaled_layers=tuple(range(9, 32)),
    scale=0.15,
    prompt_len=1024,
    gen_len=512,
    policy=Policy(mode="exit", exit_layer=8, d_max=12, tau=None, temperature=0.6, seed=1234),
)

LLAMA13B_SCORE = Workload(
    name="llama2-13b-swift-score",
    shape=ModelShape(n_layers=40, d_model=5120, n_heads=40, n_kv_heads=40, head_dim=128,
                     ffn_dim=13824, vocab=32000),
    prompt_len=2016,
    pre_generate=32,
    gen_len=128,
    policy=Policy(mode="skip", skip=(), d_max=8, tau=0.8),
    n_masks=16,
    window=32,
    mask_seed=0,
    mask_layers=tuple(range(4, 40)),
    mask_drop=16,
)

LLAMA70B_SWIFT = Workload(
    name="llama2-70b-swift-skip",
    shape=ModelShape(n_layers=80, d_model=8192, n_heads=64, n_kv_heads=8, head_dim=128,
                     ffn_dim=28672, vocab=32000),
    scaled_layers=tuple(range(20, 80, 2)),
    scale=0.1,
    prompt_len=1024,
    gen_len=256,
    policy=Policy(mode="skip", skip=tuple(range(20, 80, 2)), d_max=8, tau=0.7),
)

# The tiny model with the parity tests' sharpened LM head (x10) and random
# norm gains: drafts clear the confidence bar and are often accepted, so the
# draft loop, rollback and dynamic verification do real work (with the plain
# N(0, 0.02) head every literal threshold stops drafting at the first step).
TINY_SHARP = replace(TINY, name="tiny-L4-d256-sharp", lm_head_scale=10.0, random_gains=True,
                     policy=Policy(mode="skip", skip=(2,), d_max=4, tau=None))

# A draft-friendly 7B model (not a configured workload): the LayerSkip exit
# workload with layers 9..31's residual outputs scaled x0.01, so that the exit
# at layer 8 predicts nearly what the full model predicts.  On plain random
# weights a draft is rarely accepted; this model shows what the library's
# draft / verify / accept machinery delivers when drafts are accepted (the
# situation trained early-exit models are built for), greedy.
LLAMA7B_EXIT_AGREE = replace(LLAMA7B_LAYERSKIP, name="llama2-7b-exit8-agreeing", scale=0.01,
                             gen_len=256,
                             policy=Policy(mode="exit", exit_layer=8, d_max=12, tau=None))

WORKLOADS = {w.name: w for w in (TINY, LLAMA7B_SWIFT, LLAMA7B_LAYERSKIP, LLAMA13B_SCORE,
                                 LLAMA70B_SWIFT, LLAMA7B_SUBLAYER, TINY_SHARP,
                                 LLAMA7B_EXIT_AGREE)}


def shrink(w: Workload, **shape_changes) -> Workload:
    """A copy of ``w`` with a changed shape (for small parity cases)."""
    return replace(w, shape=replace(w.shape, **shape_changes))
