"""CPU oracle for layer-skipping self-speculative decoding — TEST INFRASTRUCTURE.

A plain, slow, fp64 numpy restatement of what the hot path computes, written
from the pages' description of the method:

* SWIFT: On-the-Fly Self-Speculative Decoding for LLM Inference Acceleration
  (paperlayer.ai digest) — skip-set drafting, confidence-aware early stop
  (§4.2), matchness scoring of candidate layer sets (§4.1, §4.1.2, D.2), the
  M / alpha metrics (B.3).
* LayerSkip blog (marsggbo.github.io, "ACL'24 | LayerSkip ...") — early-exit
  drafting through the shared LM head (§3.1), verify over d+1 positions with
  KV reuse (§3.2), min(1, p/q) acceptance with residual resampling and the
  bonus token (§3.3), lossy early exit (§3, inference mode one).
* The early-exit structure page on AdaInfer — per-layer gap / top-prob exit
  features and their labels (steps 1-2).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The CUDA library never calls it and shares no
code with it; the only common inputs come from the ``synthetic`` package.

Parity unpinned: the pages' absolute quality figures (98-100% greedy
acceptance, 1.3-1.6x speedups) need trained checkpoints and datasets that do
not exist here; nothing in this package claims them.
"""

from .numerics import bf16_round, widen  # noqa: F401
from .philox import philox4x32_10, uniforms, gumbel_argmax  # noqa: F401
from .model import OracleModel, KVCache  # noqa: F401
from .speculative import (  # noqa: F401
    SSDState,
    RoundRecord,
    prefill,
    ar_step,
    ar_generate,
    ssd_round,
    ssd_generate,
    accept_stochastic,
)
from .scoring import score_masks, score_masks_bruteforce  # noqa: F401
from .adaptive import (  # noqa: F401
    lossy_step,
    lossy_generate,
    layer_features,
    exit_features,
    LayerFeatures,
)
from .swift import (  # noqa: F401
    SplitMix64,
    SwiftParams,
    SwiftTrace,
    swift_generate,
    uniform_set,
    propose,
)
