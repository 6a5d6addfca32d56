"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the bench.

This package holds no arithmetic of the decoding method itself: only model
shapes, draft policies, and seeded generators for weights, prompts and
candidate skip masks.  Both the CPU oracle and the CUDA library consume what
it produces; neither imports the other.
"""

from .configs import (  # noqa: F401
    ModelShape,
    Policy,
    Workload,
    WORKLOADS,
    TINY,
    LLAMA7B_SWIFT,
    LLAMA7B_LAYERSKIP,
    LLAMA7B_EXIT_AGREE,
    LLAMA13B_SCORE,
    LLAMA70B_SWIFT,
    shrink,
)
from .generate import (  # noqa: F401
    make_weights,
    make_prompt,
    make_masks,
    weights_to_numpy,
    splitmix64,
)
