"""Seeded synthetic inputs for layer-end KV-cache compression.

This package is shared by the CPU oracle's tests, the CUDA path's tests,
``bench.py`` and ``__graft_entry__.smoke()``.  It draws random tensors and
holds the workload shapes; it holds none of the compression arithmetic
(no logits, softmax, pooling, selection, gather or budget allocation).
"""

from .configs import CONFIGS, Config, get_config  # noqa: F401
from .inputs import (  # noqa: F401
    LayerInputs,
    make_layer_inputs,
    stability_scores,
    heavy_hitter_scale,
)
