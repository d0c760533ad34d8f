"""Seeded synthetic workloads for the DFlash draft step.

This package only draws random inputs (weights, target hidden states, token ids,
per-step accepted counts) with the shapes and distributions of the workloads. It
holds none of the method's arithmetic, so both the CUDA path and the oracle can be
fed from it without sharing any computation.
"""
from .configs import CONFIGS, DraftConfig, get_config  # noqa: F401
from .inputs import (  # noqa: F401
    make_weights,
    make_features,
    make_context_lengths,
    make_n_new,
    make_anchors,
    make_targets,
    make_uniforms,
)
