"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke run.

This package draws random logits, drafted tokens and uniforms.  It holds none
of the verification arithmetic: no softmax, no accept test, no residual and
no inverse CDF.  Both the CUDA path and the CPU oracle consume its output.
"""

from .synth import (  # noqa: F401
    SPECS, ChainSpec, TreeSpec, CascadeSpec, make, make_chain, make_tree,
    make_cascade, tree_topology, bf16_from_float32, float32_from_bf16,
)
