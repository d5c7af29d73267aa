"""Batched draft verification for speculative decoding on GB300 (sm_103a).

The compute runs in the CUDA library libspecverify.so (C ABI in
include/spec_verify.h); this package only builds it and marshals arguments.
"""

from .api import (  # noqa: F401
    CascadePlan, ChainPlan, ChainPlanNoAlloc, ClaspPlan, LmHeadChainPlan, PipelineAsyncPlan, PipelinePlan,
    TreePlan,
    clasp_layer_select, compact_tree_path, verify_cascade, verify_chain, verify_pipeline, verify_pipeline_async,
    verify_tree, workspace_bytes,
)
from ._lib import ERR_NONFINITE, ERR_PARENT, ERR_TOKEN, ERR_WINDOW, ERR_ZERO_MASS  # noqa: F401
from .build import build as build_library, lib_path  # noqa: F401
