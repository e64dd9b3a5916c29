"""GB300-native token-tree verification: tree attention + verification.

The compute lives in ``libspec_tree.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/spec_tree.h``).  This package is only the thin
Python binding: it passes device pointers, sizes and the current CUDA stream.
Nothing here computes; there is no CPU fallback: if the library is missing the
calls raise.
"""
from .binding import (  # noqa: F401
    SpecError, load, lib_path, build_tree_mask, tree_attn, tree_attn_workspace_size,
    tree_verify, tree_verify_workspace_size, make_verify_workspace, kv_compact, tree_expand, tree_prune, status_string,
    philox_uniforms, tree_merge, STATUS,
)
