"""GB300 (sm_103a) library for one tree-verification step of Medusa/Hydra speculative decoding.

The compute lives in libspec_tree.so (C ABI declared in include/spec_tree.h);
this package holds the CUDA sources, the build script and a thin ctypes
binding whose functions carry the C entry points' names.  Importing the
binding loads the library and fails loudly when it has not been built.
"""

__all__ = [
    "spec_tree_build", "spec_tree_device_bytes",
    "hydra_draft", "hydra_draft_workspace_size", "hydra_draft_heads", "hydra_draft_folded", "hydra_fold_embedding",
    "tree_attention", "tree_attention_workspace_size", "tree_attention_noalloc",
    "tree_attention_noalloc_status",
    "tree_attention_paged", "tree_attention_paged_workspace_size",
    "tree_accept", "tree_accept_workspace_size", "tree_accept_typical",
    "tree_kv_commit", "tree_kv_commit_paged", "tree_kv_commit_workspace_size",
    "spec_philox_uniform", "spec_read_device_status", "spec_last_error", "spec_selftest_timeout",
    "spec_trace_begin", "spec_trace_end", "spec_launch_count",
    "SpecError", "Tree",
]


def __getattr__(name):
    if name in __all__:
        from . import _binding
        return getattr(_binding, name)
    raise AttributeError(name)
