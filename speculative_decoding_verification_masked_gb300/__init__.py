"""GB300-native speculative-decoding verification attention.

The compute lives in libverify_attn.so (hand-written sm_103a CUDA, C ABI in
include/verify_attn.h); this package builds it in-tree and binds it.
"""
from .api import (  # noqa: F401
    ScoreScratch,
    VerifyAttnError,
    Workspace,
    make_shape,
    verify_accept_greedy,
    verify_attn_check_status,
    verify_attn_combine,
    verify_attn_dense,
    verify_attn_paged,
    verify_attn_sparse,
    verify_build_index,
    verify_commit_kv_dense,
    verify_commit_kv_paged,
    verify_head_importance,
    verify_rope_draft_dense,
    verify_rope_draft_paged,
    verify_tree_mask_from_parents,
    version,
    workspace_size,
)
