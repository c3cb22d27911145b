"""GB300-native DSA lightning indexer + causal top-k, IndexShare layer loop and sparse MLA
attention.  The compute runs in libdsa.so (hand-written sm_103a kernels behind a C ABI,
include/dsa.h); this package is its ctypes binding plus seeded input generators.
"""
from ._lib import (AttnDesc, DsaError, IndexCache, IndexerDesc, LayerIO, PagedCache, DSA_IDX_INDEPENDENT_ROWS,
                   DSA_IDX_ROPE_K, DSA_PAGE_ROWS, ProjDesc, dsa_indexer_projections, dsa_indexer_topk_paged,
                   dsa_sparse_attn_backward, dsa_sparse_attn_backward_workspace_size, dsa_indexer_backward,
                   dsa_indexer_backward_workspace_size,
                   dsa_sparse_attn_paged, paged_cache,
                   DSA_IDX_ROPE_Q, DSA_LAYER_FULL, DSA_LAYER_SHARED, attn_desc, dsa_donor_table,
                   dsa_indexer_topk, dsa_indexer_topk_static, dsa_indexer_workspace_size, dsa_layers_workspace_size, dsa_mtp_indexshare_step,
                   dsa_profile_enable,
                   dsa_profile_indexer_last, dsa_profile_read, dsa_indexer_static_status, dsa_debug_pipeline, dsa_rope_table,
                   dsa_sparse_attn, dsa_sparse_attn_workspace_size, dsa_workspace_status, indexer_desc,
                   indexshare_layers_forward, lib)

__all__ = ["AttnDesc", "DsaError", "IndexCache", "IndexerDesc", "LayerIO", "PagedCache", "DSA_PAGE_ROWS",
           "dsa_indexer_topk_paged", "dsa_sparse_attn_paged", "paged_cache", "ProjDesc", "dsa_indexer_projections", "dsa_sparse_attn_backward",
           "dsa_sparse_attn_backward_workspace_size", "dsa_indexer_backward", "dsa_indexer_backward_workspace_size", "DSA_IDX_INDEPENDENT_ROWS", "DSA_IDX_ROPE_K",
           "DSA_IDX_ROPE_Q", "DSA_LAYER_FULL", "DSA_LAYER_SHARED", "attn_desc", "dsa_donor_table", "dsa_indexer_topk", "dsa_indexer_topk_static",
           "dsa_indexer_workspace_size", "dsa_layers_workspace_size", "dsa_mtp_indexshare_step", "dsa_profile_enable",
           "dsa_profile_indexer_last", "dsa_profile_read", "dsa_indexer_static_status", "dsa_debug_pipeline", "dsa_rope_table", "dsa_sparse_attn",
           "dsa_sparse_attn_workspace_size", "dsa_workspace_status", "indexer_desc", "indexshare_layers_forward", "lib"]
