"""gnn_sparse_attention_gb300 -- fused CSR graph attention (Graph Transformer dot
score and GATv2) for NVIDIA GB300, behind the C ABI of ``include/gattn.h``.

The CUDA library is loaded lazily on first use; importing the package does
not touch the GPU.  The public Python names mirror the C entry points.
"""
from __future__ import annotations

__all__ = ["Score", "Plan", "GattnError", "gattn_plan_create", "gattn_plan_get_info",
           "gattn_plan_export", "gattn_plan_export_tiles", "gattn_plan_export_tile_bwd",
           "gattn_workspace_size", "gattn_fwd", "gattn_bwd", "gattn_bwd_dq", "gattn_bwd_dkdv",
           "gattn_plan_check_errors", "gattn_fwd_noalloc", "gattn_reorder", "gattn_permute_csr",
           "gattn_permute_rows", "gattn_pool_workspace_size", "gattn_pool_fwd", "gattn_pool_bwd",
           "gattn_spmm_workspace_size", "gattn_spmm", "gattn_version", "load_library"]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
