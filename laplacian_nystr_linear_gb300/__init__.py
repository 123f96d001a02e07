"""lapnys: Laplacian-kernel Nystrom linear attention for GB300 (sm_103a).

The compute path is liblapnys.so (CUDA kernels behind a C ABI, declared in
include/lapnys.h); this package only marshals PyTorch tensors and streams into
it.  Importing the package does not load the library; the first call does, and
fails loudly if it has not been built.
"""
from .api import (BlockParams, Params, alloc_ctx, alloc_workspace, attention, attention_block,
                  block_bwd, block_ctx_bytes, block_fwd, block_workspace_bytes, bwd, ctx_bytes,
                  ctx_offsets, ctx_views, fwd, launch_count, pool, profile_enable, profile_read,
                  workspace_bytes)

__all__ = ["BlockParams", "Params", "alloc_ctx", "alloc_workspace", "attention", "attention_block",
           "block_bwd", "block_ctx_bytes", "block_fwd", "block_workspace_bytes", "bwd", "ctx_bytes",
           "ctx_offsets", "ctx_views", "fwd", "launch_count", "pool", "profile_enable",
           "profile_read", "workspace_bytes"]
