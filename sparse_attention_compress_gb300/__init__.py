"""GB300 (sm_103a) native-sparse-attention hot path.

The CUDA library ``libnsa.so`` (C ABI declared in ``include/nsa.h``) does all the
work; ``_lib`` marshals PyTorch tensors into its calls.  Import is cheap: the shared
library is opened on the first call.
"""
from ._lib import (NsaError, load, make_shape, nsa_block_sparse_fwd, nsa_block_sparse_workspace_size,
                   nsa_cis_block_scores, nsa_sparse_cis_fwd, nsa_topk_two_stage, nsa_cmp_attn_bwd,
                   nsa_cmp_attn_bwd_workspace_size, nsa_compress_bwd, nsa_swa_bwd, nsa_swa_bwd_workspace_size,
                   nsa_gate_combine_bwd, nsa_sparse_decode_cis, nsa_layer_fwd_train, nsa_layer_bwd, nsa_layer_saved_buffers,
                   nsa_cmp_attn_fwd, nsa_device_status, nsa_cmp_scores_pool, nsa_compress_k,  # noqa: F401
                   nsa_gate_combine, nsa_layer_fwd, nsa_select, nsa_select_workspace_size, nsa_layer_fwd_workspace_size, nsa_sparse_decode,
                   nsa_sparse_decode_noalloc, nsa_sparse_decode_workspace_size, nsa_sparse_bwd,
                   nsa_sparse_bwd_workspace_size, nsa_sparse_fwd, nsa_swa_fwd, nsa_topk_select, num_cmp,
                   nsa_set_wait_limit_ns)

__all__ = ["NsaError", "load", "make_shape", "nsa_block_sparse_fwd", "nsa_block_sparse_workspace_size",
           "nsa_cis_block_scores", "nsa_sparse_cis_fwd", "nsa_topk_two_stage", "nsa_cmp_attn_bwd",
           "nsa_cmp_attn_bwd_workspace_size", "nsa_compress_bwd", "nsa_swa_bwd", "nsa_swa_bwd_workspace_size",
           "nsa_gate_combine_bwd", "nsa_sparse_decode_cis", "nsa_layer_fwd_train", "nsa_layer_bwd", "nsa_layer_saved_buffers", "nsa_cmp_attn_fwd", "nsa_device_status", "nsa_cmp_scores_pool", "nsa_compress_k",
           "nsa_gate_combine", "nsa_layer_fwd", "nsa_select", "nsa_select_workspace_size", "nsa_layer_fwd_workspace_size", "nsa_sparse_decode",
           "nsa_sparse_decode_noalloc", "nsa_sparse_decode_workspace_size", "nsa_sparse_bwd",
           "nsa_sparse_bwd_workspace_size", "nsa_sparse_fwd", "nsa_swa_fwd", "nsa_topk_select", "num_cmp",
           "nsa_set_wait_limit_ns"]
