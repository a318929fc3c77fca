"""GB300 (sm_103a) MSA block-sparse GQA attention: index-branch block scores, per-group
top-k block selection with the forced local block, sparse main-branch attention (O, LSE),
the decode path (packed or paged KV cache), variable-length prefill batches, the main branch's
backward, and the KL alignment loss that trains the index branch with its gradient, behind the
C ABI of libmsa.so (include/msa.h)."""
from .msa import (MSAError, msa_device_status, msa_index_block_scores,  # noqa: F401
                  msa_index_select, msa_select_blocks, msa_sparse_attn_fwd, msa_sparse_attn_fwd_workspace,
                  msa_sparse_decode, msa_sparse_decode_workspace, msa_sparse_decode_paged,
                  msa_prefill_varlen, msa_prefill_varlen_workspace,
                  msa_kl_loss_fwd, msa_kl_loss_bwd, msa_kl_loss_bwd_workspace,
                  msa_kl_loss_fwd_workspace, msa_sparse_decode_noalloc,
                  msa_set_wait_limit_ns, msa_sparse_attn_bwd, msa_sparse_attn_bwd_workspace)
