"""fp64 CPU oracle for MSA -- test infrastructure only (see msa_oracle's header)."""
from .msa_oracle import *  # noqa: F401,F403
from .msa_oracle import (index_logits, pool_blocks, index_block_scores_prefill,
                         index_block_scores_decode, current_block, select_blocks,
                         block_topk_prefill, block_topk_decode, selected_keys,
                         sparse_attention, full_causal_gqa, msa_prefill, msa_decode,
                         default_scale)
