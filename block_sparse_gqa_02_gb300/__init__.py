"""MiniMax Sparse Attention (MSA) hot path for GB300 (sm_103a).

The computation lives in libmsa.so (CUDA kernels behind the C ABI of include/msa.h);
this package only marshals arguments to it.
"""
from ._lib import (MsaError, MsaShape, make_shape, msa_abi_version, msa_block_topk,
                   msa_get_device_status, msa_index_scores, msa_sparse_decode,
                   msa_sparse_prefill, msa_workspace_bytes, shape_from_config)
from .api import (alloc_decode_outputs, alloc_prefill_outputs, decode, prefill, run_decode,
                  run_prefill)
