"""Whole-pass helpers over the C ABI: allocate the outputs with torch, then run the three
MSA stages (index block scores -> per-KV-head block top-k -> sparse attention) as
library calls on the current stream, with no host synchronisation in between."""
from __future__ import annotations

import torch

from . import _lib
from ._lib import (make_shape, msa_block_topk, msa_index_scores, msa_sparse_decode,
                   msa_sparse_prefill, msa_workspace_bytes)

_DT = {torch.float32: "f32", torch.bfloat16: "bf16"}


def _shape_of(q, k, idx_q, block_size, top_k, q_tile, sm_scale, index_scale):
    B, Sq, Hq, d = q.shape
    _, Hkv, Sk, _ = k.shape
    return make_shape(B, Sq, Sk, Hq, Hkv, d, idx_q.shape[-1], block_size, top_k, q_tile,
                      _DT[q.dtype], sm_scale, index_scale)


def alloc_prefill_outputs(shape, device, dtype):
    B, Hkv = shape.batch, shape.n_heads_kv
    return dict(
        scores=torch.empty((B, Hkv, shape.n_rows, shape.n_blocks), device=device,
                           dtype=torch.float32),
        sel=torch.empty((B, Hkv, shape.n_rows, shape.top_k), device=device, dtype=torch.int32),
        out=torch.empty((B, shape.seq_q, shape.n_heads_q, shape.head_dim), device=device,
                        dtype=dtype),
        lse=torch.empty((B, shape.n_heads_q, shape.seq_q), device=device, dtype=torch.float32))


def run_prefill(shape, q, k, v, idx_q, idx_k, bufs, stream=None):
    """One prefill pass into preallocated buffers (dict from alloc_prefill_outputs)."""
    msa_index_scores(shape, idx_q, idx_k, bufs["scores"], stream)
    msa_block_topk(shape, bufs["scores"], bufs["sel"], stream)
    msa_sparse_prefill(shape, q, k, v, bufs["sel"], bufs["out"], bufs["lse"], None, 0, stream)


def run_decode(shape, q, k_cache, v_cache, idx_q, idx_k, bufs, stream=None):
    """One decode step into preallocated buffers (alloc_prefill_outputs + 'ws')."""
    msa_index_scores(shape, idx_q, idx_k, bufs["scores"], stream)
    msa_block_topk(shape, bufs["scores"], bufs["sel"], stream)
    msa_sparse_decode(shape, q, k_cache, v_cache, bufs["sel"], bufs["out"], bufs["lse"],
                      bufs["ws"], None, stream)


def prefill(q, k, v, idx_q, idx_k, block_size=128, top_k=16, q_tile=64, sm_scale=0.0,
            index_scale=0.0):
    """MSA prefill.  q [B,T,Hq,d], k/v [B,Hkv,T,d], idx_q [B,T,Hkv,dI], idx_k [B,T,dI].

    Returns a dict with out [B,T,Hq,d], lse [B,Hq,T], scores and sel."""
    shape = _shape_of(q, k, idx_q, block_size, top_k, q_tile, sm_scale, index_scale)
    bufs = alloc_prefill_outputs(shape, q.device, q.dtype)
    run_prefill(shape, q, k, v, idx_q, idx_k, bufs)
    return bufs


def alloc_decode_outputs(shape, device, dtype):
    bufs = alloc_prefill_outputs(shape, device, dtype)
    nbytes = max(16, msa_workspace_bytes(shape, 1))
    bufs["ws"] = torch.empty((nbytes + 15) // 16 * 4, device=device, dtype=torch.float32)
    return bufs


def decode(q, k_cache, v_cache, idx_q, idx_k, block_size=128, top_k=64, sm_scale=0.0,
           index_scale=0.0):
    """One MSA decode step.  q [B,1,Hq,d], caches [B,Hkv,L,d], idx_q [B,1,Hkv,dI],
    idx_k [B,L,dI]; the new token is at position L-1 and already in the caches."""
    shape = _shape_of(q, k_cache, idx_q, block_size, top_k, 1, sm_scale, index_scale)
    bufs = alloc_decode_outputs(shape, q.device, q.dtype)
    run_decode(shape, q, k_cache, v_cache, idx_q, idx_k, bufs)
    return bufs


__all__ = ["prefill", "decode", "run_prefill", "run_decode", "alloc_prefill_outputs",
           "alloc_decode_outputs", "_lib"]
