"""The failure path of the tensor-core kernels, exercised without faulting the GPU.

The test hook makes the copy-issuing warp of the prefill kernel (and of the training
kernels' query-tile passes) issue nothing, so the barrier the MMA warp waits on is never
completed (a flag nothing sets).  Every wait in the kernel
is bounded (one second): the kernel must give up, record MSA_ERR_TIMEOUT in the device
status word, and leave the context usable for the next, normal call.
"""
import ctypes

import pytest
import torch

import oracle
from block_sparse_gqa_02_gb300 import _lib
from block_sparse_gqa_02_gb300.configs import CONFIGS
from block_sparse_gqa_02_gb300.inputs import make_inputs, random_selection
from tests.parity import check_lse, check_out

import numpy as np


def test_fault_hook_rejects_unknown_modes():
    lib = _lib.load()
    assert lib.msa_debug_set_fault(7) == _lib.MSA_ERR_INVALID_ARG
    assert lib.msa_debug_set_fault(0) == _lib.MSA_OK


@pytest.mark.gpu
def test_bounded_wait_times_out_and_context_survives():
    cfg = CONFIGS["p32k"].with_(seq=256, top_k=2, n_plants=0)
    x = make_inputs(cfg, device="cuda")
    shape = _lib.shape_from_config(cfg)
    cur = np.array([(m * 64 + 63) // 128 for m in range(shape.n_rows)])
    sel_np = random_selection(np.broadcast_to(cur + 1, (1, 4, shape.n_rows)), 2, 3)
    sel = torch.from_numpy(sel_np).cuda()
    out = torch.full_like(x["q"], 3.0)
    lse = torch.zeros((1, cfg.n_heads_q, cfg.seq), device="cuda")
    _lib.msa_get_device_status()                       # start from a clean status word
    _lib.msa_debug_set_fault(1)
    try:
        _lib.msa_sparse_prefill(shape, x["q"], x["k"], x["v"], sel, out, lse)
        with pytest.raises(_lib.MsaError) as ei:
            _lib.msa_get_device_status()
        assert ei.value.status == _lib.MSA_ERR_TIMEOUT
    finally:
        _lib.msa_debug_set_fault(0)
    # the abandoned launch wrote zeros and -inf instead of leaving garbage
    assert torch.all(out == 0)
    assert torch.all(torch.isneginf(lse))
    # the status word was cleared, and the context still runs the kernel correctly
    _lib.msa_get_device_status()
    _lib.msa_sparse_prefill(shape, x["q"], x["k"], x["v"], sel, out, lse)
    _lib.msa_get_device_status()
    ref_o, ref_l = oracle.sparse_attention(x["q"], x["k"], x["v"], sel_np, 128, 64)
    check_out(out, ref_o, "bf16")
    check_lse(lse, ref_l, "bf16")


@pytest.mark.gpu
@pytest.mark.parametrize("which", ["backward", "index_kl"])
def test_training_kernels_time_out_and_context_survives(which):
    """The same hook stops the copies of the tensor-core backward's and index KL's query-tile
    kernels: the call reports MSA_ERR_TIMEOUT, and the next call on the context is exact."""
    from tests.parity import check_grad
    cfg = CONFIGS["p32k"].with_(seq=256, top_k=2, n_plants=0)
    x = make_inputs(cfg, device="cuda")
    shape = _lib.shape_from_config(cfg)
    cur = np.array([(m * 64 + 63) // 128 for m in range(shape.n_rows)])
    sel_np = random_selection(np.broadcast_to(cur + 1, (1, 4, shape.n_rows)), 2, 4)
    sel = torch.from_numpy(sel_np).cuda()
    out = torch.empty_like(x["q"])
    lse = torch.empty((1, cfg.n_heads_q, cfg.seq), device="cuda")
    _lib.msa_sparse_prefill(shape, x["q"], x["k"], x["v"], sel, out, lse)
    _lib.msa_get_device_status()
    if which == "backward":
        gen = torch.Generator(device="cuda").manual_seed(3)
        dout = torch.randn(x["q"].shape, generator=gen, device="cuda").to(x["q"].dtype)
        grads = [torch.empty(x[n].shape, device="cuda") for n in ("q", "k", "v")]
        ws = torch.empty(_lib.msa_workspace_bytes(shape, 2) // 4 + 1, device="cuda")

        def call():
            _lib.msa_sparse_prefill_backward(shape, x["q"], x["k"], x["v"], sel, out, lse, dout,
                                             *grads, ws)
    else:
        loss = torch.empty(1, device="cuda")
        grads = [torch.empty(x[n].shape, device="cuda") for n in ("idx_q", "idx_k")]
        ws = torch.empty(_lib.msa_workspace_bytes(shape, 3) // 4 + 1, device="cuda")

        def call():
            _lib.msa_index_kl_loss(shape, x["q"], x["k"], lse, x["idx_q"], x["idx_k"], sel, loss,
                                   *grads, ws)
    _lib.msa_debug_set_fault(1)
    try:
        call()
        with pytest.raises(_lib.MsaError) as ei:
            _lib.msa_get_device_status()
        assert ei.value.status == _lib.MSA_ERR_TIMEOUT
    finally:
        _lib.msa_debug_set_fault(0)
    _lib.msa_get_device_status()
    call()
    _lib.msa_get_device_status()
    if which == "backward":
        refs = oracle.sparse_attention_backward(x["q"], x["k"], x["v"], sel_np, dout, 128, 64)
    else:
        ref_loss, *refs = oracle.index_kl_loss(x["q"], x["k"], x["idx_q"], x["idx_k"], sel_np,
                                               128, 64)
    for got, ref in zip(grads, refs):
        check_grad(got, ref, "bf16", which)
