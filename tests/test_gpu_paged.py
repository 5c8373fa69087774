"""Parity of the paged, ragged decode (per-sequence cache lengths, block tables into
physical pools) with the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_02_gb300 import _lib
from block_sparse_gqa_02_gb300.configs import CONFIGS
from block_sparse_gqa_02_gb300.inputs import make_paged_decode_inputs
from tests.parity import (check_lse, check_out, check_scores, check_selection_exact,
                          check_selection_valid, to_np)

pytestmark = pytest.mark.gpu


def _run_paged(cfg, lens, seed=0):
    x = make_paged_decode_inputs(cfg, lens, device="cuda", seed=seed)
    shape = _lib.shape_from_config(cfg, batch=len(lens))
    B, nB = len(lens), shape.n_blocks
    scores = torch.empty((B, 4, 1, nB), dtype=torch.float32, device="cuda")
    sel = torch.empty((B, 4, 1, cfg.top_k), dtype=torch.int32, device="cuda")
    out = torch.empty_like(x["q"])
    lse = torch.empty((B, cfg.n_heads_q, 1), dtype=torch.float32, device="cuda")
    ws = torch.empty(_lib.msa_workspace_bytes(shape, 1) // 4 + 4, dtype=torch.float32,
                     device="cuda")
    _lib.msa_index_scores_paged(shape, x["seq_lens"], x["block_table"], x["n_phys"], x["idx_q"],
                                x["idx_k_pool"], scores)
    _lib.msa_block_topk_ragged(shape, x["seq_lens"], scores, sel)
    _lib.msa_sparse_decode_paged(shape, x["seq_lens"], x["block_table"], x["n_phys"], x["q"],
                                 x["k_pool"], x["v_pool"], sel, out, lse, ws)
    _lib.msa_get_device_status()
    ref = oracle.msa_decode_paged(x["q"], x["k_pool"], x["v_pool"], x["idx_q"], x["idx_k_pool"],
                                  x["seq_lens"].cpu().numpy(), x["block_table"].cpu().numpy(),
                                  cfg.block_size, cfg.top_k, nB)
    return x, (to_np(scores), to_np(sel), to_np(out), to_np(lse)), ref


LENS = {
    "ragged_small": [1, 127, 128, 129, 4097, 9000],
    "ragged_with_empty": [0, 5000, 1, 70001],
    "ragged_long": [1 << 18, 123457, 65536, 3],
    # the scan shares its CTAs out by length: one long cache takes most of them
    "one_long_many_short": [200_000] + [1 + 37 * i for i in range(19)],
    # more than 2048 blocks in the longest cache (the top-k's long-row form)
    "past_2048_blocks": [300_000, 64 * 128, 64 * 128 + 1, 0, 4097],
    # more sequences than SMs: the scan falls back to splitting each sequence evenly
    "more_sequences_than_sms": [1 + (97 * i) % 700 for i in range(160)],
}


@pytest.mark.parametrize("name", list(LENS))
def test_paged_ragged_decode(name):
    lens = LENS[name]
    cfg = CONFIGS["d1m"].with_(seq=max(lens) + 300, top_k=16, n_plants=0)
    x, (g_sc, g_sel, g_o, g_l), (sc, sel, o, l) = _run_paged(cfg, lens, seed=len(lens))
    check_scores(g_sc, sc, name)
    cb = np.array([[max(L - 1, 0) // 128] * 4 for L in lens])[:, :, None]
    agree = check_selection_valid(g_sel, sel, sc, np.broadcast_to(cb, g_sel.shape[:-1]), name)
    assert agree >= 0.9
    for b, L in enumerate(lens):
        if L == 0:
            continue
        # the selection bit-exactly against the oracle's top-k on the GPU's own fp32 scores
        # of this sequence's blocks; then the attention over the GPU's selection, on the
        # sequence's logical cache (the input pools' blocks in block-table order; the oracle
        # reads only the selected keys)
        nb = -(-L // 128)
        check_selection_exact(g_sel[b:b + 1],
                              oracle.block_topk_decode(g_sc[b:b + 1, :, :, :nb], L, 128,
                                                       cfg.top_k), f"{name} seq {b}")
        phys = x["block_table"][b, :nb].long()
        kc, vc = (x[n][phys].transpose(0, 1).reshape(4, nb * 128, -1)[:, :L]
                  for n in ("k_pool", "v_pool"))        # [Hkv, L, d], inputs rearranged
        ref_o, ref_l = oracle.sparse_attention(x["q"][b:b + 1], kc[None], vc[None],
                                               g_sel[b:b + 1], 128, 1, None, L - 1)
        check_out(g_o[b:b + 1], ref_o, "bf16", f"{name} seq {b}")
        check_lse(g_l[b:b + 1], ref_l, "bf16", f"{name} seq {b}")
    # an empty sequence selects nothing and attends to nothing
    for b, L in enumerate(lens):
        if L == 0:
            assert np.all(g_sel[b] == -1) and np.all(g_o[b] == 0) and np.all(np.isneginf(g_l[b]))


def test_paged_matches_contiguous_decode():
    """Identity table over a pool laid out like the contiguous cache: both paths agree."""
    cfg = CONFIGS["d1m"].with_(batch=3, seq=20480, top_k=12, n_plants=0)
    lens = [20480] * 3
    x = make_paged_decode_inputs(cfg, lens, device="cuda", seed=7, spare_blocks=0)
    B, P, nB = 3, x["n_phys"], cfg.n_blocks
    table = torch.arange(B * nB, dtype=torch.int32, device="cuda").view(B, nB)
    # contiguous caches [B, Hkv, L, d] built from the pool in table order
    k_c = x["k_pool"].view(B, nB, 4, 128, 128).permute(0, 2, 1, 3, 4).reshape(B, 4, nB * 128, 128).contiguous()
    v_c = x["v_pool"].view(B, nB, 4, 128, 128).permute(0, 2, 1, 3, 4).reshape(B, 4, nB * 128, 128).contiguous()
    ik_c = x["idx_k_pool"].view(B, nB * 128, 128).contiguous()
    shape = _lib.shape_from_config(cfg)
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    res = []
    for paged in (False, True):
        sc = torch.empty((B, 4, 1, nB), device="cuda")
        sel = torch.empty((B, 4, 1, 12), dtype=torch.int32, device="cuda")
        out = torch.empty_like(x["q"])
        lse = torch.empty((B, 64, 1), device="cuda")
        ws = torch.empty(_lib.msa_workspace_bytes(shape, 1) // 4 + 4, device="cuda")
        if paged:
            _lib.msa_index_scores_paged(shape, lens_t, table, P, x["idx_q"], x["idx_k_pool"], sc)
            _lib.msa_block_topk_ragged(shape, lens_t, sc, sel)
            _lib.msa_sparse_decode_paged(shape, lens_t, table, P, x["q"], x["k_pool"],
                                         x["v_pool"], sel, out, lse, ws)
        else:
            _lib.msa_index_scores(shape, x["idx_q"], ik_c, sc)
            _lib.msa_block_topk(shape, sc, sel)
            _lib.msa_sparse_decode(shape, x["q"], k_c, v_c, sel, out, lse, ws)
        torch.cuda.synchronize()
        res.append((sc, sel, out, lse))
    assert torch.equal(res[0][0], res[1][0])
    assert torch.equal(res[0][1], res[1][1])
    assert torch.equal(res[0][2], res[1][2])
    assert torch.equal(res[0][3], res[1][3])
