"""Fused index scores + streaming top-k against the two-call path and the oracle."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_02_gb300 import _lib
from block_sparse_gqa_02_gb300.configs import CONFIGS
from block_sparse_gqa_02_gb300.inputs import make_inputs
from tests.parity import (check_scores, check_selection_exact, check_selection_valid,
                          sample_tiles, to_np)

pytestmark = pytest.mark.gpu

CASES = {
    "ragged_1000_k4": CONFIGS["p32k"].with_(seq=1000, top_k=4, n_plants=3),
    "8192_k16": CONFIGS["p32k"].with_(seq=8192, n_plants=5),
    "k1": CONFIGS["p32k"].with_(seq=3000, top_k=1, n_plants=2),
    "k256": CONFIGS["p32k"].with_(seq=40000, top_k=256, n_plants=8),
    "p128k": CONFIGS["p128k"],
    "batch2_ragged": CONFIGS["p32k"].with_(batch=2, seq=2500, top_k=6, n_plants=3),
}


@pytest.mark.parametrize("name", list(CASES))
def test_fused_matches_two_calls_and_oracle(name):
    cfg = CASES[name]
    x = make_inputs(cfg, device="cuda")
    shape = _lib.shape_from_config(cfg)
    dims = (cfg.batch, 4, shape.n_rows)
    sc2 = torch.empty(dims + (shape.n_blocks,), device="cuda")
    sel2 = torch.empty(dims + (cfg.top_k,), dtype=torch.int32, device="cuda")
    _lib.msa_index_scores(shape, x["idx_q"], x["idx_k"], sc2)
    _lib.msa_block_topk(shape, sc2, sel2)
    sc1 = torch.full_like(sc2, 7.0)
    sel1 = torch.full_like(sel2, -7)
    _lib.msa_index_topk_fused(shape, x["idx_q"], x["idx_k"], sel1, sc1)
    sel0 = torch.full_like(sel2, -7)
    _lib.msa_index_topk_fused(shape, x["idx_q"], x["idx_k"], sel0)        # no scores
    _lib.msa_get_device_status()
    assert torch.equal(sc1, sc2)
    assert torch.equal(sel1, sel2)
    assert torch.equal(sel0, sel2)
    tiles = sample_tiles(shape.n_rows, seed=8)
    ref_sc = oracle.index_block_scores_prefill(x["idx_q"], x["idx_k"], 128, 64, tiles=tiles)
    ref_sel = oracle.block_topk_prefill(ref_sc, cfg.seq, 64, 128, cfg.top_k, tiles=tiles)
    r_idx = torch.tensor(tiles, device="cuda")
    g_sc = to_np(sc1.index_select(2, r_idx))
    check_scores(g_sc, ref_sc, name)
    cb = np.array([(min(cfg.seq - 1, m * 64 + 63)) // 128 for m in tiles])
    g_sel = to_np(sel0.index_select(2, r_idx))
    # bit-exact against the oracle's top-k on the GPU's own fp32 scores
    check_selection_exact(g_sel, oracle.block_topk_prefill(g_sc, cfg.seq, 64, 128, cfg.top_k,
                                                           tiles=tiles), name)
    assert check_selection_valid(g_sel, ref_sel, ref_sc,
                                 np.broadcast_to(cb, g_sel.shape[:-1]), name) >= 0.9
