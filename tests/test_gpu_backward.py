"""Gradients of the sparse prefill attention (training path) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_02_gb300 import _lib
from block_sparse_gqa_02_gb300.configs import CONFIGS
from block_sparse_gqa_02_gb300.inputs import make_inputs, random_selection
from tests.parity import check_grad, sample_tiles

pytestmark = pytest.mark.gpu

CASES = {
    "tiny_f32": CONFIGS["tiny"],
    "f32_ragged_qt16": CONFIGS["tiny"].with_(seq=1000, q_tile=16, block_size=32, top_k=5),
    "bf16_ragged_1000": CONFIGS["p32k"].with_(seq=1000, top_k=4, n_plants=0),
    "bf16_d64_g16": CONFIGS["p32k"].with_(seq=2048, head_dim=64, n_heads_q=64, top_k=6),
    "bf16_4096_k16": CONFIGS["p32k"].with_(seq=4096, n_plants=0),
    "bf16_qt128_ragged": CONFIGS["p32k"].with_(seq=1500, q_tile=128, top_k=4, n_plants=0),
    # tensor-core path: G = 16, 4, 2; k = 1; and blocks selected by tiles of several dK/dV CTAs
    "bf16_g16_3000": CONFIGS["p32k"].with_(seq=3000, n_heads_q=64, top_k=8, n_plants=0),
    "bf16_g4_k1": CONFIGS["p32k"].with_(seq=1200, n_heads_q=16, top_k=1, n_plants=0),
    "bf16_g2_ragged": CONFIGS["p32k"].with_(seq=700, n_heads_q=8, top_k=3, n_plants=0),
    "bf16_8192_k32": CONFIGS["p32k"].with_(seq=8192, top_k=32, n_plants=0),
    "bf16_b2_ragged": CONFIGS["p32k"].with_(batch=2, seq=1100, top_k=4, n_plants=0),
    # the largest groups of the tensor-core backward: 32, 64 and 128 heads per KV head
    "bf16_g32_ragged": CONFIGS["p32k"].with_(seq=900, n_heads_q=128, top_k=3, n_plants=0),
    "bf16_g64_ragged": CONFIGS["p32k"].with_(seq=500, n_heads_q=256, top_k=3, n_plants=0),
    "bf16_g128_ragged": CONFIGS["p32k"].with_(seq=300, n_heads_q=512, top_k=2, n_plants=0),
}


@pytest.mark.parametrize("name", list(CASES))
def test_sparse_prefill_backward(name):
    cfg = CASES[name]
    x = make_inputs(cfg, device="cuda")
    shape = _lib.shape_from_config(cfg)
    cur = np.array([min(cfg.seq - 1, m * cfg.q_tile + cfg.q_tile - 1) // cfg.block_size
                    for m in range(shape.n_rows)])
    sel_np = random_selection(np.broadcast_to(cur + 1, (cfg.batch, 4, shape.n_rows)), cfg.top_k, 5)
    sel = torch.from_numpy(sel_np).cuda()
    gen = torch.Generator(device="cuda").manual_seed(99)
    dout = torch.randn(x["q"].shape, generator=gen, device="cuda").to(x["q"].dtype)
    out = torch.empty_like(x["q"])
    lse = torch.empty((cfg.batch, cfg.n_heads_q, cfg.seq), device="cuda")
    _lib.msa_sparse_prefill(shape, x["q"], x["k"], x["v"], sel, out, lse)
    dq = torch.full(x["q"].shape, float("nan"), device="cuda")
    dk = torch.full(x["k"].shape, float("nan"), device="cuda")
    dv = torch.full(x["v"].shape, float("nan"), device="cuda")
    ws_bytes = _lib.msa_workspace_bytes(shape, 2)
    ws = torch.full((ws_bytes // 4 + 1,), float("nan"), device="cuda") if ws_bytes else None
    _lib.msa_sparse_prefill_backward(shape, x["q"], x["k"], x["v"], sel, out, lse, dout,
                                     dq, dk, dv, ws)
    _lib.msa_get_device_status()
    rq, rk, rv = oracle.sparse_attention_backward(x["q"], x["k"], x["v"], sel_np, dout,
                                                  cfg.block_size, cfg.q_tile)
    check_grad(dq, rq, cfg.dtype, f"{name} dq")
    check_grad(dk, rk, cfg.dtype, f"{name} dk")
    check_grad(dv, rv, cfg.dtype, f"{name} dv")


KL_CASES = {
    "tiny_f32": CONFIGS["tiny"],
    "bf16_ragged_1000": CONFIGS["p32k"].with_(seq=1000, top_k=4, n_plants=3),
    "bf16_d64_di64_g16": CONFIGS["p32k"].with_(seq=2048, head_dim=64, index_dim=64,
                                               n_heads_q=64, top_k=6, block_size=64),
    "bf16_4096_k16": CONFIGS["p32k"].with_(seq=4096, n_plants=5),
    "bf16_qt128_ragged": CONFIGS["p32k"].with_(seq=1500, q_tile=128, top_k=4, n_plants=2),
    # tensor-core path: G = 2, 4, 16, 32; and blocks shared by the tiles of several CTAs
    "bf16_g16_3000": CONFIGS["p32k"].with_(seq=3000, n_heads_q=64, top_k=8, n_plants=3),
    "bf16_g4_k1": CONFIGS["p32k"].with_(seq=1200, n_heads_q=16, top_k=1, n_plants=0),
    "bf16_g2_ragged": CONFIGS["p32k"].with_(seq=700, n_heads_q=8, top_k=3, n_plants=0),
    "bf16_g32_ragged": CONFIGS["p32k"].with_(seq=900, n_heads_q=128, top_k=3, n_plants=0),
    "bf16_g64_ragged": CONFIGS["p32k"].with_(seq=500, n_heads_q=256, top_k=3, n_plants=0),
    "bf16_8192_k32": CONFIGS["p32k"].with_(seq=8192, top_k=32, n_plants=4),
    # the normaliser pass (G >= 8) takes two tiles per CTA over the union of their
    # selections: k = 1 (the two tiles of a block share their current block) with an odd
    # tile count (the last CTA holds one tile), and a wider union at G = 16
    "bf16_g8_k1_odd_tiles": CONFIGS["p32k"].with_(seq=1300, top_k=1, n_plants=0),
    "bf16_g16_k24": CONFIGS["p32k"].with_(seq=2000, n_heads_q=64, top_k=24, n_plants=2),
    "bf16_b2_ragged": CONFIGS["p32k"].with_(batch=2, seq=1100, top_k=4, n_plants=2),
}


@pytest.mark.parametrize("name", list(KL_CASES))
def test_index_kl_loss(name):
    cfg = KL_CASES[name]
    x = make_inputs(cfg, device="cuda")
    shape = _lib.shape_from_config(cfg)
    cur = np.array([min(cfg.seq - 1, m * cfg.q_tile + cfg.q_tile - 1) // cfg.block_size
                    for m in range(shape.n_rows)])
    sel_np = random_selection(np.broadcast_to(cur + 1, (cfg.batch, 4, shape.n_rows)), cfg.top_k, 6)
    sel = torch.from_numpy(sel_np).cuda()
    out = torch.empty_like(x["q"])
    lse = torch.empty((cfg.batch, cfg.n_heads_q, cfg.seq), device="cuda")
    _lib.msa_sparse_prefill(shape, x["q"], x["k"], x["v"], sel, out, lse)
    loss = torch.full((1,), float("nan"), device="cuda")
    diq = torch.full(x["idx_q"].shape, float("nan"), device="cuda")
    dik = torch.full(x["idx_k"].shape, float("nan"), device="cuda")
    ws_bytes = _lib.msa_workspace_bytes(shape, 3)
    ws = torch.full((ws_bytes // 4 + 1,), float("nan"), device="cuda") if ws_bytes else None
    _lib.msa_index_kl_loss(shape, x["q"], x["k"], lse, x["idx_q"], x["idx_k"], sel, loss,
                           diq, dik, ws)
    _lib.msa_get_device_status()
    ref_loss, ref_q, ref_k = oracle.index_kl_loss(x["q"], x["k"], x["idx_q"], x["idx_k"],
                                                  sel_np, cfg.block_size, cfg.q_tile)
    tol = "f32" if cfg.dtype == "f32" else "bf16"
    check_grad(diq, ref_q, tol, f"{name} d idx_q")
    check_grad(dik, ref_k, tol, f"{name} d idx_k")
    # the loss sums one KL per (token, KV head); each is evaluated in fp32 from normalised
    # probabilities whose sum is 1 only to fp32 rounding, which leaves an absolute error of
    # order 1e-7 per term: near-uniform inputs give KLs of that order, so the bound has an
    # absolute part per term beside the relative one
    n_terms = cfg.batch * cfg.seq * cfg.n_heads_kv
    assert abs(loss.item() - ref_loss) <= 1e-3 * abs(ref_loss) + 1e-6 * n_terms, \
        (loss.item(), ref_loss)


def test_training_p32k_sampled():
    """The 32K workload the bench times, run in full on the GPU: the tensor-core backward and
    index KL against the oracle on sampled query tiles (dq, d idx_q) and sampled key blocks
    (dk, dv, d idx_k; late blocks, which few tiles select, so that the oracle's sampled
    evaluation stays short), on a seeded selection of 16 blocks per (tile, KV head)."""
    cfg = CONFIGS["p32k"]
    x = make_inputs(cfg, device="cuda")
    shape = _lib.shape_from_config(cfg)
    nR, nB = shape.n_rows, shape.n_blocks
    cur = np.array([min(cfg.seq - 1, m * cfg.q_tile + cfg.q_tile - 1) // cfg.block_size
                    for m in range(nR)])
    sel_np = random_selection(np.broadcast_to(cur + 1, (1, 4, nR)), cfg.top_k, 9)
    sel = torch.from_numpy(sel_np).cuda()
    out = torch.empty_like(x["q"])
    lse = torch.empty((1, cfg.n_heads_q, cfg.seq), device="cuda")
    _lib.msa_sparse_prefill(shape, x["q"], x["k"], x["v"], sel, out, lse)
    gen = torch.Generator(device="cuda").manual_seed(11)
    dout = torch.randn(x["q"].shape, generator=gen, device="cuda").to(x["q"].dtype)
    grads = [torch.empty(x[n].shape, device="cuda") for n in ("q", "k", "v")]
    ws = torch.empty(_lib.msa_workspace_bytes(shape, 2) // 4 + 1, device="cuda")
    _lib.msa_sparse_prefill_backward(shape, x["q"], x["k"], x["v"], sel, out, lse, dout,
                                     *grads, ws)
    loss = torch.empty(1, device="cuda")
    kl_grads = [torch.empty(x[n].shape, device="cuda") for n in ("idx_q", "idx_k")]
    ws = torch.empty(_lib.msa_workspace_bytes(shape, 3) // 4 + 1, device="cuda")
    _lib.msa_index_kl_loss(shape, x["q"], x["k"], lse, x["idx_q"], x["idx_k"], sel, loss,
                           *kl_grads, ws)
    _lib.msa_get_device_status()
    tiles = sample_tiles(nR, seed=13)
    blocks = [nB - 1, nB - 4, nB - 56]
    rows = torch.from_numpy(np.concatenate(
        [np.arange(m * cfg.q_tile, (m + 1) * cfg.q_tile) for m in tiles])).cuda()
    keys = torch.from_numpy(np.concatenate(
        [np.arange(b * cfg.block_size, (b + 1) * cfg.block_size) for b in blocks])).cuda()
    rq, rk, rv = oracle.sparse_attention_backward(x["q"], x["k"], x["v"], sel_np, dout,
                                                  cfg.block_size, cfg.q_tile, tiles=tiles,
                                                  key_blocks=blocks)
    r_rows, r_keys = rows.cpu().numpy(), keys.cpu().numpy()
    check_grad(grads[0].index_select(1, rows), rq[:, r_rows], "bf16", "p32k dq")
    check_grad(grads[1].index_select(2, keys), rk[:, :, r_keys], "bf16", "p32k dk")
    check_grad(grads[2].index_select(2, keys), rv[:, :, r_keys], "bf16", "p32k dv")
    _, riq, rik = oracle.index_kl_loss(x["q"], x["k"], x["idx_q"], x["idx_k"], sel_np,
                                       cfg.block_size, cfg.q_tile, tiles=tiles,
                                       key_blocks=blocks)
    check_grad(kl_grads[0].index_select(1, rows), riq[:, r_rows], "bf16", "p32k d idx_q")
    check_grad(kl_grads[1].index_select(1, keys), rik[:, r_keys], "bf16", "p32k d idx_k")
    assert np.isfinite(loss.item()) and loss.item() > 0
