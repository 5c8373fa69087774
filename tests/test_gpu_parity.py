"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, element by element.

Each stage is tested on its own with seeded inputs from the generator (so no oracle
input ever comes from the CUDA path), and the three stages are tested chained.  Small
ragged shapes are compared in full; the full-size configurations are run in full on the
GPU, in the launch configuration the benchmark times, and compared on sampled tiles.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_02_gb300 import _lib
from block_sparse_gqa_02_gb300.api import (alloc_decode_outputs, alloc_prefill_outputs,
                                           run_decode, run_prefill)
from block_sparse_gqa_02_gb300.configs import CONFIGS
from block_sparse_gqa_02_gb300.inputs import (add_score_ramp, make_inputs,
                                              random_block_scores, random_selection)
from tests.parity import (check_lse, check_out, check_scores, check_selection_exact,
                          check_selection_valid, sample_tiles, to_np)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def cur_blocks(shape):
    """Current block of every selection row (oracle's rule)."""
    if shape.seq_q == 1 and shape.q_tile == 1:
        return np.array([oracle.current_block(shape.seq_k - 1, shape.block_size)])
    return np.array([oracle.current_block(min(shape.seq_q - 1, m * shape.q_tile + shape.q_tile - 1),
                                          shape.block_size) for m in range(shape.n_rows)])


def small_cfg(name, **kw):
    return CONFIGS[name].with_(**kw)


# ----------------------------------------------------------------------- top-k

TOPK_CASES = [
    # (label, batch, seq, block, q_tile, top_k, kind)
    ("tiny", 1, 1024, 64, 64, 4, "normal"),
    ("ties", 1, 4096, 64, 64, 6, "ties"),
    ("mixed_ragged", 2, 5000, 128, 64, 16, "mixed"),
    ("k1", 1, 2048, 128, 64, 1, "normal"),
    ("k_exceeds_candidates", 1, 3000, 64, 32, 40, "mixed"),
    ("p32k", 1, 32768, 128, 64, 16, "mixed"),
    ("p128k", 1, 131072, 128, 64, 32, "normal"),
    ("q_tile1", 1, 700, 16, 1, 5, "ties"),
]


@pytest.mark.parametrize("case", TOPK_CASES, ids=[c[0] for c in TOPK_CASES])
def test_topk_bit_exact(case):
    label, B, T, bs, qt, k, kind = case
    seed = TOPK_CASES.index(case)
    shape = _lib.make_shape(B, T, T, 4 * 4, 4, 64, 64, bs, k, qt, "bf16")
    sc = random_block_scores((B, 4, shape.n_rows, shape.n_blocks), seed=seed,
                             kind=kind)
    sel = torch.full((B, 4, shape.n_rows, k), -7, dtype=torch.int32, device=DEV)
    _lib.msa_block_topk(shape, torch.from_numpy(sc).to(DEV), sel)
    torch.cuda.synchronize()
    ref = oracle.block_topk_prefill(sc, T, qt, bs, k)
    got = sel.cpu().numpy()
    bad = np.argwhere(np.any(got != ref, axis=-1))
    assert bad.size == 0, f"{len(bad)} rows differ, e.g. {bad[:2].tolist()}: " \
        f"{got[tuple(bad[0])]} vs {ref[tuple(bad[0])]}"


@pytest.mark.parametrize("kind", ["normal", "ties", "mixed"])
def test_topk_shared_bit_exact(kind):
    """The aggregated (shared across heads) selection used for the ablation."""
    T, bs, qt, k = 20000, 128, 64, 16
    shape = _lib.make_shape(2, T, T, 32, 4, 128, 128, bs, k, qt, "bf16")
    sc = random_block_scores((2, 4, shape.n_rows, shape.n_blocks), seed=11, kind=kind)
    sel = torch.full((2, 4, shape.n_rows, k), -7, dtype=torch.int32, device=DEV)
    _lib.msa_block_topk_shared(shape, torch.from_numpy(sc).to(DEV), sel)
    ref = oracle.block_topk_shared_prefill(sc, T, qt, bs, k)
    assert np.array_equal(sel.cpu().numpy(), ref)


def test_topk_token_level_bit_exact():
    """Token-level selection (block size 1, one query per row), the other ablation."""
    T, k = 3000, 200
    shape = _lib.make_shape(1, T, T, 16, 4, 64, 64, 1, k, 1, "bf16")
    sc = random_block_scores((1, 4, T, T), seed=12, kind="mixed")
    sel = torch.empty((1, 4, T, k), dtype=torch.int32, device=DEV)
    _lib.msa_block_topk(shape, torch.from_numpy(sc).to(DEV), sel)
    rows = sample_tiles(T, n_random=40, seed=4)
    ref = oracle.block_topk_prefill(sc[:, :, rows], T, 1, 1, k, tiles=rows)
    assert np.array_equal(sel.cpu().numpy()[:, :, rows], ref)


@pytest.mark.parametrize("kind", ["normal", "ties"])
def test_topk_decode_1m_bit_exact(kind):
    B, L, bs, k = 8, 1 << 20, 128, 64
    shape = _lib.make_shape(B, 1, L, 64, 4, 128, 128, bs, k, 1, "bf16")
    sc = random_block_scores((B, 4, 1, shape.n_blocks), seed=5, kind=kind)
    sel = torch.empty((B, 4, 1, k), dtype=torch.int32, device=DEV)
    _lib.msa_block_topk(shape, torch.from_numpy(sc).to(DEV), sel)
    ref = oracle.block_topk_decode(sc, L, bs, k)
    assert np.array_equal(sel.cpu().numpy(), ref)


def test_topk_1m_prefill_rows_bit_exact():
    """Rows of a 1M prefill (up to 8192 candidates each), sampled for the oracle."""
    T, bs, qt, k = 1 << 20, 128, 128, 64
    shape = _lib.make_shape(1, T, T, 64, 4, 128, 128, bs, k, qt, "bf16")
    sc = random_block_scores((1, 4, shape.n_rows, shape.n_blocks), seed=9, kind="mixed")
    sel = torch.empty((1, 4, shape.n_rows, k), dtype=torch.int32, device=DEV)
    _lib.msa_block_topk(shape, torch.from_numpy(sc).to(DEV), sel)
    got = sel.cpu().numpy()
    rows = sample_tiles(shape.n_rows, n_random=12, seed=3)
    ref = oracle.block_topk_prefill(sc[:, :, rows], T, qt, bs, k, tiles=rows)
    assert np.array_equal(got[:, :, rows], ref)


@pytest.mark.parametrize("k", [2, 64, 257, 258])
def test_topk_long_rows_k_bit_exact(k):
    """Rows of more than 2048 candidates (the 1024-thread form of the kernel) at k = 2,
    the decode bench's k, and k past 256."""
    B, L, bs = 2, 3001 * 128 - 5, 128
    shape = _lib.make_shape(B, 1, L, 64, 4, 128, 128, bs, k, 1, "bf16")
    sc = random_block_scores((B, 4, 1, shape.n_blocks), seed=20 + k, kind="mixed")
    sel = torch.full((B, 4, 1, k), -7, dtype=torch.int32, device=DEV)
    _lib.msa_block_topk(shape, torch.from_numpy(sc).to(DEV), sel)
    assert np.array_equal(sel.cpu().numpy(), oracle.block_topk_decode(sc, L, bs, k))


def test_topk_long_rows_equal_scores_bit_exact():
    """Every candidate of a row equal (+0 and -0 mixed; a constant), so every digit of the
    select ties and the lowest block indices are kept."""
    B, L, bs, k = 2, 2600 * 128, 128, 64
    shape = _lib.make_shape(B, 1, L, 64, 4, 128, 128, bs, k, 1, "bf16")
    rng = np.random.default_rng(21)
    sc = np.where(rng.random((B, 4, 1, shape.n_blocks)) < 0.5, 0.0, -0.0).astype(np.float32)
    sc[1, 2] = 1.5
    sc[1, 3, 0, 2000:] = -2.0                   # equal within the row's last quarters
    sel = torch.full((B, 4, 1, k), -7, dtype=torch.int32, device=DEV)
    _lib.msa_block_topk(shape, torch.from_numpy(sc).to(DEV), sel)
    assert np.array_equal(sel.cpu().numpy(), oracle.block_topk_decode(sc, L, bs, k))


def test_topk_ragged_long_rows_bit_exact():
    """Ragged decode rows under a maximum of more than 2048 blocks: empty, shorter than k,
    exactly k, one past k, and long."""
    k, bs = 64, 128
    lens = [0, 1, 63 * bs + 5, 64 * bs, 64 * bs + 1, 66 * bs + 3, 128 * bs, 5000, 2100 * bs,
            2345 * bs - 17]
    B = len(lens)
    shape = _lib.make_shape(B, 1, max(lens), 64, 4, 128, 128, bs, k, 1, "bf16")
    sc = random_block_scores((B, 4, 1, shape.n_blocks), seed=22, kind="ties")
    sel = torch.full((B, 4, 1, k), -7, dtype=torch.int32, device=DEV)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=DEV)
    _lib.msa_block_topk_ragged(shape, lens_t, torch.from_numpy(sc).to(DEV), sel)
    got = sel.cpu().numpy()
    for b, L in enumerate(lens):
        ref = (np.full((1, 4, 1, k), -1, dtype=np.int32) if L == 0 else
               oracle.block_topk_decode(sc[b:b + 1], L, bs, k))
        assert np.array_equal(got[b:b + 1], ref), f"sequence {b} (length {L})"


# -------------------------------------------------------------- index scores

def _index_case(cfg, tiles=None):
    x = make_inputs(cfg, device=DEV)
    shape = _lib.shape_from_config(cfg)
    scores = torch.empty((cfg.batch, cfg.n_heads_kv, shape.n_rows, shape.n_blocks),
                         dtype=torch.float32, device=DEV)
    _lib.msa_index_scores(shape, x["idx_q"], x["idx_k"], scores)
    torch.cuda.synchronize()
    if cfg.mode == "decode":
        ref = oracle.index_block_scores_decode(x["idx_q"], x["idx_k"], cfg.block_size)
        return to_np(scores), ref
    ref = oracle.index_block_scores_prefill(x["idx_q"], x["idx_k"], cfg.block_size, cfg.q_tile,
                                            tiles=tiles)
    if tiles is None:
        return to_np(scores), ref
    return to_np(scores.index_select(2, torch.tensor(tiles, device=DEV))), ref


INDEX_CASES = {
    "tiny_f32": lambda: small_cfg("tiny"),
    "f32_ragged_qt16": lambda: small_cfg("tiny", seq=1000, q_tile=16, block_size=32),
    "bf16_ragged_1000": lambda: small_cfg("p32k", seq=1000, n_plants=3),
    "bf16_4096_d64": lambda: small_cfg("p32k", seq=4096, index_dim=64, block_size=64),
    "bf16_8192": lambda: small_cfg("p32k", seq=8192, n_plants=5),
    "bf16_b2_ragged": lambda: small_cfg("p32k", batch=2, seq=1300, n_plants=3),
    "decode_ragged": lambda: small_cfg("d1m", batch=2, seq=5000, n_plants=4),
    "decode_tiny_cache": lambda: small_cfg("d1m", batch=3, seq=77, n_plants=0),
    "decode_f32": lambda: small_cfg("d1m", batch=3, seq=3001, dtype="f32", index_dim=64,
                                    n_plants=2),
}


@pytest.mark.parametrize("name", list(INDEX_CASES))
def test_index_scores(name):
    got, ref = _index_case(INDEX_CASES[name]())
    check_scores(got, ref, name)


def test_index_scores_p32k_sampled():
    cfg = CONFIGS["p32k"]
    tiles = sample_tiles(cfg.n_tiles, seed=1)
    got, ref = _index_case(cfg, tiles)
    check_scores(got, ref, "p32k")


def test_index_scores_d1m_full():
    got, ref = _index_case(CONFIGS["d1m"])
    check_scores(got, ref, "d1m")


# ----------------------------------------------------------- sparse attention

def _attn_case(cfg, sel_seed=0, tiles=None):
    x = make_inputs(cfg, device=DEV)
    shape = _lib.shape_from_config(cfg)
    ncand = cur_blocks(shape) + 1
    sel_np = random_selection(np.broadcast_to(ncand, (cfg.batch, cfg.n_heads_kv, len(ncand))),
                              cfg.top_k, sel_seed)
    sel = torch.from_numpy(sel_np).to(DEV)
    out = torch.empty_like(x["q"])
    lse = torch.empty((cfg.batch, cfg.n_heads_q, cfg.seq_q), dtype=torch.float32, device=DEV)
    if cfg.mode == "decode":
        nbytes = _lib.msa_workspace_bytes(shape, 1)
        ws = torch.empty(nbytes // 4 + 4, dtype=torch.float32, device=DEV)
        _lib.msa_sparse_decode(shape, x["q"], x["k"], x["v"], sel, out, lse, ws)
        torch.cuda.synchronize()
        ref_o, ref_l = oracle.sparse_attention(x["q"], x["k"], x["v"], sel_np, cfg.block_size, 1,
                                               None, cfg.seq - 1)
        return to_np(out), to_np(lse), ref_o, ref_l
    _lib.msa_sparse_prefill(shape, x["q"], x["k"], x["v"], sel, out, lse)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.sparse_attention(x["q"], x["k"], x["v"], sel_np, cfg.block_size,
                                           cfg.q_tile, None, 0, tiles)
    if tiles is None:
        return to_np(out), to_np(lse), ref_o, ref_l
    rows = np.concatenate([np.arange(m * cfg.q_tile, min(cfg.seq, (m + 1) * cfg.q_tile))
                           for m in tiles])
    r_idx = torch.from_numpy(rows).to(DEV)
    return to_np(out.index_select(1, r_idx)), to_np(lse.index_select(2, r_idx)), ref_o, ref_l


ATTN_CASES = {
    "tiny_f32": lambda: small_cfg("tiny"),
    "f32_ragged": lambda: small_cfg("tiny", seq=1000, q_tile=16, block_size=32, top_k=5),
    "bf16_ragged_1000": lambda: small_cfg("p32k", seq=1000, top_k=4, n_plants=3),
    "bf16_d64_g16": lambda: small_cfg("p32k", seq=2048, head_dim=64, n_heads_q=64, top_k=6),
    "bf16_4096_k16": lambda: small_cfg("p32k", seq=4096),
    "bf16_g4_ragged": lambda: small_cfg("p32k", seq=2000, n_heads_q=16, top_k=7),
    "bf16_g32": lambda: small_cfg("p32k", seq=1100, n_heads_q=128, top_k=3),
    # the largest groups the tensor-core prefill takes: 64 and 128 query heads per KV head
    # (a Q tile of 128 rows is then 2 tokens, or 1)
    "bf16_g64": lambda: small_cfg("p32k", seq=600, n_heads_q=256, top_k=3, n_plants=0),
    "bf16_g128": lambda: small_cfg("p32k", seq=333, n_heads_q=512, top_k=2, n_plants=0),
    "bf16_g16_k1": lambda: small_cfg("p32k", seq=700, n_heads_q=64, top_k=1),
    "bf16_b2_ragged": lambda: small_cfg("p32k", batch=2, seq=1300, top_k=5),
    # one partial query tile over one partial key block
    "bf16_t50": lambda: small_cfg("p32k", seq=50, top_k=2, n_plants=0),
    "decode_ragged": lambda: small_cfg("d1m", batch=2, seq=5000, top_k=8, n_plants=4),
    "decode_f32": lambda: small_cfg("d1m", batch=3, seq=3001, dtype="f32", top_k=5,
                                    head_dim=64, n_plants=2),
    "decode_short_cache": lambda: small_cfg("d1m", batch=2, seq=200, top_k=64, n_plants=0),
    "decode_one_key": lambda: small_cfg("d1m", batch=2, seq=1, top_k=4, n_plants=0),
    "decode_g8": lambda: small_cfg("d1m", batch=3, seq=9000, n_heads_q=32, top_k=12,
                                   n_plants=4),
    "decode_g4_k3": lambda: small_cfg("d1m", batch=5, seq=1000, n_heads_q=16, top_k=3,
                                      n_plants=2),
    # more query heads per KV head than the tensor-core decode's 16 rows
    "decode_g32": lambda: small_cfg("d1m", batch=2, seq=3000, n_heads_q=128, top_k=6,
                                    n_plants=2),
}


@pytest.mark.parametrize("name", list(ATTN_CASES))
def test_sparse_attention(name):
    cfg = ATTN_CASES[name]()
    got_o, got_l, ref_o, ref_l = _attn_case(cfg)
    check_out(got_o, ref_o, cfg.dtype, name)
    check_lse(got_l, ref_l, cfg.dtype, name)


@pytest.mark.parametrize("per_key", [0.05, 0.75, 3.0])
def test_prefill_rows_rescale_unevenly(per_key):
    """Even heads' row maxima climb by ~6 (0.05 per key), ~94 (0.75) or ~380 logits per
    block while odd heads' stay flat: rows of one warp take the rescaling path and rows
    beside them do not.  At 0.05 per key a later block lifts every key of an even head a
    little (0.8 in log2 units per block), so its P sum passes the streaming path's bound
    long before any single P would pass 2^8; at 0.75 and 3.0 single keys pass it by far."""
    cfg = small_cfg("p32k", seq=2000, top_k=6, n_plants=0)
    x = add_score_ramp(make_inputs(cfg, device=DEV), per_key, seed=3)
    shape = _lib.shape_from_config(cfg)
    ncand = cur_blocks(shape) + 1
    sel_np = random_selection(np.broadcast_to(ncand, (1, 4, len(ncand))), cfg.top_k, 4)
    sel = torch.from_numpy(sel_np).to(DEV)
    out = torch.empty_like(x["q"])
    lse = torch.empty((1, cfg.n_heads_q, cfg.seq), dtype=torch.float32, device=DEV)
    _lib.msa_sparse_prefill(shape, x["q"], x["k"], x["v"], sel, out, lse)
    _lib.msa_get_device_status()
    ref_o, ref_l = oracle.sparse_attention(x["q"], x["k"], x["v"], sel_np, cfg.block_size,
                                           cfg.q_tile)
    check_out(out, ref_o, "bf16", f"ramp {per_key}")
    # lse grows with the logits (to ~130 and ~520 here): the fp32 accumulation of Q.K^T
    # adds an error proportional to it
    lse_ref = np.asarray(ref_l)
    tol = 2e-3 + 1e-4 * np.abs(lse_ref)
    got = to_np(lse)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(got))
    assert np.all(np.abs(got[fin] - lse_ref[fin]) <= tol[fin])


def test_sparse_prefill_p32k_sampled():
    cfg = CONFIGS["p32k"]
    tiles = sample_tiles(cfg.n_tiles, seed=2)
    got_o, got_l, ref_o, ref_l = _attn_case(cfg, tiles=tiles)
    check_out(got_o, ref_o, "bf16", "p32k")
    check_lse(got_l, ref_l, "bf16", "p32k")


def test_sparse_decode_d1m_full():
    cfg = CONFIGS["d1m"]
    got_o, got_l, ref_o, ref_l = _attn_case(cfg)
    check_out(got_o, ref_o, "bf16", "d1m")
    check_lse(got_l, ref_l, "bf16", "d1m")


def test_empty_selection_rows():
    """Rows whose list is all -1 attend to nothing: out 0, lse -inf."""
    cfg = small_cfg("p32k", seq=512, top_k=3)
    x = make_inputs(cfg, device=DEV)
    shape = _lib.shape_from_config(cfg)
    sel = torch.full((1, 4, shape.n_rows, 3), -1, dtype=torch.int32, device=DEV)
    sel[:, :2, :, 0] = 0                       # heads 0-1 see block 0, heads 2-3 see nothing
    out = torch.full_like(x["q"], 7.0)
    lse = torch.zeros((1, cfg.n_heads_q, cfg.seq), dtype=torch.float32, device=DEV)
    _lib.msa_sparse_prefill(shape, x["q"], x["k"], x["v"], sel, out, lse)
    ref_o, ref_l = oracle.sparse_attention(x["q"], x["k"], x["v"], sel.cpu().numpy(),
                                           cfg.block_size, cfg.q_tile)
    check_out(out, ref_o, "bf16")
    check_lse(lse, ref_l, "bf16")
    assert torch.all(out[:, :, 16:] == 0)


# ------------------------------------------------------------- whole pipeline

def _pipeline(cfg, tiles=None):
    """The three stages chained on the GPU, checked stage by stage:
    * block scores against the oracle's fp64 scores (score tolerance);
    * the selection bit-exactly against the oracle's top-k run on the GPU's own fp32
      scores (the test hands the GPU's scores to the oracle's selection rule; the oracle
      reads nothing else from the GPU);
    * the output and lse of every sampled row against the oracle's attention over the
      GPU's selection.
    The oracle's selection from its own fp64 scores is compared too: where it differs, the
    difference must be a near-tie the score tolerance allows.  Returns the fraction of rows
    where the two selections agree."""
    x = make_inputs(cfg, device=DEV)
    shape = _lib.shape_from_config(cfg)
    qt = cfg.q_tile
    if cfg.mode == "decode":
        bufs = alloc_decode_outputs(shape, DEV, x["q"].dtype)
        run_decode(shape, x["q"], x["k"], x["v"], x["idx_q"], x["idx_k"], bufs)
        rows = [0]
    else:
        bufs = alloc_prefill_outputs(shape, DEV, x["q"].dtype)
        run_prefill(shape, x["q"], x["k"], x["v"], x["idx_q"], x["idx_k"], bufs)
        rows = list(range(shape.n_rows)) if tiles is None else tiles
    _lib.msa_get_device_status()
    # only the sampled rows leave the GPU
    r_idx = torch.tensor(rows, device=DEV)
    tok = np.concatenate([np.arange(m * qt, min(cfg.seq_q, (m + 1) * qt)) for m in rows])
    t_idx = torch.from_numpy(tok).to(DEV)
    g_sc = to_np(bufs["scores"].index_select(2, r_idx))
    g_sel = to_np(bufs["sel"].index_select(2, r_idx))
    g_o = to_np(bufs["out"].index_select(1, t_idx))
    g_l = to_np(bufs["lse"].index_select(2, t_idx))
    if cfg.mode == "decode":
        sc = oracle.index_block_scores_decode(x["idx_q"], x["idx_k"], cfg.block_size)
        own_sel = oracle.block_topk_decode(sc, cfg.seq, cfg.block_size, cfg.top_k)
        sel_on_gpu_scores = oracle.block_topk_decode(g_sc, cfg.seq, cfg.block_size, cfg.top_k)
        ref_o, ref_l = oracle.sparse_attention(x["q"], x["k"], x["v"], g_sel, cfg.block_size,
                                               1, None, cfg.seq - 1)
    else:
        sc = oracle.index_block_scores_prefill(x["idx_q"], x["idx_k"], cfg.block_size, qt,
                                               tiles=rows)
        own_sel = oracle.block_topk_prefill(sc, cfg.seq, qt, cfg.block_size, cfg.top_k, rows)
        sel_on_gpu_scores = oracle.block_topk_prefill(g_sc, cfg.seq, qt, cfg.block_size,
                                                      cfg.top_k, rows)
        full_sel = np.full((cfg.batch, cfg.n_heads_kv, shape.n_rows, cfg.top_k), -1, np.int32)
        full_sel[:, :, rows] = g_sel
        ref_o, ref_l = oracle.sparse_attention(x["q"], x["k"], x["v"], full_sel,
                                               cfg.block_size, qt, None, 0, rows)
    check_scores(g_sc, sc, cfg.name)
    check_selection_exact(g_sel, sel_on_gpu_scores, cfg.name)
    cb = np.broadcast_to(cur_blocks(shape)[rows], g_sel.shape[:-1])
    agree = check_selection_valid(g_sel, own_sel, sc, cb, cfg.name)
    r0 = 0
    for m in rows:                       # each sampled tile on its own
        n = min(cfg.seq_q, (m + 1) * qt) - m * qt
        check_out(g_o[:, r0:r0 + n], ref_o[:, r0:r0 + n], cfg.dtype, f"{cfg.name} tile {m}")
        check_lse(g_l[:, :, r0:r0 + n], ref_l[:, :, r0:r0 + n], cfg.dtype,
                  f"{cfg.name} tile {m}")
        r0 += n
    return agree


def test_pipeline_tiny():
    assert _pipeline(CONFIGS["tiny"]) >= 0.95


def test_pipeline_tiny_scaled_plants_selected():
    cfg = CONFIGS["tiny"]
    x = make_inputs(cfg, device=DEV, input_scale=cfg.head_dim ** -0.5, plant_alpha=3.0)
    shape = _lib.shape_from_config(cfg)
    bufs = alloc_prefill_outputs(shape, DEV, x["q"].dtype)
    run_prefill(shape, x["q"], x["k"], x["v"], x["idx_q"], x["idx_k"], bufs)
    sel = to_np(bufs["sel"])
    for g in range(4):
        for m in range(shape.n_rows):
            cur = cur_blocks(shape)[m]
            for p in x["plants"][0, g]:
                if p < cur:
                    assert p in sel[0, g, m]
    # heads disagree somewhere: selections are per KV head
    assert any(len({tuple(sel[0, g, m]) for g in range(4)}) > 1 for m in range(shape.n_rows))


def test_pipeline_bf16_small():
    assert _pipeline(small_cfg("p32k", seq=3000, n_plants=6)) >= 0.9


def test_pipeline_bf16_batch2():
    assert _pipeline(small_cfg("p32k", batch=2, seq=2000, n_plants=4)) >= 0.9


def test_pipeline_p32k_sampled():
    cfg = CONFIGS["p32k"]
    assert _pipeline(cfg, tiles=sample_tiles(cfg.n_tiles, seed=4)) >= 0.9


def test_pipeline_p128k_sampled():
    cfg = CONFIGS["p128k"]
    assert _pipeline(cfg, tiles=sample_tiles(cfg.n_tiles, seed=5)) >= 0.9


def test_pipeline_p1m_sampled():
    """The 1M-context prefill, run in full on the GPU, checked on sampled tiles."""
    cfg = CONFIGS["p1m"]
    assert _pipeline(cfg, tiles=sample_tiles(cfg.n_tiles, n_random=1, seed=6)) >= 0.9


def test_pipeline_d1m():
    assert _pipeline(CONFIGS["d1m"]) >= 0.9
