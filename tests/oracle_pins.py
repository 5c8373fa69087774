"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each ``pin_*`` takes the oracle module (or a deliberately broken copy of it, see
test_oracle_mutations.py) and raises AssertionError when the module disagrees with

* a library routine (numpy matmul, torch scaled_dot_product_attention in fp64),
* brute force written as plain Python loops on tiny inputs,
* exhaustive enumeration of the top-k subsets,
* closed forms and invariants of the definition (rows sum to one, unselected K/V do
  not matter, k = all blocks is full causal attention, decode = last prefill row),
* a case worked by hand (tests/golden/worked_example_t6.json),
* the planted-block and head-diversity properties of the seeded inputs.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------- index branch

def pin_scores_block1_tile1(o):
    """block = tile = 1: the block scores are the masked index logits (numpy matmul)."""
    r = _rng(1)
    B, T, NI, dI = 2, 9, 4, 5
    q, k = r.standard_normal((B, T, NI, dI)), r.standard_normal((B, T, dI))
    scale = 0.37
    got = o.index_block_scores_prefill(q, k, 1, 1, scale)
    for b in range(B):
        for g in range(NI):
            ref = scale * np.matmul(q[b, :, g, :], k[b].T)           # [T, T]
            ref[np.triu_indices(T, 1)] = -np.inf
            assert np.array_equal(np.isinf(got[b, g]), np.isinf(ref))
            fin = np.isfinite(ref)
            assert np.allclose(got[b, g][fin], ref[fin], rtol=1e-13, atol=1e-13)


def _brute_scores(q, k, bs, qt, scale, positions_of_tile):
    """Plain loops: max over tile rows t, block keys j <= t, of scale * sum_c q*k."""
    B, _, NI, dI = len(q), None, len(q[0][0]), len(q[0][0][0])
    L = len(k[0])
    nB = -(-L // bs)
    out = []
    for b in range(B):
        per_g = []
        for g in range(NI):
            rows = []
            for (rows_t, pos_t) in positions_of_tile:
                row = []
                for blk in range(nB):
                    best = -math.inf
                    for qi, t in zip(rows_t, pos_t):
                        for j in range(blk * bs, min(L, blk * bs + bs)):
                            if j > t:
                                continue
                            s = 0.0
                            for c in range(dI):
                                s += q[b][qi][g][c] * k[b][j][c]
                            best = max(best, scale * s)
                    row.append(best)
                rows.append(row)
            per_g.append(rows)
        out.append(per_g)
    return np.array(out)


def pin_scores_bruteforce(o):
    """Ragged T, block 4, tile 2: the pooled scores equal triple loops."""
    r = _rng(2)
    B, T, NI, dI, bs, qt = 1, 11, 2, 3, 4, 2
    q, k = r.standard_normal((B, T, NI, dI)), r.standard_normal((B, T, dI))
    tiles = [(list(range(m * qt, min(T, m * qt + qt))),) * 2 for m in range(-(-T // qt))]
    ref = _brute_scores(q.tolist(), k.tolist(), bs, qt, 0.5, tiles)
    got = o.index_block_scores_prefill(q, k, bs, qt, 0.5)
    assert got.shape == ref.shape
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    fin = np.isfinite(ref)
    assert np.allclose(got[fin], ref[fin], rtol=1e-12, atol=1e-12)


def pin_decode_scores_bruteforce(o):
    """Decode: one query at position L-1 against the whole cache, ragged last block."""
    r = _rng(3)
    B, L, NI, dI, bs = 2, 13, 4, 3, 4
    q, k = r.standard_normal((B, 1, NI, dI)), r.standard_normal((B, L, dI))
    ref = _brute_scores(q.tolist(), k.tolist(), bs, 1, 0.25, [([0], [L - 1])])
    got = o.index_block_scores_decode(q, k, bs, 0.25)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def _pooled_matmul(q, k, scale, bs, qt, q_pos):
    """Block scores from one dense numpy product: s = scale * q k^T for every (query, key),
    -inf where key > query position, padded with -inf to whole tiles and blocks, then the
    max over each (tile, block) rectangle.  q [B, n, NI, dI] at positions q_pos[n]; k
    [B, L, dI].  Returns [B, NI, ceil(n/qt), ceil(L/bs)]."""
    B, n, NI, _ = q.shape
    L = k.shape[1]
    s = scale * np.einsum("bngc,bjc->bgnj", q, k)
    s = np.where(np.arange(L)[None, None, None, :] <= np.asarray(q_pos)[None, None, :, None],
                 s, -np.inf)
    nT, nB = -(-n // qt), -(-L // bs)
    full = np.full((B, NI, nT * qt, nB * bs), -np.inf)
    full[:, :, :n, :L] = s
    return full.reshape(B, NI, nT, qt, nB, bs).max(axis=(3, 5))


def _check_scores_equal(got, ref):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    fin = np.isfinite(ref)
    assert np.allclose(got[fin], ref[fin], rtol=1e-12, atol=1e-12)


def pin_scores_many_blocks(o):
    """The oracle scores long key ranges a chunk of whole blocks at a time.  Prefill and
    decode with more blocks than one chunk holds (several hundred), ragged last tile and
    block, equal one dense masked product pooled by reshaping; so do small cases with the
    chunk forced to 1 and 3 blocks, where every chunk boundary cuts a tile's key range."""
    r = _rng(51)
    q, k = r.standard_normal((1, 601, 2, 3)), r.standard_normal((1, 601, 3))
    _check_scores_equal(o.index_block_scores_prefill(q, k, 2, 2, 0.3),
                        _pooled_matmul(q, k, 0.3, 2, 2, np.arange(601)))
    qd, kd = r.standard_normal((2, 1, 2, 3)), r.standard_normal((2, 701, 3))
    _check_scores_equal(o.index_block_scores_decode(qd, kd, 2, 0.3)[:, :, 0],
                        _pooled_matmul(qd, kd, 0.3, 2, 1, [700])[:, :, 0])
    saved = o._BLOCKS_PER_CHUNK
    try:
        for chunk in (1, 3):
            o._BLOCKS_PER_CHUNK = chunk
            q, k = r.standard_normal((2, 37, 3, 4)), r.standard_normal((2, 37, 4))
            _check_scores_equal(o.index_block_scores_prefill(q, k, 4, 2, 0.7),
                                _pooled_matmul(q, k, 0.7, 4, 2, np.arange(37)))
            qd, kd = r.standard_normal((1, 1, 3, 4)), r.standard_normal((1, 23, 4))
            _check_scores_equal(o.index_block_scores_decode(qd, kd, 4, 0.7)[:, :, 0],
                                _pooled_matmul(qd, kd, 0.7, 4, 1, [22])[:, :, 0])
    finally:
        o._BLOCKS_PER_CHUNK = saved


def pin_sampled_forward_equals_full(o):
    """The oracle's sampled evaluation (a list of query tiles) of the scores, the selection,
    the attention and the whole prefill returns exactly the full evaluation's values on
    those tiles, whatever order the tiles are listed in."""
    r = _rng(52)
    B, T, Hq, Hkv, d, dI, bs, qt, kk = 2, 45, 4, 2, 3, 5, 8, 4, 3
    q, k, v = (r.standard_normal((B, T, Hq, d)), r.standard_normal((B, Hkv, T, d)),
               r.standard_normal((B, Hkv, T, d)))
    iq, ik = r.standard_normal((B, T, Hkv, dI)), r.standard_normal((B, T, dI))
    tiles = [9, 0, 4, 11]
    rows = np.concatenate([np.arange(m * qt, min(T, (m + 1) * qt)) for m in tiles])
    sc_f, sel_f, out_f, lse_f = o.msa_prefill(q, k, v, iq, ik, bs, qt, kk)
    sc_s, sel_s, out_s, lse_s = o.msa_prefill(q, k, v, iq, ik, bs, qt, kk, tiles=tiles)
    assert np.array_equal(sc_s, sc_f[:, :, tiles])
    assert np.array_equal(sel_s, sel_f[:, :, tiles])
    assert np.array_equal(out_s, out_f[:, rows]) and np.array_equal(lse_s, lse_f[:, :, rows])
    assert np.array_equal(o.index_block_scores_prefill(iq, ik, bs, qt, None, tiles),
                          sc_f[:, :, tiles])
    assert np.array_equal(o.block_topk_prefill(sc_f[:, :, tiles], T, qt, bs, kk, tiles),
                          sel_f[:, :, tiles])
    out_a, lse_a = o.sparse_attention(q, k, v, sel_f, bs, qt, None, 0, tiles)
    assert np.array_equal(out_a, out_f[:, rows]) and np.array_equal(lse_a, lse_f[:, :, rows])


def pin_shared_selection_f32_sum(o):
    """The aggregated selection of the ablation: per (sequence, row), the KV heads' scores
    summed in float32 in head order, then the usual rule.  Checked against a loop that adds
    numpy float32 scalars and ranks with Python's sorted(); one row is built so that the
    float32 sum and the exact sum rank two blocks the other way round, and one so that a
    max over the heads would choose differently from their sum."""
    r = _rng(53)
    B, NI, T, qt, bs, kk = 2, 4, 40, 4, 4, 2
    nT, nB = T // qt, T // bs
    sc = r.integers(-4, 5, size=(B, NI, nT, nB)).astype(np.float64)
    # row (0, 9): cur = 9; block 2 sums to 1e8 in float32 (1e8 + 6 exactly), block 5 to
    # 1e8 + 8 in float32 (1e8 + 5 exactly); the others are far lower; one block besides
    # the current one is kept
    sc[0, :, 9, :] = -50.0
    sc[0, :, 9, 2] = [1e8, 3.0, 3.0, 0.0]
    sc[0, :, 9, 5] = [1e8, 5.0, 0.0, 0.0]
    # row (1, 7): cur = 7; block 1 has the larger maximum, block 3 the larger sum
    sc[1, :, 7, :] = -50.0
    sc[1, :, 7, 1] = [9.0, 0.0, 0.0, 0.0]
    sc[1, :, 7, 3] = [3.0, 3.0, 3.0, 3.0]
    got = o.block_topk_shared_prefill(sc, T, qt, bs, kk)
    for b in range(B):
        for m in range(nT):
            agg = []
            for blk in range(nB):
                acc = np.float32(sc[b, 0, m, blk])
                for g in range(1, NI):
                    acc = np.float32(acc + np.float32(sc[b, g, m, blk]))
                agg.append(float(acc))
            cur = (m * qt + qt - 1) // bs
            best = [blk for _, blk in sorted((-agg[blk], blk) for blk in range(cur))][:kk - 1]
            want = sorted(best + [cur])
            want += [-1] * (kk - len(want))
            for g in range(NI):
                assert list(got[b, g, m]) == want, (b, g, m, got[b, g, m], want)
    assert list(got[0, 0, 9]) == [5, 9] and list(got[1, 0, 7]) == [3, 7]


# ----------------------------------------------------------------------- top-k

def _dominates(scores, chosen, cur):
    """Every chosen non-current block beats every unchosen candidate (desc score, asc idx)."""
    others = [b for b in range(cur) if b not in chosen]
    for a in chosen:
        if a == cur:
            continue
        for b in others:
            if not (scores[a] > scores[b] or (scores[a] == scores[b] and a < b)):
                return False
    return True


def pin_topk_bruteforce(o):
    """Enumerate every k-subset holding the current block: exactly one dominates."""
    r = _rng(4)
    for trial in range(300):
        cur = int(r.integers(0, 11))
        top_k = int(r.integers(1, 5))
        # small integers make ties common; signed zeros must tie with each other
        vals = r.integers(-2, 3, size=cur + 1).astype(np.float64)
        zeros = vals == 0
        vals[zeros] = np.where(r.random(zeros.sum()) < 0.5, 0.0, -0.0)
        if trial % 7 == 0:
            vals = r.standard_normal(cur + 1)
        row = np.concatenate([vals, np.full(3, -np.inf)])
        got = o.select_blocks(row, cur, top_k)
        want_n = min(top_k, cur + 1)
        winners = []
        for sub in itertools.combinations(range(cur), want_n - 1):
            chosen = sorted(set(sub) | {cur})
            if _dominates(list(vals), chosen, cur):
                winners.append(chosen)
        assert len(winners) == 1, (vals, top_k, winners)
        expect = np.full(top_k, -1)
        expect[:want_n] = winners[0]
        assert np.array_equal(got, expect), (vals, cur, top_k, got, expect)


def pin_topk_layout(o):
    """Prefill/decode wrappers: the current block comes from the tile's last query."""
    T, qt, bs, k = 21, 4, 8, 3
    nT, nB = -(-T // qt), -(-T // bs)
    scores = np.arange(nB, dtype=np.float64)[None, None, None, :].repeat(nT, axis=2)
    sel = o.block_topk_prefill(scores, T, qt, bs, k)
    for m in range(nT):
        last = min(T - 1, m * qt + qt - 1)
        cur = last // bs
        want = sorted(set(range(max(0, cur - (k - 1)), cur)) | {cur})   # increasing scores
        expect = np.full(k, -1)
        expect[:len(want)] = want
        assert np.array_equal(sel[0, 0, m], expect), (m, sel[0, 0, m], expect)
    dsel = o.block_topk_decode(scores[:, :, :1], T, bs, k)
    assert np.array_equal(dsel[0, 0, 0], [0, 1, 2])                     # cur = 20 // 8 = 2
    # a query that opens a block: position 16 with block 8 has current block 2
    dsel = o.block_topk_decode(scores[:, :, :1], 17, bs, 2)
    assert np.array_equal(dsel[0, 0, 0], [1, 2]), dsel[0, 0, 0]
    psel = o.block_topk_prefill(np.zeros((1, 1, 17, 3)), 17, 1, bs, 1)
    assert [int(psel[0, 0, t, 0]) for t in (7, 8, 15, 16)] == [0, 1, 1, 2]


# ------------------------------------------------------------------- attention

def _brute_attention(q, k, v, sel, bs, qt, scale, q_offset):
    """Plain loops over (b, t, h): softmax over selected, causally visible keys."""
    B, Sq, Hq, d = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Sq, Hq, d))
    lse = np.full((B, Hq, Sq), -np.inf)
    for b in range(B):
        for t in range(Sq):
            pos = q_offset + t
            for h in range(Hq):
                g = h // G
                keys = []
                for blk in sel[b, g, t // qt]:
                    if blk < 0:
                        continue
                    for j in range(blk * bs, min(Sk, blk * bs + bs)):
                        if j <= pos:
                            keys.append(j)
                if not keys:
                    continue
                z = [scale * sum(q[b, t, h, c] * k[b, g, j, c] for c in range(d)) for j in keys]
                zm = max(z)
                w = [math.exp(x - zm) for x in z]
                s = sum(w)
                lse[b, h, t] = zm + math.log(s)
                for c in range(d):
                    out[b, t, h, c] = sum(wi * v[b, g, j, c] for wi, j in zip(w, keys)) / s
    return out, lse


def _small_attn_case(seed, B=1, T=10, Hq=4, Hkv=2, d=3):
    r = _rng(seed)
    return (r.standard_normal((B, T, Hq, d)), r.standard_normal((B, Hkv, T, d)),
            r.standard_normal((B, Hkv, T, d)))


def pin_full_k_bruteforce(o):
    """k >= number of blocks: MSA is full causal GQA attention (plain loops)."""
    q, k, v = _small_attn_case(5)
    T, bs, qt = 10, 4, 2
    nT, nB = -(-T // qt), -(-T // bs)
    sel = o.block_topk_prefill(np.zeros((1, 2, nT, nB)), T, qt, bs, nB + 1)
    out, lse = o.sparse_attention(q, k, v, sel, bs, qt, 0.7)
    ref_o, ref_l = _brute_attention(q, k, v, sel, bs, qt, 0.7, 0)
    assert np.allclose(out, ref_o, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, ref_l, rtol=1e-12, atol=1e-12)
    fo, fl = o.full_causal_gqa(q, k, v, 0.7)
    assert np.allclose(fo, ref_o, rtol=1e-12, atol=1e-12)
    assert np.allclose(fl, ref_l, rtol=1e-12, atol=1e-12)


def pin_full_k_sdpa(o):
    """k = all blocks against torch's scaled_dot_product_attention in float64."""
    import torch
    r = _rng(6)
    B, T, Hq, Hkv, d, bs, qt = 2, 70, 8, 4, 16, 16, 8
    q = r.standard_normal((B, T, Hq, d))
    k = r.standard_normal((B, Hkv, T, d))
    v = r.standard_normal((B, Hkv, T, d))
    nT, nB = -(-T // qt), -(-T // bs)
    sel = o.block_topk_prefill(r.standard_normal((B, Hkv, nT, nB)), T, qt, bs, nB)
    out, lse = o.sparse_attention(q, k, v, sel, bs, qt, None)
    tq = torch.from_numpy(q).permute(0, 2, 1, 3)
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq, torch.from_numpy(k), torch.from_numpy(v), is_causal=True, enable_gqa=True)
    assert np.allclose(out, ref.permute(0, 2, 1, 3).numpy(), rtol=1e-10, atol=1e-10)
    kk = torch.from_numpy(k).repeat_interleave(Hq // Hkv, dim=1)
    z = (tq @ kk.transpose(-1, -2)) / math.sqrt(d)
    z = z.masked_fill(torch.triu(torch.ones(T, T, dtype=torch.bool), 1), -math.inf)
    assert np.allclose(lse, torch.logsumexp(z, dim=-1).numpy(), rtol=1e-10, atol=1e-10)


def _random_sel(o, T, qt, bs, k, Hkv, seed, B=1):
    r = _rng(seed)
    nT, nB = -(-T // qt), -(-T // bs)
    return o.block_topk_prefill(r.standard_normal((B, Hkv, nT, nB)), T, qt, bs, k)


def pin_sparse_bruteforce(o):
    """A sparse selection: output and lse equal the plain-loop restatement."""
    q, k, v = _small_attn_case(7, B=2, T=23, Hq=6, Hkv=3, d=4)
    T, bs, qt, kk = 23, 4, 2, 3
    sel = _random_sel(o, T, qt, bs, kk, 3, 8, B=2)
    out, lse = o.sparse_attention(q, k, v, sel, bs, qt, 0.6)
    ref_o, ref_l = _brute_attention(q, k, v, sel, bs, qt, 0.6, 0)
    assert np.allclose(out, ref_o, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, ref_l, rtol=1e-12, atol=1e-12)


def pin_rows_sum_to_one(o):
    """With V = 1 every output is 1 (the weights sum to one), for any selection."""
    q, k, _ = _small_attn_case(9, T=40, Hq=4, Hkv=2, d=5)
    v = np.ones_like(k)
    sel = _random_sel(o, 40, 4, 8, 2, 2, 10)
    out, lse = o.sparse_attention(q, k, v, sel, 8, 4, None)
    assert np.allclose(out, 1.0, rtol=0, atol=1e-13)
    assert np.all(np.isfinite(lse))


def pin_unselected_invariance(o):
    """Changing K/V inside blocks no tile selects leaves the output unchanged."""
    q, k, v = _small_attn_case(11, T=48, Hq=4, Hkv=2, d=4)
    T, bs, qt = 48, 8, 4
    nT, nB = T // qt, T // bs
    sel = np.full((1, 2, nT, 2), -1, dtype=np.int32)
    for m in range(nT):
        cur = (m * qt + qt - 1) // bs
        sel[0, :, m, 0] = 0 if cur > 0 else -1
        sel[0, :, m, 1] = cur
        if cur == 0:
            sel[0, :, m] = [0, -1]
    out1, lse1 = o.sparse_attention(q, k, v, sel, bs, qt, None)
    k2, v2 = k.copy(), v.copy()
    # blocks 1..nB-1 are only ever used as the current block, so block 1's keys are
    # unseen by tiles of blocks 2+; change them where only those tiles could look
    r = _rng(12)
    for g in range(2):
        for j in range(bs, 2 * bs):
            k2[0, g, j] = r.standard_normal(4) * 5
            v2[0, g, j] = r.standard_normal(4) * 5
    out2, lse2 = o.sparse_attention(q, k2, v2, sel, bs, qt, None)
    rows = np.arange(2 * bs, T)              # queries whose tiles do not select block 1
    assert np.allclose(out1[0, rows], out2[0, rows], rtol=0, atol=0)
    assert np.allclose(lse1[0][:, rows], lse2[0][:, rows], rtol=0, atol=0)
    changed = np.arange(bs, 2 * bs)          # queries inside block 1 must see the change
    assert not np.allclose(out1[0, changed], out2[0, changed])


def pin_decode_equals_prefill_row(o):
    """Decode at cache length L = the prefill row t = L-1 with q_tile = 1."""
    r = _rng(13)
    B, L, Hq, Hkv, d, dI, bs, kk = 1, 37, 8, 4, 6, 5, 8, 3
    q = r.standard_normal((B, L, Hq, d))
    k = r.standard_normal((B, Hkv, L, d))
    v = r.standard_normal((B, Hkv, L, d))
    iq = r.standard_normal((B, L, Hkv, dI))
    ik = r.standard_normal((B, L, dI))
    sc_p, sel_p, out_p, lse_p = o.msa_prefill(q, k, v, iq, ik, bs, 1, kk)
    sc_d, sel_d, out_d, lse_d = o.msa_decode(q[:, L - 1:], k, v, iq[:, L - 1:], ik, bs, kk)
    assert np.array_equal(sc_d[:, :, 0], sc_p[:, :, L - 1])
    assert np.array_equal(sel_d[:, :, 0], sel_p[:, :, L - 1])
    assert np.allclose(out_d[:, 0], out_p[:, L - 1], rtol=1e-13, atol=1e-13)
    assert np.allclose(lse_d[:, :, 0], lse_p[:, :, L - 1], rtol=1e-13, atol=1e-13)


# ------------------------------------------------------ seeded-input properties

def _tiny_scaled_inputs():
    from block_sparse_gqa_02_gb300.configs import CONFIGS
    from block_sparse_gqa_02_gb300.inputs import make_inputs
    cfg = CONFIGS["tiny"]
    return cfg, make_inputs(cfg, input_scale=cfg.head_dim ** -0.5, plant_alpha=3.0)


def pin_planted_selected(o):
    """Scaled tiny inputs: every planted block before a tile's current block is chosen."""
    cfg, x = _tiny_scaled_inputs()
    sc = o.index_block_scores_prefill(x["idx_q"], x["idx_k"], cfg.block_size, cfg.q_tile)
    sel = o.block_topk_prefill(sc, cfg.seq, cfg.q_tile, cfg.block_size, cfg.top_k)
    hits = 0
    for g in range(cfg.n_heads_kv):
        for m in range(cfg.n_tiles):
            cur = (m * cfg.q_tile + cfg.q_tile - 1) // cfg.block_size
            before = [int(p) for p in x["plants"][0, g] if p < cur]
            for p in before:
                assert p in sel[0, g, m], (g, m, p, sel[0, g, m])
                hits += 1
    assert hits > 0


def pin_head_diversity(o):
    """Different KV heads select different blocks (an aggregated selection would not)."""
    cfg, x = _tiny_scaled_inputs()
    sc = o.index_block_scores_prefill(x["idx_q"], x["idx_k"], cfg.block_size, cfg.q_tile)
    sel = o.block_topk_prefill(sc, cfg.seq, cfg.q_tile, cfg.block_size, cfg.top_k)
    differing = 0
    for m in range(cfg.n_tiles):
        rows = {tuple(sel[0, g, m]) for g in range(cfg.n_heads_kv)}
        differing += len(rows) > 1
    assert differing >= cfg.n_tiles // 2, differing


# --------------------------------------------------------------- worked example

def _val(x):
    if isinstance(x, (int, float)):
        return float(x)
    if x == "-inf":
        return -math.inf
    if x.startswith("ln"):
        return math.log(float(x[2:]))
    if "/" in x:
        a, b = x.split("/")
        return float(a) / float(b)
    return float(x)


def pin_worked_example(o):
    """The hand-worked T=6 case (tests/golden/worked_example_t6.json)."""
    with open(os.path.join(GOLDEN, "worked_example_t6.json")) as f:
        case = json.load(f)
    inp, exp = case["inputs"], case["expected"]
    sh = case["shape"]
    T = sh["T"]
    vec = lambda key: np.array([_val(x) for x in inp[key]])
    idx_q = np.stack([vec("idx_q_head0"), vec("idx_q_head1")], axis=1)[None, :, :, None]
    idx_k = vec("idx_k")[None, :, None]
    q = np.stack([vec("q_head0"), vec("q_head1")], axis=1)[None, :, :, None]
    k = np.stack([vec("k_head0"), vec("k_head1")], axis=0)[None, :, :, None]
    v = np.stack([vec("v_head0"), vec("v_head1")], axis=0)[None, :, :, None]
    sc, sel, out, lse = o.msa_prefill(q, k, v, idx_q, idx_k, sh["block_size"], sh["q_tile"],
                                      sh["top_k"], sh["sm_scale"], sh["index_scale"])
    for g in range(2):
        want_sc = np.array([[_val(x) for x in row] for row in exp[f"scores_head{g}"]])
        assert np.array_equal(np.isinf(sc[0, g]), np.isinf(want_sc))
        assert np.allclose(sc[0, g][np.isfinite(want_sc)], want_sc[np.isfinite(want_sc)],
                           atol=1e-15)
        assert np.array_equal(sel[0, g], np.array(exp[f"sel_head{g}"])), (g, sel[0, g])
        want_o = np.array([_val(x) for x in exp[f"out_head{g}"]])
        want_l = np.array([_val(x) for x in exp[f"lse_head{g}"]])
        assert np.allclose(out[0, :, g, 0], want_o, rtol=1e-13, atol=1e-13), out[0, :, g, 0]
        assert np.allclose(lse[0, g], want_l, rtol=1e-13, atol=1e-13), lse[0, g]
    assert out.shape == (1, T, 2, 1)


def pin_paged_equals_contiguous(o):
    """A paged cache is storage only: scattering each sequence's blocks into a pool in a
    shuffled order and decoding through the block table equals the contiguous decode of the
    same sequence truncated to its length."""
    r = _rng(21)
    bs, nb_max, Hq, Hkv, d, dI, kk = 4, 6, 4, 2, 3, 5, 2
    lens = [1, 4, 5, 13, 24]
    B = len(lens)
    full_k = r.standard_normal((B, Hkv, nb_max * bs, d))
    full_v = r.standard_normal((B, Hkv, nb_max * bs, d))
    full_ik = r.standard_normal((B, nb_max * bs, dI))
    q = r.standard_normal((B, 1, Hq, d))
    iq = r.standard_normal((B, 1, Hkv, dI))
    nbs = [-(-L // bs) for L in lens]
    P = sum(nbs) + 2
    perm = r.permutation(P)
    table = np.full((B, nb_max), -1)
    k_pool = r.standard_normal((P, Hkv, bs, d))
    v_pool = r.standard_normal((P, Hkv, bs, d))
    ik_pool = r.standard_normal((P, bs, dI))
    off = 0
    for b, nb in enumerate(nbs):
        for j in range(nb):
            ph = perm[off + j]
            table[b, j] = ph
            k_pool[ph] = full_k[b, :, j * bs:(j + 1) * bs]
            v_pool[ph] = full_v[b, :, j * bs:(j + 1) * bs]
            ik_pool[ph] = full_ik[b, j * bs:(j + 1) * bs]
        off += nb
    sc, sel, out, lse = o.msa_decode_paged(q, k_pool, v_pool, iq, ik_pool, lens, table, bs, kk,
                                           nb_max)
    for b, L in enumerate(lens):
        sc1, sel1, out1, lse1 = o.msa_decode(q[b:b + 1], full_k[b:b + 1, :, :L],
                                             full_v[b:b + 1, :, :L], iq[b:b + 1],
                                             full_ik[b:b + 1, :L], bs, kk)
        nb = nbs[b]
        assert np.array_equal(sc[b, :, :, :nb], sc1[0]) and np.all(np.isneginf(sc[b, :, :, nb:]))
        assert np.array_equal(sel[b], sel1[0])
        assert np.allclose(out[b], out1[0], rtol=1e-13, atol=1e-13)
        assert np.allclose(lse[b], lse1[0], rtol=1e-13, atol=1e-13)


def pin_backward_finite_differences(o):
    """Sparse-attention gradients against central finite differences of sum(dout * out)."""
    r = _rng(31)
    B, T, Hq, Hkv, d, bs, qt, kk = 1, 12, 4, 2, 3, 4, 2, 2
    q, k, v = (r.standard_normal((B, T, Hq, d)), r.standard_normal((B, Hkv, T, d)),
               r.standard_normal((B, Hkv, T, d)))
    dout = r.standard_normal((B, T, Hq, d))
    sel = _random_sel(o, T, qt, bs, kk, Hkv, 32)
    dq, dk, dv = o.sparse_attention_backward(q, k, v, sel, dout, bs, qt, 0.8)

    def loss(q_, k_, v_):
        out, _ = o.sparse_attention(q_, k_, v_, sel, bs, qt, 0.8)
        return float((dout * out).sum())
    h = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(12):
            idx = tuple(int(r.integers(0, n)) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": (q, k, v), "k": (q, k, v), "v": (q, k, v)}[name]
            fp = loss(*[xp if a is x else a for a in args])
            fm = loss(*[xm if a is x else a for a in args])
            num = (fp - fm) / (2 * h)
            assert abs(num - grad[idx]) <= 1e-6 * max(1.0, abs(num)), (name, idx, num, grad[idx])


def pin_backward_full_k_autograd(o):
    """k = all blocks: the gradients equal torch autograd of causal GQA SDPA in float64."""
    import torch
    r = _rng(33)
    B, T, Hq, Hkv, d, bs, qt = 1, 40, 8, 2, 8, 8, 4
    q = r.standard_normal((B, T, Hq, d))
    k = r.standard_normal((B, Hkv, T, d))
    v = r.standard_normal((B, Hkv, T, d))
    dout = r.standard_normal((B, T, Hq, d))
    nT, nB = T // qt, T // bs
    sel = o.block_topk_prefill(r.standard_normal((B, Hkv, nT, nB)), T, qt, bs, nB)
    dq, dk, dv = o.sparse_attention_backward(q, k, v, sel, dout, bs, qt, None)
    tq = torch.from_numpy(q).permute(0, 2, 1, 3).requires_grad_()
    tk = torch.from_numpy(k).requires_grad_()
    tv = torch.from_numpy(v).requires_grad_()
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True,
                                                           enable_gqa=True)
    out.backward(torch.from_numpy(dout).permute(0, 2, 1, 3))
    assert np.allclose(dq, tq.grad.permute(0, 2, 1, 3).numpy(), rtol=1e-9, atol=1e-10)
    assert np.allclose(dk, tk.grad.numpy(), rtol=1e-9, atol=1e-10)
    assert np.allclose(dv, tv.grad.numpy(), rtol=1e-9, atol=1e-10)


def pin_index_kl(o):
    """KL of the index branch: zero with zero gradient when the index branch is the main
    branch (G = 1, same queries, keys and scale); positive otherwise, with gradients equal
    to central finite differences."""
    r = _rng(41)
    B, T, Hkv, d, bs, qt, kk = 1, 16, 2, 4, 4, 2, 3
    q = r.standard_normal((B, T, Hkv, d))                 # G = 1
    k = r.standard_normal((B, Hkv, T, d))
    sel = _random_sel(o, T, qt, bs, kk, Hkv, 42)
    # index keys are shared by the KV heads: use one KV head's keys for both heads' test
    k_shared = np.repeat(k[:, :1], Hkv, axis=1)
    loss0, gq0, gk0 = o.index_kl_loss(q, k_shared, q, k_shared[:, 0], sel, bs, qt, 0.5, 0.5)
    assert abs(loss0) < 1e-12 and np.abs(gq0).max() < 1e-12 and np.abs(gk0).max() < 1e-12
    iq = r.standard_normal((B, T, Hkv, 3))
    ik = r.standard_normal((B, T, 3))
    loss, gq, gk = o.index_kl_loss(q, k, iq, ik, sel, bs, qt, 0.5, 0.7)
    assert loss > 0
    h = 1e-6
    for name, x, grad in (("iq", iq, gq), ("ik", ik, gk)):
        for _ in range(10):
            idx = tuple(int(r.integers(0, n)) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            if name == "iq":
                fp = o.index_kl_loss(q, k, xp, ik, sel, bs, qt, 0.5, 0.7)[0]
                fm = o.index_kl_loss(q, k, xm, ik, sel, bs, qt, 0.5, 0.7)[0]
            else:
                fp = o.index_kl_loss(q, k, iq, xp, sel, bs, qt, 0.5, 0.7)[0]
                fm = o.index_kl_loss(q, k, iq, xm, sel, bs, qt, 0.5, 0.7)[0]
            num = (fp - fm) / (2 * h)
            assert abs(num - grad[idx]) <= 1e-6 * max(1.0, abs(num)), (name, idx, num, grad[idx])


def pin_index_kl_group_mean(o):
    """KL with G = 2 query heads per KV head against a plain-loop restatement: per (token,
    KV head), each head's softmax over the visible selected keys, their mean as the target,
    the index softmax, and scipy's relative entropy of the two."""
    from scipy.special import softmax
    from scipy.stats import entropy
    r = _rng(43)
    B, T, Hkv, G, d, dI, bs, qt, kk = 1, 14, 2, 2, 3, 2, 3, 2, 2
    q = r.standard_normal((B, T, Hkv * G, d))
    k = r.standard_normal((B, Hkv, T, d))
    iq = r.standard_normal((B, T, Hkv, dI))
    ik = r.standard_normal((B, T, dI))
    sel = _random_sel(o, T, qt, bs, kk, Hkv, 44)
    loss = o.index_kl_loss(q, k, iq, ik, sel, bs, qt, 0.9, 0.6)[0]
    ref = 0.0
    for t in range(T):
        for g in range(Hkv):
            J = [j for blk in sel[0, g, t // qt] if blk >= 0
                 for j in range(blk * bs, min(T, (blk + 1) * bs)) if j <= t]
            heads = [softmax([0.9 * sum(q[0, t, g * G + hh, c] * k[0, g, j, c] for c in range(d))
                              for j in J]) for hh in range(G)]
            target = [sum(hp[i] for hp in heads) / G for i in range(len(J))]
            index = softmax([0.6 * sum(iq[0, t, g, c] * ik[0, j, c] for c in range(dI))
                             for j in J])
            ref += entropy(target, index)
    assert abs(loss - ref) <= 1e-10 * max(1.0, abs(ref)), (loss, ref)


ALL_PINS = [
    pin_scores_block1_tile1, pin_scores_bruteforce, pin_decode_scores_bruteforce,
    pin_scores_many_blocks, pin_sampled_forward_equals_full, pin_shared_selection_f32_sum,
    pin_topk_bruteforce, pin_topk_layout, pin_full_k_bruteforce, pin_full_k_sdpa,
    pin_sparse_bruteforce, pin_rows_sum_to_one, pin_unselected_invariance,
    pin_decode_equals_prefill_row, pin_planted_selected, pin_head_diversity,
    pin_worked_example, pin_paged_equals_contiguous, pin_backward_finite_differences,
    pin_backward_full_k_autograd, pin_index_kl, pin_index_kl_group_mean,
]
