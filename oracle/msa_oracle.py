"""Plain fp64 CPU oracle for MiniMax Sparse Attention (MSA).

TEST INFRASTRUCTURE ONLY.  This module is the independent reference the CUDA
library is checked against.  Only the test suite, the package smoke check and the
benchmark's CPU-baseline leg may import it; the library itself never does, and this
module imports nothing from the library.

What it follows (cited by page title and section):

* "Sparse Attention Cannot Be Directly Ported Across Architectures" (disconfirmai.com
  news article), paragraph introducing MSA: a lightweight index branch runs full
  attention with four query heads and one key head; the main branch attends only to
  the blocks the index selects.  Paragraph "MSA addresses these issues": the index
  outputs are not aggregated, each KV head selects its own set, and retrieval is per
  block rather than per token.
* "How MiniMax M3 was built" (aietalks.com), sections "MSA uses a lightweight index
  branch before sparse attention" and "Block-level retrieval makes sparse attention
  easier to run on GPUs" -- the same two branches and the per-head block retrieval.
* The Chinese topic page on MSA (disconfirmai.com), summary paragraph: each KV head
  independently selects its top-k key/value blocks and the main branch computes exact
  attention only on the selected blocks.

The pages fix no block size, k, pooling rule, scale or tie-break.  The readings
taken here are: index logits scaled by index_scale (1/sqrt(dI) by default) and
pooled raw (no softmax / ReLU / head weights); a block's score for a query tile is
the MAX over the tile's queries and the block's keys of the causally visible logits;
k counts the current block, which is always kept; the other k-1 blocks are the
highest scores, ties to the lower block index, compared as reals (-0 == +0); the
result is written ascending and padded with -1; fewer than k visible blocks means
all of them are taken.  Attention is exact softmax over the union of the selected
blocks intersected with the causal range, with all G query heads of a KV group
sharing their group's selection (head h uses KV head h // G).

Everything is computed in float64.  Inputs stored as bf16 or fp32 are exactly
representable in float64, so the oracle sees the very values the kernels see.
"""
from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    """Any array-like (numpy or torch, any float dtype) as a float64 numpy array."""
    if hasattr(x, "detach"):                      # torch tensor: go through fp32
        x = x.detach().to("cpu").float().numpy()
    return np.asarray(x, dtype=np.float64)


def _rows(x, *index) -> np.ndarray:
    """x[index] as a float64 numpy array; x is a numpy array or a torch tensor on any
    device.  Only the requested slice is converted, so large caches never are."""
    if hasattr(x, "detach"):
        import torch
        idx = tuple(torch.as_tensor(i, device=x.device) if isinstance(i, np.ndarray) else i
                    for i in index)
        return x[idx].detach().to("cpu").double().numpy()
    return np.asarray(np.asarray(x)[index], dtype=np.float64)


# Index keys are scored this many blocks at a time (the scores are defined per block).
_BLOCKS_PER_CHUNK = 256


def default_scale(dim: int) -> float:
    """Softmax scale used when a caller passes 0: 1/sqrt(dim)."""
    return 1.0 / np.sqrt(dim)


# ---------------------------------------------------------------------------
# Index branch: causal index logits, max-pooled per (query tile, key block)
# ---------------------------------------------------------------------------

def index_logits(idx_q_rows, idx_k, index_scale, q_pos, key_pos0=0):
    """Causal index logits for a set of query tokens.

    idx_q_rows [n, NI, dI] are the index queries of n tokens at positions q_pos[n];
    idx_k [L, dI] holds the single shared index key head at positions key_pos0 ..
    key_pos0 + L - 1.  Returns s [NI, n, L] with s[g, i, j] = index_scale *
    <idx_q_rows[i, g], idx_k[j]> where key j is visible (position <= q_pos[i]) and -inf
    elsewhere (four index query heads against one key head: the MSA paragraph of the
    disconfirmai.com article).
    """
    qr = _f64(idx_q_rows)
    kk = _f64(idx_k)
    s = index_scale * np.matmul(qr.transpose(1, 0, 2), kk.T)          # [NI, n, L]
    j = key_pos0 + np.arange(kk.shape[0])
    visible = j[None, :] <= np.asarray(q_pos)[:, None]          # [n, L]
    return np.where(visible[None, :, :], s, -np.inf)


def pool_blocks(s, block_size):
    """Max of s [NI, n, L] over all n query rows and over each key block of block_size.

    Returns [NI, nB]; a block with no visible key gives -inf.  Block-level retrieval:
    "Block-level retrieval makes sparse attention easier to run on GPUs" (aietalks.com).
    """
    NI, n, L = s.shape
    nB = -(-L // block_size)
    pad = nB * block_size - L
    if pad:
        s = np.concatenate([s, np.full((NI, n, pad), -np.inf)], axis=2)
    return s.reshape(NI, n, nB, block_size).max(axis=(1, 3))


def _pooled_row(q_rows, idx_k_b, index_scale, q_pos, block_size, n_blocks):
    """Block scores [NI, n_blocks] of a group of query tokens against one sequence's keys.

    Blocks that hold no key visible to any of the tokens score -inf; the others are
    pooled chunk by chunk of whole blocks.
    """
    NI = q_rows.shape[1]
    out = np.full((NI, n_blocks), -np.inf)
    n_visible = int(np.max(q_pos)) + 1                  # keys 0 .. max position
    vis_blocks = -(-n_visible // block_size)
    for c0 in range(0, vis_blocks, _BLOCKS_PER_CHUNK):
        c1 = min(vis_blocks, c0 + _BLOCKS_PER_CHUNK)
        j0, j1 = c0 * block_size, min(n_visible, c1 * block_size)
        s = index_logits(q_rows, _rows(idx_k_b, slice(j0, j1)), index_scale, q_pos, j0)
        out[:, c0:c1] = pool_blocks(s, block_size)
    return out


def index_block_scores_prefill(idx_q, idx_k, block_size, q_tile, index_scale=None,
                               tiles=None):
    """Prefill block scores S[b, g, m, blk] for query tiles m of q_tile tokens.

    idx_q [B, T, NI, dI], idx_k [B, T, dI].  Tile m holds tokens m*q_tile .. (m+1)*q_tile-1
    (the last tile may be short).  S is the max, over the tile's tokens t and the block's
    keys j <= t, of the scaled index logit; -inf when no key of the block is visible.
    ``tiles`` restricts the result to a list of tile indices (axis 2 follows that list).
    """
    B, T, NI, dI = idx_q.shape
    if index_scale is None or index_scale == 0:
        index_scale = default_scale(dI)
    nT = -(-T // q_tile)
    tile_list = list(range(nT)) if tiles is None else [int(m) for m in tiles]
    nB = -(-T // block_size)
    out = np.empty((B, NI, len(tile_list), nB))
    for b in range(B):
        for col, m in enumerate(tile_list):
            t = np.arange(m * q_tile, min(T, (m + 1) * q_tile))
            q_rows = _rows(idx_q, b, slice(int(t[0]), int(t[-1]) + 1))
            out[b, :, col, :] = _pooled_row(q_rows, idx_k[b], index_scale, t, block_size, nB)
    return out


def index_block_scores_decode(idx_q, idx_k, block_size, index_scale=None):
    """Decode block scores S[b, g, 0, blk] for the one new token at position L-1.

    idx_q [B, 1, NI, dI] (the new token's index queries), idx_k [B, L, dI] (the index-key
    cache, the new token included).  Selection is per token in decode.
    """
    B, _, NI, dI = idx_q.shape
    L = idx_k.shape[1]
    if index_scale is None or index_scale == 0:
        index_scale = default_scale(dI)
    nB = -(-L // block_size)
    out = np.empty((B, NI, 1, nB))
    for b in range(B):
        q_rows = _rows(idx_q, b, slice(0, 1))
        out[b, :, 0, :] = _pooled_row(q_rows, idx_k[b], index_scale, np.array([L - 1]),
                                      block_size, nB)
    return out


# ---------------------------------------------------------------------------
# Per-KV-head block top-k
# ---------------------------------------------------------------------------

def current_block(last_query_pos: int, block_size: int) -> int:
    """The block that holds a tile's last query: it is always selected."""
    return int(last_query_pos) // block_size


def select_blocks(row_scores, cur: int, top_k: int):
    """One row of the per-KV-head selection.

    Candidates are blocks 0..cur (no block after the current one holds a visible key).
    The current block is kept; the other top_k-1 are the best of 0..cur-1 by score,
    descending, ties to the lower block index, scores compared as reals so that -0 and
    +0 tie.  Returned ascending, padded with -1 to top_k entries.  (Independent top-k per
    KV head: the Chinese topic page's summary; "MSA addresses these issues" paragraph of
    the disconfirmai.com article.)
    """
    r = np.asarray(row_scores, dtype=np.float64)[:cur]
    idx = np.arange(cur)
    order = np.lexsort((idx, -r))             # primary key -score, then block index
    chosen = np.sort(np.concatenate([order[: top_k - 1], [cur]]))
    out = np.full(top_k, -1, dtype=np.int32)
    out[: len(chosen)] = chosen
    return out


def block_topk_prefill(scores, seq_len, q_tile, block_size, top_k, tiles=None):
    """sel[b, g, m, :] for prefill block scores [B, NI, nT (or len(tiles)), nB]."""
    sc = np.asarray(scores, dtype=np.float64)
    B, NI, nR, _ = sc.shape
    nT = -(-seq_len // q_tile)
    tile_list = list(range(nT)) if tiles is None else [int(m) for m in tiles]
    assert len(tile_list) == nR
    sel = np.empty((B, NI, nR, top_k), dtype=np.int32)
    for col, m in enumerate(tile_list):
        cur = current_block(min(seq_len - 1, m * q_tile + q_tile - 1), block_size)
        for b in range(B):
            for g in range(NI):
                sel[b, g, col] = select_blocks(sc[b, g, col], cur, top_k)
    return sel


def block_topk_decode(scores, seq_len, block_size, top_k):
    """sel[b, g, 0, :] for decode block scores [B, NI, 1, nB]; the query is at seq_len-1."""
    sc = np.asarray(scores, dtype=np.float64)
    B, NI, _, _ = sc.shape
    cur = current_block(seq_len - 1, block_size)
    sel = np.empty((B, NI, 1, top_k), dtype=np.int32)
    for b in range(B):
        for g in range(NI):
            sel[b, g, 0] = select_blocks(sc[b, g, 0], cur, top_k)
    return sel


# ---------------------------------------------------------------------------
# Main branch: exact softmax attention over the selected blocks
# ---------------------------------------------------------------------------

def selected_keys(sel_row, block_size, seq_k):
    """All key positions of the selected blocks of one row (padding -1 ignored)."""
    blocks = [int(b) for b in sel_row if b >= 0]
    if not blocks:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate([np.arange(b * block_size, min(seq_k, (b + 1) * block_size))
                           for b in blocks])


def sparse_attention(q, k, v, sel, block_size, q_tile, sm_scale=None, q_offset=0,
                     tiles=None):
    """Exact attention of every query head over its KV group's selected blocks.

    q [B, Sq, Hq, d] with query i at position q_offset + i; k, v [B, Hkv, Sk, d];
    sel [B, Hkv, nT, top_k] (one row per tile of q_tile queries).  For query t and head
    h (KV head g = h // G): J = keys of the selected blocks with j <= t,
    z_j = sm_scale * <q[t, h], k[g, j]>, lse = log sum_J exp(z_j),
    out = sum_J exp(z_j - lse) v[g, j].  A row with empty J gets out = 0, lse = -inf.
    The main branch "attends only to the selected blocks" (aietalks.com, section "MSA
    uses a lightweight index branch before sparse attention"), exactly (Chinese topic
    page summary), with the GQA group sharing its KV head's selection.

    Returns (out [B, Sq, Hq, d] or only the listed tiles' rows, lse [B, Hq, Sq or rows]).
    """
    B, Sq, Hq, d = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    G = Hq // Hkv
    if sm_scale is None or sm_scale == 0:
        sm_scale = default_scale(d)
    nT = -(-Sq // q_tile)
    tile_list = list(range(nT)) if tiles is None else [int(m) for m in tiles]
    rows = np.concatenate([np.arange(m * q_tile, min(Sq, (m + 1) * q_tile))
                           for m in tile_list]) if tile_list else np.zeros(0, int)
    out = np.zeros((B, len(rows), Hq, d))
    lse = np.full((B, Hq, len(rows)), -np.inf)
    r0 = 0
    for m in tile_list:
        t_idx = np.arange(m * q_tile, min(Sq, (m + 1) * q_tile))
        pos = q_offset + t_idx
        for b in range(B):
            for g in range(Hkv):
                J = selected_keys(sel[b, g, m], block_size, Sk)
                if J.size == 0:
                    continue
                q_rows = _rows(q, b, slice(int(t_idx[0]), int(t_idx[-1]) + 1),
                               slice(g * G, (g + 1) * G))                     # [n, G, d]
                z = sm_scale * np.matmul(q_rows, _rows(k, b, g, J).T)        # [n, G, |J|]
                z = np.where((J[None, None, :] <= pos[:, None, None]), z, -np.inf)
                zmax = z.max(axis=2, keepdims=True)
                has = np.isfinite(zmax[..., 0])
                zmax = np.where(np.isfinite(zmax), zmax, 0.0)
                e = np.exp(z - zmax)
                ssum = e.sum(axis=2)
                with np.errstate(divide="ignore", invalid="ignore"):
                    l = np.where(has, np.log(ssum) + zmax[..., 0], -np.inf)
                    p = np.where(has[..., None], e / ssum[..., None], 0.0)
                o = np.matmul(p, _rows(v, b, g, J))                          # [n, G, d]
                out[b, r0:r0 + len(t_idx), g * G:(g + 1) * G, :] = o
                lse[b, g * G:(g + 1) * G, r0:r0 + len(t_idx)] = l.T
        r0 += len(t_idx)
    return out, lse


def full_causal_gqa(q, k, v, sm_scale=None, q_offset=0):
    """Dense causal GQA attention (every key j <= t), the k = all-blocks limit of MSA."""
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    B, Sq, Hq, d = qf.shape
    Hkv, Sk = kf.shape[1], kf.shape[2]
    G = Hq // Hkv
    if sm_scale is None or sm_scale == 0:
        sm_scale = default_scale(d)
    kh = np.repeat(kf, G, axis=1)                       # [B, Hq, Sk, d]
    vh = np.repeat(vf, G, axis=1)
    z = sm_scale * np.einsum("bthc,bhjc->bhtj", qf, kh)
    pos = q_offset + np.arange(Sq)
    z = np.where(np.arange(Sk)[None, None, None, :] <= pos[None, None, :, None], z, -np.inf)
    zmax = z.max(axis=3, keepdims=True)
    e = np.exp(z - zmax)
    ssum = e.sum(axis=3, keepdims=True)
    lse = (np.log(ssum) + zmax)[..., 0]                # [B, Hq, Sq]
    out = np.einsum("bhtj,bhjc->bthc", e / ssum, vh)
    return out, lse


# ---------------------------------------------------------------------------
# Whole pipelines (index -> top-k -> attention), as the three stages chain
# ---------------------------------------------------------------------------

def msa_prefill(q, k, v, idx_q, idx_k, block_size, q_tile, top_k, sm_scale=None,
                index_scale=None, tiles=None):
    """Index scores, per-KV-head selection and sparse attention for prefill."""
    T = q.shape[1]
    scores = index_block_scores_prefill(idx_q, idx_k, block_size, q_tile, index_scale, tiles)
    sel = block_topk_prefill(scores, T, q_tile, block_size, top_k, tiles)
    nT = -(-T // q_tile)
    if tiles is None:
        full_sel = sel
    else:
        full_sel = np.full(sel.shape[:2] + (nT, top_k), -1, dtype=np.int32)
        full_sel[:, :, [int(m) for m in tiles]] = sel
    out, lse = sparse_attention(q, k, v, full_sel, block_size, q_tile, sm_scale, 0, tiles)
    return scores, sel, out, lse


def msa_decode(q, k_cache, v_cache, idx_q, idx_k, block_size, top_k, sm_scale=None,
               index_scale=None):
    """One decode step: the new token (position L-1) scores, selects and attends."""
    L = k_cache.shape[2]
    scores = index_block_scores_decode(idx_q, idx_k, block_size, index_scale)
    sel = block_topk_decode(scores, L, block_size, top_k)
    out, lse = sparse_attention(q, k_cache, v_cache, sel, block_size, 1, sm_scale, L - 1)
    return scores, sel, out, lse


# ---------------------------------------------------------------------------
# Decode over a paged cache with a length per sequence
# ---------------------------------------------------------------------------

def gather_logical(pool_rows, length, block_size):
    """One sequence's logical cache from its physical blocks: pool_rows [nb, ..., Bk, c]
    stacked in logical order, truncated to `length` positions along the block axis."""
    x = np.concatenate([_f64(r) for r in pool_rows], axis=-2)
    return x[..., :length, :]


def msa_decode_paged(q, k_pool, v_pool, idx_q, idx_k_pool, seq_lens, block_table, block_size,
                     top_k, n_blocks, sm_scale=None, index_scale=None):
    """Decode on a paged cache: sequence b's logical cache is the concatenation of the physical
    blocks block_table[b, 0..nb_b-1] truncated to seq_lens[b] positions, and the step is the
    contiguous decode on that cache (the paging is storage only).  k_pool/v_pool
    [P, Hkv, Bk, d], idx_k_pool [P, Bk, dI].  Scores have n_blocks columns, -inf past each
    sequence's blocks; an empty sequence gives sel -1, out 0, lse -inf."""
    seq_lens = np.asarray(seq_lens)
    table = np.asarray(block_table)
    B = len(seq_lens)
    NI = idx_q.shape[2]
    Hq, d = q.shape[2], q.shape[3]
    scores = np.full((B, NI, 1, n_blocks), -np.inf)
    sel = np.full((B, NI, 1, top_k), -1, dtype=np.int32)
    out = np.zeros((B, 1, Hq, d))
    lse = np.full((B, Hq, 1), -np.inf)
    for b in range(B):
        L = int(seq_lens[b])
        if L <= 0:
            continue
        nb = -(-L // block_size)
        phys = [int(x) for x in table[b, :nb]]
        ik = gather_logical([_rows(idx_k_pool, p) for p in phys], L, block_size)   # [L, dI]
        kc = gather_logical([_rows(k_pool, p) for p in phys], L, block_size)       # [Hkv, L, d]
        vc = gather_logical([_rows(v_pool, p) for p in phys], L, block_size)
        sc_b, sel_b, o_b, l_b = msa_decode(_rows(q, slice(b, b + 1)), kc[None], vc[None],
                                           _rows(idx_q, slice(b, b + 1)), ik[None],
                                           block_size, top_k, sm_scale, index_scale)
        scores[b, :, 0, :nb] = sc_b[0, :, 0, :]
        sel[b] = sel_b[0]
        out[b] = o_b[0]
        lse[b] = l_b[0]
    return scores, sel, out, lse


# ---------------------------------------------------------------------------
# Ablation: one selection shared by all KV heads (what MSA does not do)
# ---------------------------------------------------------------------------

def block_topk_shared_prefill(scores, seq_len, q_tile, block_size, top_k):
    """The aggregated selection the pages contrast MSA with ("Sparse Attention Cannot Be
    Directly Ported Across Architectures", paragraph on applying DSA to GQA: aggregating the
    index output into one selection makes every KV head attend to the same set).  The heads'
    block scores are summed -- in float32, in head order, since the sum decides an integer
    selection and is taken in the precision the kernel uses -- and one selection by the usual
    rule is given to every head."""
    sc = np.asarray(scores, dtype=np.float32)
    B, NI, nT, nB = sc.shape
    agg = sc[:, 0].copy()
    for g in range(1, NI):
        agg = (agg + sc[:, g]).astype(np.float32)
    one = block_topk_prefill(agg[:, None].astype(np.float64), seq_len, q_tile, block_size,
                             top_k)
    return np.repeat(one, NI, axis=1)


# ---------------------------------------------------------------------------
# Training: gradients of the sparse attention (the main branch's backward pass)
# ---------------------------------------------------------------------------

def _sample_masks(m, J, block_size, tiles, key_blocks):
    """For a sampled evaluation: whether query tile m's rows are wanted, and which of its
    keys J lie in the wanted key blocks (None: all outputs wanted)."""
    if tiles is None and key_blocks is None:
        return True, np.ones(J.shape, dtype=bool)
    rows = tiles is not None and m in tiles
    keys = (np.isin(J // block_size, key_blocks) if key_blocks is not None
            else np.zeros(J.shape, dtype=bool))
    return rows, keys


def sparse_attention_backward(q, k, v, sel, dout, block_size, q_tile, sm_scale=None,
                              tiles=None, key_blocks=None):
    """Gradients of L = sum(dout * out) for out = sparse_attention(q, k, v, sel, ...) (prefill).

    With z_j = sm_scale q.k_j over the row's keys J (selected blocks, j <= t),
    p = softmax(z), out = sum_j p_j v_j and D = dout . out:
      dv_j += p_j dout,   dp_j = dout . v_j,   ds_j = p_j (dp_j - D),
      dq    = sm_scale sum_j ds_j k_j,        dk_j += sm_scale ds_j q.
    A key block selected by several tiles collects the contributions of all of them.
    Returns (dq [B,T,Hq,d], dk [B,Hkv,T,d], dv [B,Hkv,T,d]) in float64.  Given `tiles` and /
    or `key_blocks`, only dq of those query tiles and dk, dv of those key blocks are formed
    (every tile that selected a wanted block still contributes); the rest stays zero.
    """
    B, T, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    if sm_scale is None or sm_scale == 0:
        sm_scale = default_scale(d)
    tiles = None if tiles is None else set(int(x) for x in tiles)
    key_blocks = None if key_blocks is None else np.asarray(list(key_blocks))
    dq = np.zeros((B, T, Hq, d))
    dk = np.zeros((B, Hkv, T, d))
    dv = np.zeros((B, Hkv, T, d))
    nT = -(-T // q_tile)
    for m in range(nT):
        t_idx = np.arange(m * q_tile, min(T, (m + 1) * q_tile))
        for b in range(B):
            for g in range(Hkv):
                J = selected_keys(sel[b, g, m], block_size, T)
                if J.size == 0:
                    continue
                want_rows, want_keys = _sample_masks(m, J, block_size, tiles, key_blocks)
                if not want_rows and not want_keys.any():
                    continue
                hs = slice(g * G, (g + 1) * G)
                qr = _rows(q, b, slice(int(t_idx[0]), int(t_idx[-1]) + 1), hs)     # [n, G, d]
                dor = _rows(dout, b, slice(int(t_idx[0]), int(t_idx[-1]) + 1), hs)
                kj, vj = _rows(k, b, g, J), _rows(v, b, g, J)                      # [|J|, d]
                z = sm_scale * np.matmul(qr, kj.T)                                 # [n, G, |J|]
                z = np.where(J[None, None, :] <= t_idx[:, None, None], z, -np.inf)
                zmax = z.max(axis=2, keepdims=True)
                zmax = np.where(np.isfinite(zmax), zmax, 0.0)
                e = np.exp(z - zmax)
                ssum = e.sum(axis=2, keepdims=True)
                p = np.where(ssum > 0, e / np.where(ssum > 0, ssum, 1.0), 0.0)
                o = np.matmul(p, vj)                                               # [n, G, d]
                D = (dor * o).sum(axis=2, keepdims=True)                           # [n, G, 1]
                dp = np.matmul(dor, vj.T)                                          # [n, G, |J|]
                ds = p * (dp - D)
                if want_rows:
                    dq[b, t_idx, hs] += sm_scale * np.matmul(ds, kj)
                Jw = J[want_keys]
                dk[b, g, Jw] += sm_scale * np.einsum("ngj,ngc->jc", ds[:, :, want_keys], qr)
                dv[b, g, Jw] += np.einsum("ngj,ngc->jc", p[:, :, want_keys], dor)
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Training the index branch: KL to the main branch's attention
# ---------------------------------------------------------------------------

def index_kl_loss(q, k, idx_q, idx_k, sel, block_size, q_tile, sm_scale=None,
                  index_scale=None, tiles=None, key_blocks=None):
    """KL loss that trains the index branch toward the main branch's attention ("Sparse
    Attention Cannot Be Directly Ported Across Architectures", paragraph introducing MSA;
    aietalks.com, "MSA uses a lightweight index branch before sparse attention": the index
    branch is trained with a KL loss to match the main branch's attention scores).

    Reading taken (the pages give no formula): for token t and KV head g, over the keys J the
    main branch attends (selected blocks, j <= t), the target is the main branch's attention
    distribution averaged over the group's G query heads, held constant; the index
    distribution is the softmax over J of the index logits index_scale <idx_q[t,g], idx_k[j]>;
    the loss is sum over (t, g) of KL(target || index).  Returns (loss, d idx_q, d idx_k) in
    float64, the gradients being those of the summed loss.  Given `tiles` and / or
    `key_blocks`, only the loss and d idx_q of those query tiles and d idx_k of those key
    blocks are formed; the rest stays zero.
    """
    B, T, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    dI = idx_q.shape[-1]
    if sm_scale is None or sm_scale == 0:
        sm_scale = default_scale(d)
    if index_scale is None or index_scale == 0:
        index_scale = default_scale(dI)
    tiles = None if tiles is None else set(int(x) for x in tiles)
    key_blocks = None if key_blocks is None else np.asarray(list(key_blocks))
    loss = 0.0
    diq = np.zeros((B, T, Hkv, dI))
    dik = np.zeros((B, T, dI))
    nT = -(-T // q_tile)
    for m in range(nT):
        t_idx = np.arange(m * q_tile, min(T, (m + 1) * q_tile))
        ts = slice(int(t_idx[0]), int(t_idx[-1]) + 1)
        for b in range(B):
            for g in range(Hkv):
                J = selected_keys(sel[b, g, m], block_size, T)
                if J.size == 0:
                    continue
                want_rows, want_keys = _sample_masks(m, J, block_size, tiles, key_blocks)
                if not want_rows and not want_keys.any():
                    continue
                vis = J[None, :] <= t_idx[:, None]                                 # [n, |J|]
                # target: main attention over J, averaged over the group's heads
                z = sm_scale * np.matmul(_rows(q, b, ts, slice(g * G, (g + 1) * G)),
                                         _rows(k, b, g, J).T)                      # [n, G, |J|]
                z = np.where(vis[:, None, :], z, -np.inf)
                z = z - z.max(axis=2, keepdims=True)
                pm = np.exp(z)
                pm = pm / pm.sum(axis=2, keepdims=True)
                target = pm.mean(axis=1)                                           # [n, |J|]
                # index distribution over the same keys
                qi = _rows(idx_q, b, ts, g)                                        # [n, dI]
                ki = _rows(idx_k, b, J)                                            # [|J|, dI]
                s = np.where(vis, index_scale * np.matmul(qi, ki.T), -np.inf)
                s = s - s.max(axis=1, keepdims=True)
                log_pi = s - np.log(np.exp(s).sum(axis=1, keepdims=True))
                pi = np.exp(log_pi)
                with np.errstate(divide="ignore", invalid="ignore"):
                    terms = np.where(target > 0, target * (np.log(target) - log_pi), 0.0)
                gs = np.where(vis, pi - target, 0.0)                               # dL/ds
                if want_rows:
                    loss += float(terms.sum())
                    diq[b, ts, g] += index_scale * np.matmul(gs, ki)
                Jw = J[want_keys]
                dik[b, Jw] += index_scale * np.matmul(gs[:, want_keys].T, qi)
    return loss, diq, dik
