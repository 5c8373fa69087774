"""Seeded synthetic inputs for MSA, shared by the tests, the bench and the oracle runs.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Layouts (row-major, contiguous):

    prefill  q [B, T, Hq, d]   k, v [B, Hkv, T, d]   idx_q [B, T, NI, dI]   idx_k [B, T, dI]
    decode   q [B, 1, Hq, d]   k, v [B, Hkv, L, d]   idx_q [B, 1, NI, dI]   idx_k [B, L, dI]

Recipe (one per named config): Q, K, V, index queries and index keys are i.i.d.
N(0, 1) draws (times the config's ``input_scale``), taken from one torch generator
seeded with the config seed in the fixed order q, k, v, idx_q, idx_k, in fp32, then
cast to the config dtype.  Planting: for every (sequence b, KV head g) a unit
vector u_g (numpy ``default_rng(seed)``) is added to that head's index queries at
every token, and ``plant_alpha * u_g`` is added to the index keys of
``n_plants`` blocks drawn without replacement from blocks 0..nB-2.  The planted
blocks are returned so tests can check that they win the selection.
"""
from __future__ import annotations

import numpy as np
import torch

from .configs import MsaConfig

_TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}

# Rows of the big tensors are drawn in chunks of at most this many fp32 elements, so
# that generating a 16 GiB bf16 tensor never holds a full fp32 copy.
_CHUNK_ELEMS = 1 << 28


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPES[name]


def _randn(shape, gen, device, dtype, scale):
    """N(0,1)*scale drawn in fp32 chunk by chunk along dim 0 (then dim 1), cast to dtype."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1, *shape[2:]) if len(shape) > 2 else out.view(-1, 1)
    row_elems = int(np.prod(flat.shape[1:]))
    rows_per_chunk = max(1, _CHUNK_ELEMS // row_elems)
    for r0 in range(0, flat.shape[0], rows_per_chunk):
        r1 = min(flat.shape[0], r0 + rows_per_chunk)
        x = torch.randn((r1 - r0, *flat.shape[1:]), generator=gen, device=device,
                        dtype=torch.float32)
        if scale != 1.0:
            x.mul_(scale)
        flat[r0:r1].copy_(x)
    return out


def draw_plants(cfg: MsaConfig, seed: int | None = None):
    """Unit vectors u[b, g] (fp32, [B, NI, dI]) and planted block lists per (b, g)."""
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    B, NI, dI = cfg.batch, cfg.n_heads_kv, cfg.index_dim
    n_cand = max(cfg.n_blocks - 1, 0)
    u = np.zeros((B, NI, dI), dtype=np.float32)
    plants = np.zeros((B, NI, min(cfg.n_plants, n_cand)), dtype=np.int64)
    for b in range(B):
        for g in range(NI):
            x = rng.standard_normal(dI)
            u[b, g] = (x / np.linalg.norm(x)).astype(np.float32)
            plants[b, g] = np.sort(rng.choice(n_cand, size=plants.shape[2], replace=False))
    return u, plants


def make_inputs(cfg: MsaConfig, device="cpu", seed: int | None = None,
                input_scale: float | None = None, plant_alpha: float | None = None):
    """Return a dict of tensors on ``device`` plus the planting record.

    ``input_scale`` / ``plant_alpha`` override the config's values (the planted-block
    tests use the tiny shapes with inputs scaled by 1/sqrt(d)).
    """
    seed = cfg.seed if seed is None else seed
    scale = cfg.input_scale if input_scale is None else input_scale
    alpha = cfg.plant_alpha if plant_alpha is None else plant_alpha
    dt = torch_dtype(cfg.dtype)
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    B, Sq, Sk = cfg.batch, cfg.seq_q, cfg.seq_k
    Hq, Hkv, d, dI = cfg.n_heads_q, cfg.n_heads_kv, cfg.head_dim, cfg.index_dim
    q = _randn((B, Sq, Hq, d), gen, dev, dt, scale)
    k = _randn((B, Hkv, Sk, d), gen, dev, dt, scale)
    v = _randn((B, Hkv, Sk, d), gen, dev, dt, scale)
    idx_q = _randn((B, Sq, Hkv, dI), gen, dev, dt, scale)
    idx_k = _randn((B, Sk, dI), gen, dev, dt, scale)

    u, plants = draw_plants(cfg, seed)
    if alpha != 0.0 and plants.shape[2] > 0:
        bs = cfg.block_size
        for b in range(B):
            for g in range(Hkv):
                ug = torch.from_numpy(u[b, g]).to(dev)
                # the query side: every token of head g leans towards u_g
                idx_q[b, :, g, :] = (idx_q[b, :, g, :].float() + ug).to(dt)
                for blk in plants[b, g]:
                    r0, r1 = int(blk) * bs, min(Sk, (int(blk) + 1) * bs)
                    idx_k[b, r0:r1, :] = (idx_k[b, r0:r1, :].float() + alpha * ug).to(dt)
    return {"q": q, "k": k, "v": v, "idx_q": idx_q, "idx_k": idx_k,
            "u": u, "plants": plants}


def random_selection(n_candidates: np.ndarray, top_k: int, seed: int) -> np.ndarray:
    """A random valid block list per row, for testing the attention step on its own.

    ``n_candidates[..., m]`` is the number of visible blocks of row m (blocks
    0..n-1, the last one being the row's current block).  Each row gets the last
    candidate plus ``top_k - 1`` others drawn uniformly, written ascending and
    padded with -1, the same format the top-k step produces.
    """
    rng = np.random.default_rng(seed)
    n_candidates = np.asarray(n_candidates)
    out = np.full(n_candidates.shape + (top_k,), -1, dtype=np.int32)
    for idx in np.ndindex(n_candidates.shape):
        n = int(n_candidates[idx])
        cur = n - 1
        extra = min(top_k - 1, cur)
        others = rng.choice(cur, size=extra, replace=False) if extra > 0 else np.array([], int)
        chosen = np.sort(np.concatenate([others, [cur]]).astype(np.int32))
        out[idx][: len(chosen)] = chosen
    return out


def random_block_scores(shape, seed: int, kind: str = "normal") -> np.ndarray:
    """fp32 block-score tensors for testing the top-k step on its own.

    kind "normal": N(0,1); "ties": small integers (many equal scores, both signed zeros);
    "mixed": normal values with runs of repeated values and signed zeros spliced in.
    """
    rng = np.random.default_rng(seed)
    if kind == "normal":
        x = rng.standard_normal(shape)
    elif kind == "ties":
        x = rng.integers(-3, 4, size=shape).astype(np.float64)
        zero = x == 0
        x[zero] = np.where(rng.random(int(zero.sum())) < 0.5, 0.0, -0.0)
    elif kind == "mixed":
        x = rng.standard_normal(shape)
        flat = x.reshape(-1)
        n = flat.size
        pick = rng.integers(0, n, size=max(1, n // 8))
        flat[pick] = flat[rng.integers(0, n, size=pick.size)]
        flat[rng.integers(0, n, size=max(1, n // 64))] = 0.0
        flat[rng.integers(0, n, size=max(1, n // 64))] = -0.0
    else:
        raise ValueError(kind)
    return x.astype(np.float32)


def make_paged_decode_inputs(cfg: MsaConfig, seq_lens, device="cpu", seed: int | None = None,
                             spare_blocks: int = 3):
    """A paged decode batch: pools of physical 128-key blocks in a shuffled order.

    Sequence b owns ceil(seq_lens[b] / Bk) physical blocks, listed in logical order in
    ``block_table`` (width = the config's block count; unused entries -1).  The pools hold
    ``spare_blocks`` extra blocks nobody owns.  Values are N(0,1) * input_scale draws from
    one torch generator in the order q, k_pool, v_pool, idx_q, idx_k_pool; no planting.
    """
    seed = cfg.seed if seed is None else seed
    rng = np.random.default_rng(seed)
    dt = torch_dtype(cfg.dtype)
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    bs, B = cfg.block_size, len(seq_lens)
    nbs = [-(-int(L) // bs) for L in seq_lens]
    P = sum(nbs) + spare_blocks
    perm = rng.permutation(P)
    table = np.full((B, cfg.n_blocks), -1, dtype=np.int32)
    off = 0
    for b, nb in enumerate(nbs):
        table[b, :nb] = perm[off:off + nb]
        off += nb
    Hq, Hkv, d, dI = cfg.n_heads_q, cfg.n_heads_kv, cfg.head_dim, cfg.index_dim
    s = cfg.input_scale
    return {
        "q": _randn((B, 1, Hq, d), gen, dev, dt, s),
        "k_pool": _randn((P, Hkv, bs, d), gen, dev, dt, s),
        "v_pool": _randn((P, Hkv, bs, d), gen, dev, dt, s),
        "idx_q": _randn((B, 1, Hkv, dI), gen, dev, dt, s),
        "idx_k_pool": _randn((P, bs, dI), gen, dev, dt, s),
        "seq_lens": torch.tensor(np.asarray(seq_lens, dtype=np.int32), device=dev),
        "block_table": torch.from_numpy(table).to(dev),
        "n_phys": P,
    }


def add_score_ramp(x: dict, per_key: float, seed: int = 0) -> dict:
    """Prefill inputs whose attention logits climb along the sequence for half of the query
    heads: a unit vector u (numpy ``default_rng(seed)``) gets weight ``per_key * j / 10`` in
    key j of every KV head and weight 10 in every even query head, so q.k grows by
    ``per_key`` per key for even heads and not at all for odd ones.  Each later block then
    raises an even head's running row maximum by a wide margin while the odd heads' maxima
    stay put (the softmax's rescaling path, taken by some rows of a tile and not others).
    Returns new q and k tensors (same dtype and device); v and the index tensors are kept."""
    q, k = x["q"], x["k"]
    d = q.shape[-1]
    u = np.random.default_rng(seed).standard_normal(d)
    u = torch.from_numpy(u / np.linalg.norm(u)).float()
    T = k.shape[2]
    ramp = (per_key / 10.0) * torch.arange(T, dtype=torch.float32)[:, None] * u[None, :]
    k2 = (k.float().cpu() + ramp[None, None]).to(k.dtype).to(k.device)
    even = torch.zeros(q.shape[2], 1)
    even[0::2] = 10.0
    q2 = (q.float().cpu() + even[None, None] * u[None, None, None]).to(q.dtype).to(q.device)
    out = dict(x)
    out["q"], out["k"] = q2, k2
    return out
