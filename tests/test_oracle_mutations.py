"""The pins are strong enough: each plausible mistake planted in a copy of the oracle
(on the CPU) makes at least one pin fail."""
import importlib.util
import os
import warnings

import numpy as np
import pytest

from tests.oracle_pins import ALL_PINS

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "oracle", "msa_oracle.py")


@pytest.fixture(autouse=True)
def _one_thread_per_library():
    """The pins' problems are tiny: BLAS and torch run them on one thread, so their float64
    results do not depend on how a library splits a product across threads."""
    import torch
    n = torch.get_num_threads()
    torch.set_num_threads(1)
    try:
        from threadpoolctl import threadpool_limits
    except ImportError:
        threadpool_limits = None
    try:
        if threadpool_limits is None:
            yield
        else:
            with threadpool_limits(limits=1, user_api="blas"):
                yield
    finally:
        torch.set_num_threads(n)

def _fresh_oracle():
    spec = importlib.util.spec_from_file_location("msa_oracle_mutant", ORACLE_SRC)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _mut_strict_mask(o):
    base = o.index_logits

    def index_logits(idx_q_rows, idx_k, index_scale, q_pos, key_pos0=0):
        return base(idx_q_rows, idx_k, index_scale, np.asarray(q_pos) - 1, key_pos0)  # j < t
    o.index_logits = index_logits


def _mut_no_index_scale(o):
    base = o.index_logits
    o.index_logits = lambda qr, kk, sc, pos, key_pos0=0: base(qr, kk, 1.0, pos, key_pos0)


def _mut_mean_pool(o):
    def pool_blocks(s, block_size):
        NI, n, L = s.shape
        nB = -(-L // block_size)
        s = np.concatenate([s, np.full((NI, n, nB * block_size - L), -np.inf)], axis=2)
        s = s.reshape(NI, n, nB, block_size)
        fin = np.where(np.isfinite(s), s, np.nan)
        with np.errstate(all="ignore"), warnings.catch_warnings():
            warnings.simplefilter("ignore", RuntimeWarning)
            m = np.nanmean(fin, axis=(1, 3))
        return np.where(np.isnan(m), -np.inf, m)
    o.pool_blocks = pool_blocks


def _mut_ties_high(o):
    def select_blocks(row_scores, cur, top_k):
        r = np.asarray(row_scores, dtype=np.float64)[:cur]
        order = np.lexsort((-np.arange(cur), -r))
        chosen = np.sort(np.concatenate([order[: top_k - 1], [cur]]))
        out = np.full(top_k, -1, dtype=np.int32)
        out[: len(chosen)] = chosen
        return out
    o.select_blocks = select_blocks


def _mut_no_forced_current(o):
    def select_blocks(row_scores, cur, top_k):
        r = np.asarray(row_scores, dtype=np.float64)[:cur + 1]
        order = np.lexsort((np.arange(cur + 1), -r))
        chosen = np.sort(order[:top_k])
        out = np.full(top_k, -1, dtype=np.int32)
        out[: len(chosen)] = chosen
        return out
    o.select_blocks = select_blocks


def _mut_unsorted_output(o):
    def select_blocks(row_scores, cur, top_k):
        r = np.asarray(row_scores, dtype=np.float64)[:cur]
        order = np.lexsort((np.arange(cur), -r))
        chosen = np.concatenate([[cur], order[: top_k - 1]])
        out = np.full(top_k, -1, dtype=np.int32)
        out[: len(chosen)] = chosen
        return out
    o.select_blocks = select_blocks


def _mut_current_block_first_query(o):
    o.current_block = lambda last, bs: max(0, (int(last) - 1)) // bs


def _mut_block_keys_short(o):
    def selected_keys(sel_row, block_size, seq_k):
        blocks = [int(b) for b in sel_row if b >= 0]
        if not blocks:
            return np.zeros(0, dtype=np.int64)
        return np.concatenate([np.arange(b * block_size, min(seq_k, (b + 1) * block_size - 1))
                               for b in blocks])
    o.selected_keys = selected_keys


def _mut_strided_groups(o):
    base = o.sparse_attention

    def sparse_attention(q, k, v, sel, *a, **kw):
        # serve query head h from KV head h % Hkv instead of h // G
        q = np.asarray(q, dtype=np.float64)
        Hq, Hkv = q.shape[2], np.asarray(k).shape[1]
        G = Hq // Hkv
        perm = np.array([(h % Hkv) * G + h // Hkv for h in range(Hq)])
        inv = np.argsort(perm)
        out, lse = base(q[:, :, inv], k, v, sel, *a, **kw)
        return out[:, :, perm], lse[:, perm]
    o.sparse_attention = sparse_attention


def _mut_transposed_index(o):
    # the index key of token j dotted with the index query of head g at token j's slot
    def index_logits(idx_q_rows, idx_k, index_scale, q_pos, key_pos0=0):
        qr = np.asarray(idx_q_rows, dtype=np.float64)
        kk = np.asarray(idx_k, dtype=np.float64)
        s = index_scale * np.einsum("ngc,jc->gnj", qr[:, ::-1, :], kk)
        j = key_pos0 + np.arange(kk.shape[0])
        vis = j[None, :] <= np.asarray(q_pos)[:, None]
        return np.where(vis[None], s, -np.inf)
    o.index_logits = index_logits


def _mut_backward_no_D(o):
    # dq with ds = p * dp, the -D term of the softmax Jacobian dropped: that adds
    # sm_scale * D * (sum_j p_j k_j), the attention output with v replaced by k
    base = o.sparse_attention_backward

    def sparse_attention_backward(q, k, v, sel, dout, block_size, q_tile, sm_scale=None):
        dq, dk, dv = base(q, k, v, sel, dout, block_size, q_tile, sm_scale)
        out, _ = o.sparse_attention(q, k, v, sel, block_size, q_tile, sm_scale)
        kbar, _ = o.sparse_attention(q, k, k, sel, block_size, q_tile, sm_scale)
        scale = sm_scale if sm_scale else 1.0 / np.sqrt(np.asarray(q).shape[-1])
        D = (np.asarray(dout, np.float64) * out).sum(-1, keepdims=True)
        return dq + scale * D * kbar, dk, dv
    o.sparse_attention_backward = sparse_attention_backward


def _mut_kl_first_head_target(o):
    # the target built from the group's first query head only instead of the mean
    base = o.index_kl_loss

    def index_kl_loss(q, k, idx_q, idx_k, sel, block_size, q_tile, sm_scale=None,
                      index_scale=None):
        q = np.asarray(q, dtype=np.float64).copy()
        Hq, Hkv = q.shape[2], np.asarray(k).shape[1]
        G = Hq // Hkv
        for g in range(Hkv):
            q[:, :, g * G:(g + 1) * G] = q[:, :, g * G:g * G + 1]
        return base(q, k, idx_q, idx_k, sel, block_size, q_tile, sm_scale, index_scale)
    o.index_kl_loss = index_kl_loss


def _mut_chunk_keys_from_zero(o):
    # every chunk of index keys masked as if it started at key 0 (causality broken for
    # every chunk after the first)
    base = o.index_logits
    o.index_logits = lambda qr, kk, sc, pos, key_pos0=0: base(qr, kk, sc, pos, 0)


def _mut_shared_max(o):
    # the shared selection ranks by the heads' maximum instead of their sum
    base = o.block_topk_shared_prefill

    def block_topk_shared_prefill(scores, seq_len, q_tile, block_size, top_k):
        sc = np.asarray(scores, dtype=np.float64)
        mx = np.repeat(sc.max(axis=1, keepdims=True), sc.shape[1], axis=1)
        return base(mx / sc.shape[1], seq_len, q_tile, block_size, top_k)
    o.block_topk_shared_prefill = block_topk_shared_prefill


def _mut_shared_exact_sum(o):
    # the shared selection ranks by the exact (float64) sum, not the float32 one
    def block_topk_shared_prefill(scores, seq_len, q_tile, block_size, top_k):
        sc = np.asarray(scores, dtype=np.float64)
        one = o.block_topk_prefill(sc.sum(axis=1, keepdims=True), seq_len, q_tile,
                                   block_size, top_k)
        return np.repeat(one, sc.shape[1], axis=1)
    o.block_topk_shared_prefill = block_topk_shared_prefill


def _mut_sampled_tile_position(o):
    # a sampled evaluation reads the selection row of the tile's place in the list
    # instead of the tile's own row
    base = o.sparse_attention

    def sparse_attention(q, k, v, sel, block_size, q_tile, sm_scale=None, q_offset=0,
                         tiles=None):
        if tiles is not None:
            sel = np.array(sel)
            rows = [int(m) for m in tiles]
            sel[:, :, rows] = np.array(sel)[:, :, list(range(len(rows)))]
        return base(q, k, v, sel, block_size, q_tile, sm_scale, q_offset, tiles)
    o.sparse_attention = sparse_attention


MUTATIONS = [_mut_strict_mask, _mut_no_index_scale, _mut_mean_pool, _mut_ties_high,
             _mut_no_forced_current, _mut_unsorted_output, _mut_current_block_first_query,
             _mut_block_keys_short, _mut_strided_groups, _mut_transposed_index,
             _mut_backward_no_D, _mut_kl_first_head_target, _mut_chunk_keys_from_zero,
             _mut_shared_max, _mut_shared_exact_sum, _mut_sampled_tile_position]


@pytest.mark.parametrize("mutate", MUTATIONS, ids=[m.__name__[5:] for m in MUTATIONS])
def test_some_pin_catches(mutate):
    o = _fresh_oracle()
    mutate(o)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught {mutate.__name__}"
