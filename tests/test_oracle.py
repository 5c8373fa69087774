"""The oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
from tests.oracle_pins import ALL_PINS



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

@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(pin):
    pin(oracle.msa_oracle)


def test_shared_selection_loses_head_diversity():
    """Ablation semantics: the shared selection is identical across heads and recalls fewer
    of each head's own planted blocks than the per-head selection."""
    import numpy as np
    from block_sparse_gqa_02_gb300.configs import CONFIGS
    from block_sparse_gqa_02_gb300.inputs import make_inputs
    cfg = CONFIGS["tiny"]
    x = make_inputs(cfg, input_scale=cfg.head_dim ** -0.5, plant_alpha=3.0)
    sc = oracle.index_block_scores_prefill(x["idx_q"], x["idx_k"], 64, 64)
    own = oracle.block_topk_prefill(sc, cfg.seq, 64, 64, cfg.top_k)
    shared = oracle.block_topk_shared_prefill(sc, cfg.seq, 64, 64, cfg.top_k)
    assert all(np.array_equal(shared[0, 0], shared[0, g]) for g in range(4))

    def recall(sel):
        hit = tot = 0
        for g in range(4):
            for m in range(cfg.n_tiles):
                cur = (m * 64 + 63) // 64
                for pl in x["plants"][0, g]:
                    if pl < cur:
                        tot += 1
                        hit += pl in sel[0, g, m]
        return hit / tot
    assert recall(own) == 1.0
    assert recall(shared) < 0.8


def test_sampled_training_gradients_equal_full():
    """The oracle's sampled evaluation (chosen query tiles, chosen key blocks) returns exactly
    the full evaluation's values there."""
    r = np.random.default_rng(12)
    B, T, Hq, Hkv, d, bs, qt, kk = 1, 40, 4, 2, 3, 4, 2, 3
    q, dout = r.standard_normal((B, T, Hq, d)), r.standard_normal((B, T, Hq, d))
    k, v = r.standard_normal((B, Hkv, T, d)), r.standard_normal((B, Hkv, T, d))
    iq, ik = r.standard_normal((B, T, Hkv, 5)), r.standard_normal((B, T, 5))
    nT, nB = T // qt, T // bs
    sel = oracle.block_topk_prefill(r.standard_normal((B, Hkv, nT, nB)), T, qt, bs, kk)
    tiles, blocks = [1, 7, 19], [0, 4, 9]
    rows = np.concatenate([np.arange(m * qt, (m + 1) * qt) for m in tiles])
    keys = np.concatenate([np.arange(b * bs, (b + 1) * bs) for b in blocks])
    full = oracle.sparse_attention_backward(q, k, v, sel, dout, bs, qt)
    part = oracle.sparse_attention_backward(q, k, v, sel, dout, bs, qt, tiles=tiles,
                                            key_blocks=blocks)
    assert np.array_equal(part[0][:, rows], full[0][:, rows])
    for i in (1, 2):
        assert np.allclose(part[i][:, :, keys], full[i][:, :, keys], rtol=1e-13, atol=1e-14)
    lf, qf, kf = oracle.index_kl_loss(q, k, iq, ik, sel, bs, qt)
    lp, qp, kp = oracle.index_kl_loss(q, k, iq, ik, sel, bs, qt, tiles=tiles, key_blocks=blocks)
    assert np.array_equal(qp[:, rows], qf[:, rows])
    assert np.allclose(kp[:, keys], kf[:, keys], rtol=1e-13, atol=1e-14)
    assert 0 < lp < lf
