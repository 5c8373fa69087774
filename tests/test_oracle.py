"""The oracle against its pins (CPU only)."""
import pytest

import oracle
from tests.oracle_pins import ALL_PINS


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
