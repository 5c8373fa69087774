"""The decode entry point that allocates nothing (msa_sparse_decode_static).

Some callers cannot call cudaMalloc where decode runs -- a plugin whose host framework
owns all device memory and gives it no allocator, or a serving loop that must not
allocate after start-up.  msa_sparse_decode_static serves them: it takes no workspace and
keeps the split-KV partial results in a scratch array the library holds on the device.
These tests call it through the C ABI twice in a row (the second call on a different
shape, so it runs over the first call's leftovers) and compare each result with the
regular msa_sparse_decode on the same inputs.  Both entry points run the same kernels in
the same order on the same inputs, so their outputs must be bit-identical (which also puts
them within the bf16 output tolerance the parity tests use).  The file is named so pytest
collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_sparse_gqa_02_gb300 import _lib
from block_sparse_gqa_02_gb300.configs import CONFIGS
from block_sparse_gqa_02_gb300.inputs import make_inputs, random_selection
from tests.parity import check_lse, check_out, to_np


def _decode_both(cfg, sel_seed):
    dev = "cuda"
    x = make_inputs(cfg, device=dev)
    shape = _lib.shape_from_config(cfg)
    cur = (cfg.seq - 1) // cfg.block_size
    sel = torch.from_numpy(random_selection(np.full((cfg.batch, cfg.n_heads_kv, 1), cur + 1),
                                            cfg.top_k, sel_seed)).to(dev)
    lse_shape = (cfg.batch, cfg.n_heads_q, 1)
    # the regular entry point, with a caller-provided workspace
    ws = torch.empty(_lib.msa_workspace_bytes(shape, 1) // 4 + 4, dtype=torch.float32,
                     device=dev)
    out_ref = torch.empty_like(x["q"])
    lse_ref = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    _lib.msa_sparse_decode(shape, x["q"], x["k"], x["v"], sel, out_ref, lse_ref, ws)
    # the entry point without workspace
    out = torch.full_like(x["q"], float("nan"))
    lse = torch.full(lse_shape, float("nan"), dtype=torch.float32, device=dev)
    _lib.msa_sparse_decode_static(shape, x["q"], x["k"], x["v"], sel, out, lse)
    _lib.msa_get_device_status()
    return to_np(out), to_np(lse), to_np(out_ref), to_np(lse_ref)


@pytest.mark.gpu
def test_static_scratch_decode_matches_regular_twice():
    first = CONFIGS["d1m"].with_(batch=8, seq=300_000, n_plants=8)
    second = CONFIGS["d1m"].with_(batch=3, seq=70_001, top_k=24, n_plants=5, seed=11)
    for cfg, seed in ((first, 1), (second, 2)):
        out, lse, out_ref, lse_ref = _decode_both(cfg, seed)
        assert np.array_equal(out, out_ref), f"static decode {cfg.batch}x{cfg.seq}: out differs"
        assert np.array_equal(lse, lse_ref), f"static decode {cfg.batch}x{cfg.seq}: lse differs"
        check_out(out, out_ref, "bf16", f"static decode {cfg.batch}x{cfg.seq}")
        check_lse(lse, lse_ref, "bf16", f"static decode {cfg.batch}x{cfg.seq}")


def test_static_scratch_rejects_oversized_shapes():
    """A shape whose scratch exceeds the static array is refused before anything runs."""
    lib = _lib.load()
    shape = _lib.make_shape(64, 1, 1 << 16, 512, 8, 128, 128, 128, 64, 1, "bf16")
    need = lib.msa_workspace_bytes(ctypes.byref(shape), 1)
    assert need > (8 << 20)
    fake = 1 << 20
    st = lib.msa_sparse_decode_static(ctypes.byref(shape), fake, fake, fake, fake, fake, None,
                                      None)
    assert st == _lib.MSA_ERR_UNSUPPORTED
    assert b"static array" in lib.msa_last_error()
