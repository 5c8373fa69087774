"""Cases for the sanitizer substitute, run by tests/test_gpu_debug_build.py in a process of
their own for each library variant (MSA_LIBRARY_VARIANT=release or debug; one variant per
process).

compute-sanitizer is not available here, so out-of-bounds accesses are looked for in two
other ways.  Every output of these calls is allocated with guard bytes before and after it
(tests/canary.py); after the calls the guards must be intact.  The debug library
(libmsa_debug.so, built with -DMSA_DEBUG) checks every selection entry, block-table entry and
cache length it is given and the coordinates of its tensor copies, and reports a violation
as MSA_ERR_BOUNDS through the device status word without trapping.  On valid inputs the
status must stay clean and the results must match the oracle; on inputs with a bad index the
debug build must report it while the release build skips the entry as documented, and both
give the output of the row without it.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_02_gb300 import _lib
from block_sparse_gqa_02_gb300.configs import CONFIGS
from block_sparse_gqa_02_gb300.inputs import (make_inputs, make_paged_decode_inputs,
                                              random_selection)
from tests.canary import guarded_like
from tests.parity import (check_grad, check_lse, check_out, check_scores,
                          check_selection_exact, to_np)

DEV = "cuda"
VARIANT = os.environ.get("MSA_LIBRARY_VARIANT", "release")
DEBUG = VARIANT == "debug"


def _status_clean():
    _lib.msa_get_device_status()


def _prefill_chain(cfg):
    x = make_inputs(cfg, device=DEV)
    shape = _lib.shape_from_config(cfg)
    B, nR, nB = cfg.batch, shape.n_rows, shape.n_blocks
    sc = guarded_like((B, 4, nR, nB), torch.float32)
    sel = guarded_like((B, 4, nR, cfg.top_k), torch.int32)
    out = guarded_like(tuple(x["q"].shape), x["q"].dtype)
    lse = guarded_like((B, cfg.n_heads_q, cfg.seq), torch.float32)
    _lib.msa_index_scores(shape, x["idx_q"], x["idx_k"], sc.tensor)
    _lib.msa_block_topk(shape, sc.tensor, sel.tensor)
    _lib.msa_sparse_prefill(shape, x["q"], x["k"], x["v"], sel.tensor, out.tensor, lse.tensor)
    _status_clean()
    for gbuf, what in ((sc, "scores"), (sel, "sel"), (out, "out"), (lse, "lse")):
        gbuf.check(f"{cfg.name} {what}")
    g_sc, g_sel = to_np(sc.tensor), to_np(sel.tensor)
    check_scores(g_sc, oracle.index_block_scores_prefill(x["idx_q"], x["idx_k"], cfg.block_size,
                                                         cfg.q_tile))
    check_selection_exact(g_sel, oracle.block_topk_prefill(g_sc, cfg.seq, cfg.q_tile,
                                                           cfg.block_size, cfg.top_k))
    ref_o, ref_l = oracle.sparse_attention(x["q"], x["k"], x["v"], g_sel, cfg.block_size,
                                           cfg.q_tile)
    check_out(out.tensor, ref_o, cfg.dtype)
    check_lse(lse.tensor, ref_l, cfg.dtype)


PREFILL = {
    "tiny_f32": lambda: CONFIGS["tiny"].with_(seq=700),
    "bf16_ragged": lambda: CONFIGS["p32k"].with_(seq=1000, top_k=4, n_plants=3),
    "bf16_b2_g4": lambda: CONFIGS["p32k"].with_(batch=2, seq=1300, n_heads_q=16, top_k=5,
                                                n_plants=2),
}


def test_library_variant():
    assert _lib.load().msa_debug_build() == (1 if DEBUG else 0)


@pytest.mark.parametrize("name", list(PREFILL))
def test_prefill_guarded(name):
    _prefill_chain(PREFILL[name]())


def test_decode_guarded():
    cfg = CONFIGS["d1m"].with_(batch=2, seq=5000, top_k=8, n_plants=3)
    x = make_inputs(cfg, device=DEV)
    shape = _lib.shape_from_config(cfg)
    sc = guarded_like((2, 4, 1, shape.n_blocks), torch.float32)
    sel = guarded_like((2, 4, 1, cfg.top_k), torch.int32)
    out = guarded_like(tuple(x["q"].shape), x["q"].dtype)
    lse = guarded_like((2, cfg.n_heads_q, 1), torch.float32)
    ws = guarded_like((_lib.msa_workspace_bytes(shape, 1) // 4 + 4,), torch.float32)
    _lib.msa_index_scores(shape, x["idx_q"], x["idx_k"], sc.tensor)
    _lib.msa_block_topk(shape, sc.tensor, sel.tensor)
    _lib.msa_sparse_decode(shape, x["q"], x["k"], x["v"], sel.tensor, out.tensor, lse.tensor,
                           ws.tensor)
    _status_clean()
    for gbuf, what in ((sc, "scores"), (sel, "sel"), (out, "out"), (lse, "lse"),
                       (ws, "workspace")):
        gbuf.check(f"decode {what}")
    g_sc, g_sel = to_np(sc.tensor), to_np(sel.tensor)
    check_selection_exact(g_sel, oracle.block_topk_decode(g_sc, cfg.seq, 128, cfg.top_k))
    ref_o, ref_l = oracle.sparse_attention(x["q"], x["k"], x["v"], g_sel, 128, 1, None,
                                           cfg.seq - 1)
    check_out(out.tensor, ref_o, "bf16")
    check_lse(lse.tensor, ref_l, "bf16")


def _paged(cfg, lens, table_fix=None, lens_fix=None):
    x = make_paged_decode_inputs(cfg, lens, device=DEV, seed=3)
    if table_fix:
        table_fix(x["block_table"])
    if lens_fix:
        lens_fix(x["seq_lens"])
    shape = _lib.shape_from_config(cfg, batch=len(lens))
    B, nB = len(lens), shape.n_blocks
    sc = guarded_like((B, 4, 1, nB), torch.float32)
    sel = guarded_like((B, 4, 1, cfg.top_k), torch.int32)
    out = guarded_like(tuple(x["q"].shape), x["q"].dtype)
    lse = guarded_like((B, cfg.n_heads_q, 1), torch.float32)
    ws = guarded_like((_lib.msa_workspace_bytes(shape, 1) // 4 + 4,), torch.float32)
    _lib.msa_index_scores_paged(shape, x["seq_lens"], x["block_table"], x["n_phys"],
                                x["idx_q"], x["idx_k_pool"], sc.tensor)
    _lib.msa_block_topk_ragged(shape, x["seq_lens"], sc.tensor, sel.tensor)
    _lib.msa_sparse_decode_paged(shape, x["seq_lens"], x["block_table"], x["n_phys"], x["q"],
                                 x["k_pool"], x["v_pool"], sel.tensor, out.tensor,
                                 lse.tensor, ws.tensor)
    torch.cuda.synchronize()
    for gbuf, what in ((sc, "scores"), (sel, "sel"), (out, "out"), (lse, "lse"),
                       (ws, "workspace")):
        gbuf.check(f"paged {what}")
    return x, sc, sel, out, lse


def test_paged_decode_guarded():
    lens = [1, 127, 129, 4097, 0]
    cfg = CONFIGS["d1m"].with_(seq=5000, top_k=8, n_plants=0)
    x, sc, sel, out, lse = _paged(cfg, lens)
    _status_clean()
    ref = oracle.msa_decode_paged(x["q"], x["k_pool"], x["v_pool"], x["idx_q"], x["idx_k_pool"],
                                  lens, x["block_table"].cpu().numpy(), 128, cfg.top_k,
                                  -(-cfg.seq // 128))
    check_scores(to_np(sc.tensor), ref[0])


def test_training_guarded():
    """The tensor-core backward and index KL of a small bf16 prefill, guarded."""
    cfg = CONFIGS["p32k"].with_(seq=700, top_k=3, n_plants=0)
    x = make_inputs(cfg, device=DEV)
    shape = _lib.shape_from_config(cfg)
    cur = np.array([min(cfg.seq - 1, m * 64 + 63) // 128 for m in range(shape.n_rows)])
    sel_np = random_selection(np.broadcast_to(cur + 1, (1, 4, shape.n_rows)), cfg.top_k, 5)
    sel = torch.from_numpy(sel_np).to(DEV)
    out = torch.empty_like(x["q"])
    lse = torch.empty((1, cfg.n_heads_q, cfg.seq), dtype=torch.float32, device=DEV)
    _lib.msa_sparse_prefill(shape, x["q"], x["k"], x["v"], sel, out, lse)
    dout = torch.randn(x["q"].shape, generator=torch.Generator(DEV).manual_seed(9),
                       device=DEV).to(x["q"].dtype)
    grads = [guarded_like(tuple(x[n].shape), torch.float32) for n in ("q", "k", "v")]
    ws2 = guarded_like((_lib.msa_workspace_bytes(shape, 2) // 4 + 4,), torch.float32)
    _lib.msa_sparse_prefill_backward(shape, x["q"], x["k"], x["v"], sel, out, lse, dout,
                                     *(gb.tensor for gb in grads), ws2.tensor)
    loss = guarded_like((1,), torch.float32)
    diq = guarded_like(tuple(x["idx_q"].shape), torch.float32)
    dik = guarded_like(tuple(x["idx_k"].shape), torch.float32)
    ws3 = guarded_like((_lib.msa_workspace_bytes(shape, 3) // 4 + 4,), torch.float32)
    _lib.msa_index_kl_loss(shape, x["q"], x["k"], lse, x["idx_q"], x["idx_k"], sel,
                           loss.tensor, diq.tensor, dik.tensor, ws3.tensor)
    _status_clean()
    for gbuf, what in zip(grads + [ws2, loss, diq, dik, ws3],
                          ["dq", "dk", "dv", "ws2", "loss", "d_idx_q", "d_idx_k", "ws3"]):
        gbuf.check(f"training {what}")
    refs = oracle.sparse_attention_backward(x["q"], x["k"], x["v"], sel_np, dout, 128, 64)
    for gbuf, ref, what in zip(grads, refs, ("dq", "dk", "dv")):
        check_grad(gbuf.tensor, ref, "bf16", what)
    l_ref, q_ref, k_ref = oracle.index_kl_loss(x["q"], x["k"], x["idx_q"], x["idx_k"], sel_np,
                                               128, 64)
    assert abs(float(loss.tensor.item()) - l_ref) <= 1e-3 * abs(l_ref) + 1e-6 * cfg.seq * 4
    check_grad(diq.tensor, q_ref, "bf16", "d_idx_q")
    check_grad(dik.tensor, k_ref, "bf16", "d_idx_k")


# ------------------------------------------------------------- bad index inputs

def _prefill_with_sel(cfg, x, sel):
    shape = _lib.shape_from_config(cfg)
    out = torch.empty_like(x["q"])
    lse = torch.empty((cfg.batch, cfg.n_heads_q, cfg.seq), dtype=torch.float32, device=DEV)
    _lib.msa_sparse_prefill(shape, x["q"], x["k"], x["v"], sel, out, lse)
    try:
        _lib.msa_get_device_status()
        status = _lib.MSA_OK
    except _lib.MsaError as e:
        status = e.status
    return status, out, lse


def test_bad_selection_entries():
    """A selection entry past the last block is skipped by both builds (same output as the
    row without it); only the debug build reports it.  A block listed twice is reported by
    the debug build."""
    cfg = CONFIGS["p32k"].with_(seq=1000, top_k=4, n_plants=0)
    x = make_inputs(cfg, device=DEV)
    shape = _lib.shape_from_config(cfg)
    cur = np.array([min(cfg.seq - 1, m * 64 + 63) // 128 for m in range(shape.n_rows)])
    sel_np = random_selection(np.broadcast_to(cur + 1, (1, 4, shape.n_rows)), cfg.top_k, 2)
    # early tiles have fewer candidate blocks than top_k, so their rows end in -1 padding:
    # one padding entry of two rows becomes a block past the last one
    bad = sel_np.copy()
    for (b, g, m) in [(0, 1, 2), (0, 3, 4)]:
        pad = np.flatnonzero(bad[b, g, m] < 0)
        assert pad.size > 0
        bad[b, g, m, pad[0]] = shape.n_blocks + 3
    sel_ok = torch.from_numpy(sel_np).to(DEV)
    sel_bad = torch.from_numpy(bad.astype(np.int32)).to(DEV)
    st_ok, out_ok, lse_ok = _prefill_with_sel(cfg, x, sel_ok)
    st_bad, out_bad, lse_bad = _prefill_with_sel(cfg, x, sel_bad)
    assert st_ok == _lib.MSA_OK
    assert st_bad == (_lib.MSA_ERR_BOUNDS if DEBUG else _lib.MSA_OK)
    assert torch.equal(out_bad, out_ok) and torch.equal(lse_bad, lse_ok)
    if DEBUG:
        # a duplicate: one row lists its first block twice
        dup = sel_np.copy()
        b, g, m = 0, 2, shape.n_rows - 1
        row = [e for e in dup[b, g, m] if e >= 0]
        assert len(row) >= 2
        dup[b, g, m, 1] = row[0]
        st_dup, _, _ = _prefill_with_sel(cfg, x, torch.from_numpy(dup).to(DEV))
        assert st_dup == _lib.MSA_ERR_BOUNDS
        # the status word was cleared by the report: the next valid call is clean
        st_next, out_next, _ = _prefill_with_sel(cfg, x, sel_ok)
        assert st_next == _lib.MSA_OK and torch.equal(out_next, out_ok)


def test_bad_block_table_and_length():
    """A block-table entry outside the pools (its copy reads zeros: no fault) and a cache
    length past the table's capacity (clamped) are reported by the debug build only."""
    lens = [300, 4097, 129]
    cfg = CONFIGS["d1m"].with_(seq=5000, top_k=8, n_plants=0)

    def bad_table(t):
        t[1, 3] = 10 ** 6

    def bad_len(sl):
        sl[2] = 6000
    for fix in ({"table_fix": bad_table}, {"lens_fix": bad_len}):
        _paged(cfg, lens, **fix)
        try:
            _lib.msa_get_device_status()
            status = _lib.MSA_OK
        except _lib.MsaError as e:
            status = e.status
        assert status == (_lib.MSA_ERR_BOUNDS if DEBUG else _lib.MSA_OK), (fix, status)
