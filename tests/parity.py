"""Comparison rules between the CUDA path and the fp64 oracle.

Tolerances (written here once, used by every parity test):
* block scores: |gpu - ref| <= 1e-3 * max(|ref|, 1e-2 * max_row |ref|); -inf must match;
* attention output: bf16 rel-L2 <= 5e-3 and max-abs <= 2e-2; fp32 rel-L2 <= 1e-4 and
  max-abs <= 1e-4;
* lse (natural log): |gpu - ref| <= 2e-3 for bf16 inputs, 1e-4 for fp32 -- fp32
  accumulation of exact bf16 products over <= 8192 keys;
* gradients (dq, dk, dv of the sparse attention): rel-L2 <= 1e-4 for fp32 inputs; for bf16
  rel-L2 <= 1e-2, because the backward uses the forward output rounded to bf16 in
  D = dout . out (relative 2^-9 per element), and max-abs <= 5e-2 of the largest |ref|;
* selections: bit-exact against the oracle's top-k run on the GPU's own fp32 block scores;
  against the oracle's selection from its own fp64 scores, a differing choice must be one
  the score tolerance allows (the agreement rate is reported).
"""
from __future__ import annotations

import numpy as np

SCORE_RTOL = 1e-3
SCORE_FLOOR = 1e-2
OUT_TOL = {"bf16": (5e-3, 2e-2), "f32": (1e-4, 1e-4)}
LSE_TOL = {"bf16": 2e-3, "f32": 1e-4}


def to_np(x):
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        if x.dtype.is_floating_point:
            x = x.double()
        return x.numpy()
    return np.asarray(x)


def score_bound(ref):
    fin = np.isfinite(ref)
    rowmax = np.max(np.where(fin, np.abs(ref), 0.0), axis=-1, keepdims=True)
    return SCORE_RTOL * np.maximum(np.abs(ref), SCORE_FLOOR * rowmax)


def check_scores(gpu, ref, what="scores"):
    gpu, ref = to_np(gpu).astype(np.float64), np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    g_inf, r_inf = np.isneginf(gpu), np.isneginf(ref)
    assert np.array_equal(g_inf, r_inf), f"{what}: -inf pattern differs at " \
        f"{np.argwhere(g_inf != r_inf)[:5].tolist()}"
    assert not np.isnan(gpu).any(), f"{what}: NaN"
    fin = ~r_inf
    err = np.where(fin, np.abs(np.where(fin, gpu, 0.0) - np.where(fin, ref, 0.0)), 0.0)
    bound = score_bound(ref)
    bad = fin & (err > bound)
    assert not bad.any(), f"{what}: {bad.sum()} entries out of tolerance, worst " \
        f"{np.max(err[fin] / bound[fin]):.3g}x bound at {np.argwhere(bad)[:3].tolist()}"
    return float(np.max(err[fin] / np.maximum(bound[fin], 1e-300))) if fin.any() else 0.0


def check_out(gpu, ref, dtype, what="out"):
    gpu, ref = to_np(gpu).astype(np.float64), np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.isfinite(gpu).all(), f"{what}: non-finite values"
    diff = gpu - ref
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))
    mx = float(np.max(np.abs(diff))) if diff.size else 0.0
    rtol, atol = OUT_TOL[dtype]
    assert rel <= rtol and mx <= atol, f"{what}: rel-L2 {rel:.3g} (<= {rtol}), " \
        f"max-abs {mx:.3g} (<= {atol})"
    return rel, mx


def check_lse(gpu, ref, dtype, what="lse"):
    gpu, ref = to_np(gpu).astype(np.float64), np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape
    g_inf, r_inf = np.isneginf(gpu), np.isneginf(ref)
    assert np.array_equal(g_inf, r_inf), f"{what}: -inf pattern differs"
    fin = ~r_inf
    err = np.abs(gpu[fin] - ref[fin])
    mx = float(err.max()) if err.size else 0.0
    assert mx <= LSE_TOL[dtype], f"{what}: max error {mx:.3g} > {LSE_TOL[dtype]}"
    return mx


GRAD_TOL = {"bf16": (1e-2, 5e-2), "f32": (1e-4, 1e-3)}


def check_grad(gpu, ref, dtype, what="grad"):
    gpu, ref = to_np(gpu).astype(np.float64), np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.isfinite(gpu).all(), f"{what}: non-finite values"
    diff = gpu - ref
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))
    mx = float(np.max(np.abs(diff)) / max(np.max(np.abs(ref)), 1e-300))
    rtol, atol = GRAD_TOL[dtype]
    assert rel <= rtol and mx <= atol, f"{what}: rel-L2 {rel:.3g} (<= {rtol}), " \
        f"max-abs / max|ref| {mx:.3g} (<= {atol})"
    return rel, mx


def check_selection_exact(gpu_sel, ref_sel, what="sel"):
    """Bit-exact selection: both sides ranked the same fp32 scores."""
    gpu_sel, ref_sel = to_np(gpu_sel), np.asarray(ref_sel)
    assert gpu_sel.shape == ref_sel.shape, (gpu_sel.shape, ref_sel.shape)
    bad = np.argwhere(np.any(gpu_sel != ref_sel, axis=-1))
    assert bad.size == 0, f"{what}: {len(bad)} selection rows differ, e.g. " \
        f"{bad[:2].tolist()}: {gpu_sel[tuple(bad[0])]} vs {ref_sel[tuple(bad[0])]}"


def check_selection_valid(gpu_sel, ref_sel, ref_scores, cur_blocks, what="sel"):
    """Rows may differ only where fp32-vs-fp64 near-ties make both choices valid.

    gpu_sel, ref_sel [..., k]; ref_scores [..., nB] (oracle fp64); cur_blocks [...].
    Returns the fraction of rows whose selection equals the oracle's exactly.
    """
    gpu_sel, ref_sel = to_np(gpu_sel), np.asarray(ref_sel)
    assert gpu_sel.shape == ref_sel.shape
    same = np.all(gpu_sel == ref_sel, axis=-1)
    bound = score_bound(ref_scores)
    for idx in zip(*np.nonzero(~same)):
        row_g, row_r = gpu_sel[idx], ref_sel[idx]
        cur = int(cur_blocks[idx])
        sc, bd = ref_scores[idx], bound[idx]
        chosen = set(int(b) for b in row_g if b >= 0)
        assert list(row_g[row_g >= 0]) == sorted(chosen), f"{what} {idx}: not ascending"
        assert cur in chosen and all(0 <= b <= cur for b in chosen), f"{what} {idx}: {row_g}"
        assert len(chosen) == len([b for b in row_r if b >= 0]), f"{what} {idx}: count"
        rest = [b for b in range(cur) if b not in chosen]
        # every block the GPU kept must be at least as good as every block it left out,
        # up to the score tolerance on both sides
        lo_in = min((sc[b] for b in chosen if b != cur), default=np.inf)
        hi_out = max((sc[b] for b in rest), default=-np.inf)
        tol = max((bd[b] for b in chosen | set(rest)), default=0.0)
        assert hi_out <= lo_in + 2 * tol, f"{what} {idx}: chose {row_g}, oracle {row_r}, " \
            f"gap {hi_out - lo_in:.3g} > {2 * tol:.3g}"
    return float(same.mean()) if same.size else 1.0


def sample_tiles(n_tiles, n_random=2, seed=0):
    r = np.random.default_rng(seed)
    base = {0, 1, n_tiles // 2, n_tiles - 1}
    base |= set(int(x) for x in r.integers(0, n_tiles, size=n_random))
    return sorted(m for m in base if 0 <= m < n_tiles)
