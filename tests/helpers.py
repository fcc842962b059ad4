"""Acceptance checks shared by the GPU parity tests (pure numpy; no GPU, no oracle internals).

Tolerances (the stated bars, with the readings written down where the stated bar cannot hold):
  * FP4 codes and scales: bit-exact.
  * Top-K: the GPU's set equals the oracle's except for positions whose oracle score lies within
    1e-5 relative of the oracle's k-th largest score; the GPU output must also be ascending,
    duplicate-free, drawn from the candidates, and exactly min(K, #candidates) long, -1 padded.
  * Attention (bf16 output): |gpu - ref_bf16| <= max(2e-3, 1 bf16 ulp of ref) elementwise and
    ||gpu - ref_bf16|| / ||ref_bf16|| <= 1e-3, where ref_bf16 is the oracle's double result
    rounded to bf16.  (A literal 2e-3 max-abs bound on bf16 values of magnitude >= 1, and a
    1e-3 rel-L2 bound against the unrounded double result, are below bf16's own rounding error:
    bf16 rounding alone gives ~1.5e-3 rel-L2.)
  * lse: |gpu - ref| <= 1e-4 * max(1, |ref|).
"""
from __future__ import annotations

import numpy as np

TOPK_BAND = 1e-5
ATTN_ABS = 2e-3
ATTN_REL_L2 = 1e-3
LSE_REL = 1e-4


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)


def check_topk(gpu_row: np.ndarray, ref: dict, K: int, what: str = ""):
    """gpu_row: [K] int32 from the GPU; ref: oracle result {"idx", "pos", "scores"}."""
    pos, scores = ref["pos"], ref["scores"]
    n_cand = len(pos)
    k_eff = min(K, n_cand)
    sel = gpu_row[:k_eff]
    assert np.all(gpu_row[k_eff:] == -1), f"{what}: padding"
    assert np.all(sel >= 0), f"{what}: {int((sel < 0).sum())} empty slots among first {k_eff}"
    assert np.all(np.diff(sel) > 0), f"{what}: not strictly ascending"
    cand = set(pos.tolist())
    assert set(sel.tolist()) <= cand, f"{what}: position outside the candidates"
    ref_set = set(ref["idx"][:k_eff].tolist())
    diff = set(sel.tolist()) ^ ref_set
    if not diff:
        return 0
    kth = np.sort(scores)[::-1][k_eff - 1]
    score_of = dict(zip(pos.tolist(), scores.tolist()))
    bad = [t for t in diff if abs(score_of[t] - kth) > TOPK_BAND * abs(kth)]
    assert not bad, (f"{what}: {len(bad)} selection differences outside the 1e-5 band of the "
                     f"k-th score {kth}: e.g. {[(t, score_of[t]) for t in bad[:5]]}")
    return len(diff)


def check_attn(gpu_out_bits: np.ndarray, gpu_lse: np.ndarray | None, ref_out: np.ndarray,
               ref_lse: np.ndarray, ref_out_bf16_bits: np.ndarray, what: str = ""):
    g = bf16_bits_to_f64(gpu_out_bits)
    r = bf16_bits_to_f64(ref_out_bf16_bits)
    err = np.abs(g - r)
    tol = np.maximum(ATTN_ABS, bf16_ulp(r))
    worst = float((err / tol).max()) if err.size else 0.0
    assert np.all(err <= tol), f"{what}: max err/tol {worst:.3f}"
    nr = np.linalg.norm(r)
    rel = float(np.linalg.norm(g - r) / nr) if nr > 0 else float(np.linalg.norm(g))
    assert rel <= ATTN_REL_L2, f"{what}: rel-L2 {rel:.3e}"
    if gpu_lse is not None:
        fin = np.isfinite(ref_lse)
        assert np.array_equal(fin, np.isfinite(gpu_lse)), f"{what}: lse finiteness"
        d = np.abs(gpu_lse[fin] - ref_lse[fin])
        assert np.all(d <= LSE_REL * np.maximum(1.0, np.abs(ref_lse[fin]))), f"{what}: lse"
    return worst, rel
