"""Comparison rules shared by the GPU parity tests.

Tolerances (fixed by the parity contract of this library):
  attention outputs   max |out_gpu - out_ref| <= 2e-3 * max|V|   (bf16 K/V, fp32 accumulation)
  importance scores   |s_gpu - s_ref| <= 1e-4 * s_ref + 1e-30   (relative, with an underflow floor)
  index sets          bit-exact on every row whose reference gap (s_(k) - s_(k+1)) / s_(k) >= 1e-3;
                      other rows: same size, distinct, ascending, and no unselected token scores more
                      than 2e-4 * s_(k) above a selected one (ties may resolve either way).
"""
import numpy as np
import torch

OUT_TOL = 2e-3
SCORE_RTOL = 1e-4
SCORE_ATOL = 1e-30
GAP = 1e-3
TIE_TOL = 2e-4


def to_np(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu").double().numpy()
    return np.asarray(t, dtype=np.float64)


def assert_out_close(gpu, ref, vmax, what="out"):
    g, r = to_np(gpu), to_np(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    err = float(np.max(np.abs(g - r))) if g.size else 0.0
    bound = OUT_TOL * float(vmax)
    assert err <= bound, f"{what}: max abs error {err:.3e} > {bound:.3e}"
    return err


def assert_scores_close(gpu, ref, what="scores"):
    g, r = to_np(gpu), to_np(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    bad = np.abs(g - r) > SCORE_RTOL * np.abs(r) + SCORE_ATOL
    if np.any(bad):
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} entries off; first at {tuple(i)}: gpu {g[tuple(i)]!r} "
                             f"ref {r[tuple(i)]!r}")
    rel = np.abs(g - r) / np.maximum(np.abs(r), 1e-300)
    return float(np.max(rel)) if rel.size else 0.0


def row_gaps(ref_scores, k):
    """Relative gap (s_(k) - s_(k+1)) / s_(k) of each row (inf when k == n)."""
    s = to_np(ref_scores).reshape(-1, np.asarray(ref_scores).shape[-1] if not isinstance(ref_scores, torch.Tensor)
                                  else ref_scores.shape[-1])
    n = s.shape[1]
    if k >= n:
        return np.full(s.shape[0], np.inf)
    part = -np.sort(-s, axis=1)
    sk, sk1 = part[:, k - 1], part[:, k]
    return np.where(sk > 0, (sk - sk1) / np.maximum(sk, 1e-300), np.where(sk1 < sk, np.inf, 0.0))


def check_index_sets(gpu_idx, ref_idx, ref_scores, k):
    """Returns (n_rows, n_gapped, n_exact_match_total).  Raises on any violation."""
    g = gpu_idx.detach().cpu().numpy().reshape(-1, k) if isinstance(gpu_idx, torch.Tensor) else np.asarray(gpu_idx).reshape(-1, k)
    r = np.asarray(ref_idx).reshape(-1, k)
    s = to_np(ref_scores)
    s = s.reshape(-1, s.shape[-1])
    gaps = row_gaps(s, k)
    gapped = 0
    exact = 0
    for row in range(g.shape[0]):
        gi = g[row]
        assert np.all(np.diff(gi) > 0), f"row {row}: indices not strictly ascending"
        assert gi.min() >= 0 and gi.max() < s.shape[1], f"row {row}: index out of range"
        same = np.array_equal(gi, r[row])
        exact += int(same)
        if gaps[row] >= GAP:
            gapped += 1
            assert same, f"row {row}: gapped row (gap {gaps[row]:.2e}) differs from the oracle"
        else:
            sel = np.zeros(s.shape[1], bool)
            sel[gi] = True
            sk = -np.sort(-s[row])[k - 1]
            lo_sel = s[row][sel].min()
            hi_uns = s[row][~sel].max() if (~sel).any() else -np.inf
            assert hi_uns <= lo_sel + TIE_TOL * sk, f"row {row}: unselected {hi_uns} above selected {lo_sel}"
    return g.shape[0], gapped, exact
