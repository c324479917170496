"""The end-to-end selection rule shared by the parity tests and the smoke check.

A top-k row computed on the GPU from its own fp32 scores is compared with the
oracle's selection from fp64 scores.  It passes when:
  - it is well formed: min(k, n_vis) distinct visible entries in ascending
    order, then -1 up to k;
  - it equals the oracle's row, or the two differ only inside the near-tie
    band at the k-th boundary: the oracle's gap between its k-th and
    (k+1)-th score is below GAP, every entry the GPU kept has oracle score
    >= I_(k) - GAP, and every visible entry it left out has oracle score
    <= I_(k) + GAP (I_(k) = the oracle's k-th largest score of the row).
"""
import numpy as np

import oracle

GAP = 1e-5


def check_row(grow: np.ndarray, orow: np.ndarray, scores: np.ndarray, nv: int, k: int,
              gap: float = GAP, label="") -> bool:
    """Checks one row; returns True when it equals the oracle's row."""
    keep = min(k, int(nv))
    assert np.all(grow[keep:] == -1), f"{label}: padding is not -1"
    v = grow[:keep]
    assert np.all(np.diff(v) > 0), f"{label}: not strictly ascending"
    assert keep == 0 or (v[0] >= 0 and v[-1] < nv), f"{label}: entry outside the visible range"
    if np.array_equal(grow, orow):
        return True
    s = np.sort(scores[:nv])[::-1]
    ik = s[k - 1]
    assert s[k - 1] - s[k] < gap, f"{label}: selection differs, boundary gap {s[k - 1] - s[k]}"
    chosen = np.zeros(int(nv), dtype=bool)
    chosen[v] = True
    lo = scores[:nv][chosen].min()
    hi = scores[:nv][~chosen].max()
    assert lo >= ik - gap, f"{label}: kept an entry with score {lo} below I_(k) {ik} - gap"
    assert hi <= ik + gap, f"{label}: left out an entry with score {hi} above I_(k) {ik} + gap"
    return False


def check_selection(gsel: np.ndarray, I: np.ndarray, nvis, k: int, gap: float = GAP):
    """gsel: GPU top-k rows; I: oracle scores of the same rows (columns <
    nvis[r] visible).  Returns (oracle selection, mask of identical rows)."""
    nvis = np.asarray(nvis, dtype=np.int64)
    rsel = oracle.topk(I, nvis, k)
    same = np.array([check_row(gsel[r], rsel[r], I[r], int(nvis[r]), k, gap, f"row {r}")
                     for r in range(gsel.shape[0])], dtype=bool)
    return rsel, same
