"""Plain fp64 restatement of the multi-modal patterns (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use this module.  It shares nothing with the CUDA path.

Source: MMInference, in the MInference README mirror (gittoolsai.com), "TL;DR"
(modality-aware permutation sparse attention for the grid pattern of visual
inputs and for modality boundaries in mixed inputs), and the MInference talk
slides (boteman.cn), "MMInference: Grid Head in Multi-Modality" (lines evenly
spaced, horizontal and vertical, often symmetrical; stride and starting
position vary with the context; the vertical-slash pattern turns into a grid
when the input turns from text to visual) and "MMInference: Q-Boundary
pattern" (intra-modality consistency; modality-separated continuity).

The pages give no formula.  The readings this module restates:

Grid head.  One lattice {j : j = phi (mod sigma)} carries both the vertical
lines (key columns) and the horizontal lines (query rows): row q keeps key
j <= q when j < blk, j is in q's own aligned blk-block (the structure every
vertical-slash row keeps), j = phi (mod sigma), or q = phi (mod sigma) (the
whole causal row).  (sigma, phi) are estimated online from the vertical
scores v of the last ``last_q`` queries: over sigma_min <= sigma <= sigma_max
and 0 <= phi < sigma, the lattice whose columns hold the most attention above
the average column, E(sigma, phi) = sum_{j = phi mod sigma} v[j] -
count(sigma, phi) * last_q / N (the scores sum to last_q over N keys); the
largest E wins, ties go to the smaller sigma, then the smaller phi, decided
on E rounded to fp32 (the GPU's precision).

Q-Boundary head.  Each token carries a modality id; a query row follows the
vertical-slash pattern of its own modality.  The index sets of modality m are
estimated, as for a vertical-slash head, from the ``last_q`` query rows that
end at the last token of modality m (the first ``last_q`` rows when that token
comes earlier), over all keys in original positions.

2D-Boundary head (slides, "MMInference: 2D-Boundary pattern"; the boundary
splits both axes).  Each modality's tokens, taken in order, form a
sub-sequence of their own, in which the modality is a vertical-slash head:
its index sets are estimated from the sub-sequence's last ``last_q`` tokens
and its columns, offsets, first block and own block are counted in the
sub-sequence's positions (so a diagonal continues across the other modality's
tokens: "modality-separated continuity").  A query keeps every key of another
modality before it (the cross-modality blocks are kept whole).
"""
from __future__ import annotations

import math

import numpy as np

from .mi_oracle import BLK, as_f64, topk_sorted, vs_mask_rows

__all__ = [
    "window_estimate_scores",
    "modality_row_end",
    "qboundary_estimate",
    "qboundary_mask_rows",
    "grid_scores",
    "grid_fit",
    "grid_estimate",
    "grid_mask_rows",
    "modality_positions",
    "boundary2d_estimate",
    "boundary2d_mask_rows",
]


# ---------------------------------------------------------------------------
# Q-Boundary: estimation windows per modality, masks per query modality
# ---------------------------------------------------------------------------

def window_estimate_scores(q_h, k_g, row_end: int, last_q: int = 64):
    """Vertical and slash scores of one head from the query rows that end at ``row_end``.

    The rows are p_i = max(row_end, last_q) - last_q + i (i < last_q); for each,
      l_ij = <q_{p_i}, k_j> / sqrt(d) for j <= p_i,  a_ij = softmax_j(l_ij),
      v[j] = sum_i a_ij,  s[o] = sum_i a_{i, p_i - o}  (o = p_i - j >= 0).
    Returns (v, s), float64 [N] each (entries no row reaches stay 0).
    """
    q_h = as_f64(q_h)
    k_g = as_f64(k_g)
    N, d = q_h.shape
    last_q = min(last_q, N)
    end = min(max(int(row_end), last_q), N)
    v = np.zeros(N, dtype=np.float64)
    s = np.zeros(N, dtype=np.float64)
    for p in range(end - last_q, end):
        logits = (k_g[: p + 1] @ q_h[p]) / math.sqrt(d)
        a = np.exp(logits - logits.max())
        a /= a.sum()
        v[: p + 1] += a
        s[: p + 1] += a[::-1]          # key p - o sits at offset o
    return v, s


def modality_row_end(modality, m: int) -> int:
    """One past the last token of modality ``m`` (0 when it has none)."""
    idx = np.nonzero(np.asarray(modality) == m)[0]
    return int(idx[-1]) + 1 if idx.size else 0


def qboundary_estimate(q_h, k_g, modality, n_mod: int, last_q: int, k_v: int, k_s: int):
    """Per modality m < n_mod: (v_idx_m, s_idx_m) from the window ending at its last token."""
    out = []
    for m in range(n_mod):
        v, s = window_estimate_scores(q_h, k_g, modality_row_end(modality, m), last_q)
        out.append((topk_sorted(v, k_v), topk_sorted(s, k_s)))
    return out


def qboundary_mask_rows(N: int, rows, modality, idx_sets, blk: int = BLK) -> np.ndarray:
    """Row q keeps what the vertical-slash rule keeps with its modality's sets idx_sets[m]."""
    rows = np.asarray(rows, dtype=np.int64)
    mod = np.asarray(modality)
    out = np.zeros((rows.shape[0], N), dtype=bool)
    for n, q in enumerate(rows):
        v_idx, s_idx = idx_sets[int(mod[q])]
        out[n] = vs_mask_rows(N, [q], v_idx, s_idx, blk=blk)[0]
    return out


# ---------------------------------------------------------------------------
# Grid: lattice fit and mask
# ---------------------------------------------------------------------------

def grid_scores(v, sigma: int, last_q: int = 64) -> np.ndarray:
    """E(sigma, phi) for phi = 0 .. sigma-1: the lattice's vertical score above average."""
    v = np.asarray(v, dtype=np.float64)
    N = v.shape[0]
    out = np.empty(sigma, dtype=np.float64)
    for phi in range(sigma):
        lattice = v[phi::sigma]
        out[phi] = lattice.sum() - lattice.size * (last_q / N)
    return out


def grid_fit(v, sigma_min: int, sigma_max: int, last_q: int = 64):
    """(sigma, phi) of the lattice with the largest E (fp32-rounded); ties: smaller sigma, phi."""
    best = None
    for sigma in range(sigma_min, sigma_max + 1):
        e = grid_scores(v, sigma, last_q).astype(np.float32).astype(np.float64)
        phi = int(np.argmax(e))        # first maximum: the smaller phi
        if best is None or e[phi] > best[0]:
            best = (e[phi], sigma, phi)
    return best[1], best[2]


def grid_estimate(q_h, k_g, last_q: int, sigma_min: int, sigma_max: int):
    """(sigma, phi) of a grid head from the vertical scores of its last ``last_q`` queries."""
    v, _ = window_estimate_scores(q_h, k_g, int(q_h.shape[0]), last_q)
    return grid_fit(v, sigma_min, sigma_max, last_q)


def grid_mask_rows(N: int, rows, sigma: int, phi: int, blk: int = BLK) -> np.ndarray:
    """M[q, j] = j <= q and (j < blk or j//blk == q//blk or j = phi or q = phi (mod sigma))."""
    r = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.arange(N, dtype=np.int64)[None, :]
    keep = (j < blk) | ((j // blk) == (r // blk)) | ((j % sigma) == phi) | ((r % sigma) == phi)
    return (j <= r) & keep


# ---------------------------------------------------------------------------
# 2D-Boundary: each modality a vertical-slash head in its own sub-sequence
# ---------------------------------------------------------------------------

def modality_positions(modality) -> np.ndarray:
    """Position of every token inside its modality's sub-sequence (0-based rank)."""
    mod = np.asarray(modality)
    pos = np.zeros(mod.shape[0], dtype=np.int64)
    for m in np.unique(mod):
        idx = np.nonzero(mod == m)[0]
        pos[idx] = np.arange(idx.size)
    return pos


def boundary2d_estimate(q_h, k_g, modality, n_mod: int, last_q: int, k_v: int, k_s: int):
    """Per modality m: (v_idx_m, s_idx_m) of the vertical-slash estimation of its own
    sub-sequence (positions inside the sub-sequence)."""
    from .mi_oracle import vs_estimate
    mod = np.asarray(modality)
    q_h = as_f64(q_h)
    k_g = as_f64(k_g)
    out = []
    for m in range(n_mod):
        idx = np.nonzero(mod == m)[0]
        if idx.size < last_q:
            out.append((np.zeros(0, dtype=np.int64), np.zeros(0, dtype=np.int64)))
            continue
        vi, si, _, _ = vs_estimate(q_h[idx], k_g[idx], last_q, k_v, k_s)
        out.append((vi, si))
    return out


def boundary2d_mask_rows(N: int, rows, modality, idx_sets, blk: int = BLK, min_len: int = 64) -> np.ndarray:
    """Row q (modality a, sub-sequence position p) keeps key j <= q when j has another
    modality, or when j has modality a and the vertical-slash rule with idx_sets[a] keeps
    sub-sequence positions (p, pos(j)).  A modality with fewer than ``min_len`` tokens
    (too short to estimate) keeps its whole causal sub-sequence."""
    rows = np.asarray(rows, dtype=np.int64)
    mod = np.asarray(modality)
    pos = modality_positions(mod)
    out = np.zeros((rows.shape[0], N), dtype=bool)
    for n, q in enumerate(rows):
        a = int(mod[q])
        same = np.nonzero(mod[: q + 1] == a)[0]
        cross = np.nonzero(mod[: q + 1] != a)[0]
        out[n, cross] = True
        Na = int((mod == a).sum())
        if Na < min_len:
            out[n, same] = True
            continue
        v_idx, s_idx = idx_sets[a]
        keep = vs_mask_rows(Na, [pos[q]], v_idx, s_idx, blk=blk)[0]
        out[n, same] = keep[pos[same]]
    return out
