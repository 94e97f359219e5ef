"""Work counts used to report throughput: kept keys per query row and executed tiles.

Measurement helpers for the benchmark, not part of the compute path.

* Algorithmic FLOPs of a head = 4 * d * (number of (q, j) pairs the pattern
  keeps): one multiply-add for q.k and one for p.v per kept pair and dim.
* Executed FLOPs = 4 * 128^3 per 128x128 tile the attention kernel issues,
  masked elements included (the tensor cores run whole tiles).

Vertical-slash row counts: with A(q) the first block [0, 64) and B(q) the
query's own block [64*(q//64), q] (both always kept), a row keeps
|A u B| + |V outside A u B| + |diagonals outside A u B| - |V and diagonals
both hitting the same key outside A u B|; the last term is a correlation of
the column and offset indicators, done with one FFT.
"""
from __future__ import annotations

import numpy as np
import torch

D = 128
TILE_FLOPS = 4 * 128 * 128 * 128


def _indicator(idx, N, device):
    x = torch.zeros(N, dtype=torch.float64, device=device)
    idx = torch.as_tensor(idx, device=device).long()
    idx = idx[(idx >= 0) & (idx < N)]
    x[idx] = 1.0
    return x


def _prefix(x):
    return torch.cat([torch.zeros(1, dtype=x.dtype, device=x.device), torch.cumsum(x, 0)])


def vs_kept_per_row(N: int, v_idx, s_idx, blk: int = 64, device="cpu") -> torch.Tensor:
    """Kept keys of every row of a vertical-slash head (int64 [N])."""
    V = _indicator(v_idx, N, device)
    S = _indicator(s_idx, N, device)
    q = torch.arange(N, device=device)
    lb = (q // blk) * blk
    ab = torch.clamp(q + 1, max=blk) + torch.where(q >= blk, q - lb + 1, torch.zeros_like(q))
    PV, PS = _prefix(V), _prefix(S)
    c_out = torch.where(q >= blk, PV[lb] - PV[blk], torch.zeros_like(PV[lb]))
    hi = torch.clamp(q - blk + 1, min=0)
    lo = torch.clamp(q - lb + 1, min=0)
    d_out = torch.where(q >= 2 * blk, PS[hi] - PS[torch.minimum(lo, hi)], torch.zeros_like(PV[lb]))
    L = 1 << (2 * N - 1).bit_length()
    full = torch.fft.irfft(torch.fft.rfft(V, L) * torch.fft.rfft(S, L), L)[:N]
    first = torch.zeros(N, dtype=torch.float64, device=device)
    for j in range(min(blk, N)):
        if V[j] > 0:
            first[j:] += S[: N - j]
    local = torch.zeros(N, dtype=torch.float64, device=device)
    for t in range(blk):
        j = lb + t
        ok = (j <= q) & (j >= blk)
        jj = torch.where(ok, j, torch.zeros_like(j))
        local += torch.where(ok, V[jj] * S[torch.where(ok, q - jj, torch.zeros_like(q))],
                             torch.zeros_like(local))
    mid = torch.round(full) - first - local
    return (ab.double() + c_out + d_out - mid).round().long()


def _expanded_dist(N: int, s_idx, blk: int = 64) -> torch.Tensor:
    """Block distances a block-expanded head keeps (bool over 0 .. N//blk)."""
    nb = (N + blk - 1) // blk
    dist = torch.zeros(nb + 2, dtype=torch.bool)
    s = torch.as_tensor(s_idx).long()
    s = s[(s >= 0) & (s < N)]
    dist[s // blk] = True
    dist[(s // blk + 1)[(s % blk) > 0]] = True
    dist[0] = True
    return dist[:nb]


def vs_expanded_kept_per_row(N: int, v_idx, s_idx, blk: int = 64) -> torch.Tensor:
    """Kept keys of every row of a block-expanded vertical-slash head (int64 [N]).

    Row q in block R keeps its own block up to q, the blocks at distances in D
    (1 <= delta <= R, blk keys each), the first block when R is not in D, and the
    selected columns of blocks 1 .. R-1 whose distance is not in D.
    """
    nb = (N + blk - 1) // blk
    dist = _expanded_dist(N, s_idx, blk)
    d1 = dist.clone()
    d1[0] = False
    pd = _prefix(d1.double())                         # |D n [1, x)|
    R = torch.arange(nb)
    blocks = blk * pd[R + 1]                          # distances 1..R
    first = torch.where((R >= 1) & ~dist[R], torch.full_like(R, blk), torch.zeros_like(R)).double()
    v = torch.as_tensor(v_idx).long()
    v = v[(v >= blk) & (v < N)]
    cols = torch.bincount(v // blk, minlength=nb).double()
    notd = (~dist).double()
    notd[0] = 0.0
    L = 1 << (2 * nb).bit_length()
    resid = torch.fft.irfft(torch.fft.rfft(cols, L) * torch.fft.rfft(notd, L), L)[:nb].round()
    per_block = blocks + first + resid
    q = torch.arange(N)
    own = q - (q // blk) * blk + 1
    return (own.double() + per_block[q // blk]).round().long()


def block_kept_per_row(N: int, sel_rows, blk: int = 64) -> torch.Tensor:
    """Kept keys per row of a block-sparse head; sel_rows[r] = selected blocks of query block r."""
    out = torch.zeros(N, dtype=torch.int64)
    for r, sel in enumerate(sel_rows):
        sel = [int(c) for c in sel if int(c) >= 0]
        full = sum(1 for c in sel if c < r)
        rows = torch.arange(r * blk, min(N, r * blk + blk))
        out[rows] = full * blk + ((rows - r * blk + 1) if r in sel else 0)
    return out


def ashape_kept_per_row(N: int, n_init: int, window: int) -> torch.Tensor:
    q = torch.arange(N)
    sink = torch.clamp(q + 1, max=n_init)
    w_lo = torch.clamp(q - window + 1, min=0)
    win = q + 1 - w_lo
    overlap = torch.clamp(sink - w_lo, min=0)
    return sink + win - overlap


def dense_kept_per_row(N: int) -> torch.Tensor:
    return torch.arange(1, N + 1, dtype=torch.int64)


# ------------------------------------------------------ executed tiles ----

def vs_windows(N: int, s_idx) -> np.ndarray:
    """Key windows of an exact vertical-slash head, as positions p (ascending, p < N).

    Row block r (rows 128 r .. 128 r + 127) reads keys 128 r - p .. 128 r - p + 127
    for every window p < 128 r, besides tile 0 (keys 0 .. 127).  A window at p meets
    the offsets p + i - 127 .. p + i in row i of the block, so the windows must hit
    every interval [x, x + 127] with x in [o - 127, o] for each selected offset o
    (and o = 0, the query's own block): the greedy hitting set starts at p = 0 and
    moves to p + 128 while a selected offset lies in (p, p + 128], else to the next
    selected offset.
    """
    s = np.asarray(torch.as_tensor(s_idx).long())
    o = np.unique(np.concatenate([[0], s[(s >= 0) & (s < N)]]))
    ws = []
    p = 0
    while p < N:
        ws.append(p)
        i = int(np.searchsorted(o, p, side="right"))  # first offset > p
        if i >= len(o):
            break
        p = p + 128 if o[i] <= p + 128 else int(o[i])
    return np.asarray(ws, dtype=np.int64)


def _column_tiles(N: int, v_idx, NT: int, residual, first: int = 128) -> int:
    """Column tiles: chunks of 128 entries of the sorted column list from the first
    column at or past key `first` (past tile 0, or past block 0) to the last before
    the row block; a chunk is issued when one of its columns is residual
    (residual(rr, j) over the entries' columns j)."""
    v = torch.as_tensor(v_idx).long()
    v = torch.unique(v[(v >= 0) & (v < N)]).numpy()
    lo = int((v < first).sum())
    col_tiles = 0
    for rr in range(1, NT):
        hi = int(np.searchsorted(v, 128 * rr))  # entries with key < 128 rr
        if hi <= lo:
            continue
        res = residual(rr, v[lo:hi])
        col_tiles += int(np.unique(np.nonzero(res)[0] // 128).size)
    return col_tiles


def vs_tiles(N: int, v_idx, s_idx, expanded: bool = False) -> int:
    """128x128 tiles the vertical-slash kernel issues for one head (all row blocks)."""
    NT = (N + 127) // 128
    if not expanded:
        W = vs_windows(N, s_idx)
        q0 = 128 * np.arange(NT)
        contig = 1 + np.searchsorted(W, q0, side="left")  # tile 0 and the windows p < 128 r
        cov = np.zeros(N + 128, dtype=bool)                # x + 127 for x = 128 r - j
        for p in W:
            cov[p:p + 128] = True
        return int(contig.sum()) + _column_tiles(N, v_idx, NT, lambda rr, j: ~cov[128 * rr - j + 127])
    # block-expanded: row block r needs key block kb when 2r - kb or 2r + 1 - kb (the
    # distances from its two 64-row halves) is a kept 64-block distance, and block 0;
    # with x = 2r + 1 - kb that is f[x] = e[x] | e[x - 1] for x in [0, 2r], plus x = 2r + 1.
    # The needed blocks are paired two per tile.
    e = _expanded_dist(N, s_idx, 64).numpy()
    f = np.zeros(2 * NT + 2, dtype=bool)
    f[: e.shape[0]] = e
    f[1: e.shape[0] + 1] |= e
    pf = np.concatenate([[0], np.cumsum(f)])          # pf[x] = f[0 .. x - 1].sum()
    r = np.arange(NT)
    n = pf[2 * r + 1] + 1
    pairs = int(((n + 1) // 2).sum())
    return pairs + _column_tiles(N, v_idx, NT, lambda rr, j: ~f[2 * rr + 1 - (j >> 6)], first=64)


def dense_tiles(N: int) -> int:
    NT = (N + 127) // 128
    return NT * (NT + 1) // 2


def ashape_tiles(N: int, n_init: int, window: int) -> int:
    total = 0
    for r in range((N + 127) // 128):
        t_lo = max(0, r * 128 - window + 1) // 128
        total += min((n_init + 127) // 128, t_lo) + (r - t_lo + 1)
    return total


def block_tiles(sel_rows) -> int:
    """Tiles of the block-sparse kernel: per 128-row block, the blocks both 64-row halves
    selected pair with each other, and the blocks only one half selected pair with the
    other half's, two 64-key blocks per 128-key tile."""
    total = 0
    for r in range(0, len(sel_rows), 2):
        s0 = {int(c) for c in sel_rows[r] if int(c) >= 0}
        s1 = {int(c) for c in sel_rows[r + 1] if int(c) >= 0} if r + 1 < len(sel_rows) else set()
        both = s0 & s1
        total += (len(both) + 1) // 2 + max(len(s0 - both), len(s1 - both))
    return total
