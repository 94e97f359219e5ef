"""Work counts used by the benchmark, checked against explicit oracle masks (no GPU)."""
import math

import numpy as np
import pytest

import oracle as O
from dynamic_sparse_attention_vertical_gb300 import flops as F


@pytest.mark.parametrize("N,kv,ks,seed", [(700, 30, 40, 0), (1024, 200, 5, 1), (2048, 64, 300, 2), (64, 3, 3, 3)])
def test_vs_kept_counts_match_oracle_mask(N, kv, ks, seed):
    rng = np.random.default_rng(seed)
    v = np.sort(rng.choice(N, size=min(kv, N), replace=False))
    s = np.sort(rng.choice(N, size=min(ks, N), replace=False))
    ref = O.vs_mask_rows(N, np.arange(N), v, s).sum(axis=1)
    np.testing.assert_array_equal(F.vs_kept_per_row(N, v, s).numpy(), ref)


def test_block_ashape_dense_counts_match_oracle_masks():
    N = 640
    rng = np.random.default_rng(4)
    sel = [np.sort(rng.choice(r + 1, size=min(3, r + 1), replace=False)) for r in range(N // 64)]
    np.testing.assert_array_equal(F.block_kept_per_row(N, sel).numpy(),
                                  O.block_sparse_mask_rows(N, np.arange(N), sel).sum(1))
    for n_init, w in [(128, 100), (0, 1), (64, 4096), (100, 300)]:
        np.testing.assert_array_equal(F.ashape_kept_per_row(N, n_init, w).numpy(),
                                      O.ashape_mask_rows(N, np.arange(N), n_init, w).sum(1))
    np.testing.assert_array_equal(F.dense_kept_per_row(N).numpy(), O.causal_mask_rows(N, np.arange(N)).sum(1))


def _windows_brute(N, s):
    """Windows as the textbook stabbing greedy: row i of a block needs, for each selected
    offset o (and o = 0), a window p with o - i <= p <= o - i + 127; take the intervals
    [x, x + 127] by ascending x and stab each one not yet hit at its right end."""
    xs = sorted({o - i for o in set(s) | {0} for i in range(128)})
    ws, last = [], None
    for x in xs:
        if last is None or x > last:
            last = x + 127
            ws.append(last)
    return [p for p in ws if p < N]


def _vs_tiles_brute(N, v, s):
    NT = (N + 127) // 128
    W = _windows_brute(N, s)
    cols = sorted(v)
    lo = sum(1 for j in cols if j < 128)
    total = 0
    for r in range(NT):
        q0 = 128 * r
        win = [p for p in W if p < q0]
        total += 1 + len(win)
        # column chunks: entries from the first column past tile 0 to the last before the
        # row block; a chunk is issued when one of its columns no window covers
        issued = set()
        for e, j in enumerate(cols):
            if 128 <= j < q0 and not any(q0 - p <= j <= q0 - p + 127 for p in win):
                issued.add((e - lo) // 128)
        total += len(issued)
    return total


@pytest.mark.parametrize("N,kv,ks,seed", [(4096, 300, 7, 0), (8192, 1000, 40, 1), (2112, 50, 0, 2), (3000, 20, 200, 3)])
def test_vs_tile_count_matches_enumeration(N, kv, ks, seed):
    rng = np.random.default_rng(seed)
    v = np.sort(rng.choice(N, size=kv, replace=False))
    s = np.sort(rng.choice(N, size=ks, replace=False)) if ks else np.zeros(0, dtype=np.int64)
    assert F.vs_windows(N, s).tolist() == _windows_brute(N, s.tolist())
    assert F.vs_tiles(N, v, s) == _vs_tiles_brute(N, v.tolist(), s.tolist())


@pytest.mark.parametrize("N,kv,ks,seed", [(1500, 40, 60, 5), (1024, 5, 400, 6), (2048, 300, 9, 7)])
def test_vs_windows_cover_every_kept_key_once(N, kv, ks, seed):
    """Every kept (q, j) of the oracle mask falls in exactly one unit of its row block:
    tile 0 (j < 128), one window (windows mask keys below 128), or the column tiles
    (a column no window covers)."""
    rng = np.random.default_rng(seed)
    v = np.sort(rng.choice(N, size=kv, replace=False))
    s = np.sort(rng.choice(N, size=ks, replace=False))
    W = F.vs_windows(N, s)
    mask = O.vs_mask_rows(N, np.arange(N), v, s)
    vset = set(v.tolist())
    for q in range(N):
        q0 = 128 * (q // 128)
        win = [int(p) for p in W if p < q0]
        for j in np.nonzero(mask[q])[0]:
            n_win = sum(1 for p in win if q0 - p <= j <= q0 - p + 127) if j >= 128 else 0
            units = (1 if j < 128 else 0) + n_win + (1 if (j >= 128 and j < q0 and j in vset and n_win == 0) else 0)
            if j >= q0:  # the own row block: window p = 0 (or tile 0 when q0 = 0)
                assert units == 1 and (q0 == 0 or 0 in win), (q, j)
            assert units == 1, (q, int(j), units)
    # windows are disjoint in key space: consecutive positions at least 128 apart
    assert np.all(np.diff(W) >= 128) and W[0] == 0


def test_windows_of_a_dense_offset_band_are_aligned():
    # offsets 0 .. 999 selected: the windows step by 128 from 0, as aligned tiles would
    N = 4096
    W = F.vs_windows(N, np.arange(1000))
    assert W.tolist() == list(range(0, 1000 + 128, 128))


def test_dense_and_ashape_tiles():
    assert F.dense_tiles(1024) == 8 * 9 // 2
    assert F.ashape_tiles(1024, 128, 4096) == F.dense_tiles(1024)
    # n_init=128, window=128, 16 row blocks: block 0 one tile, block 1 two,
    # blocks 2..15 the sink tile plus two window tiles
    assert F.ashape_tiles(2048, 128, 128) == 1 + 2 + 14 * 3


@pytest.mark.parametrize("N,kv,ks,seed", [(700, 30, 4, 0), (1024, 200, 5, 1), (2048, 64, 40, 2), (64, 3, 3, 3),
                                          (4096, 100, 0, 4)])
def test_vs_expanded_kept_counts_match_oracle_mask(N, kv, ks, seed):
    rng = np.random.default_rng(seed)
    v = np.sort(rng.choice(N, size=min(kv, N), replace=False))
    s = np.sort(rng.choice(N, size=min(ks, N), replace=False)) if ks else np.zeros(0, dtype=np.int64)
    ref = O.vs_expanded_mask_rows(N, np.arange(N), v, s).sum(axis=1)
    np.testing.assert_array_equal(F.vs_expanded_kept_per_row(N, v, s).numpy(), ref)


def _expanded_blocks_brute(r, D):
    """Key blocks row block r needs in the block-expanded mode: a 64-row half at 64-block
    row 2r + rh keeps block kb when (2r + rh) - kb is a kept block distance; block 0 always."""
    return {0} | {kb for kb in range(2 * r + 2) for rh in (0, 1) if (2 * r + rh) - kb in D}


def _vs_expanded_tiles_brute(N, v, s):
    """Enumerate: the needed 64-key blocks of each row block are paired two per tile; a column
    tile (128 entries of the sorted column list past block 0) is issued when one of its columns
    lies in a block the row block does not need."""
    NT = (N + 127) // 128
    D = {0} | {o // 64 for o in s} | {o // 64 + 1 for o in s if o % 64}
    cols = sorted(v)
    lo = sum(1 for j in cols if j < 64)
    total = 0
    for r in range(NT):
        need = _expanded_blocks_brute(r, D)
        total += (len(need) + 1) // 2
        issued = set()
        for e, j in enumerate(cols):
            if 64 <= j < 128 * r and (j >> 6) not in need:
                issued.add((e - lo) // 128)
        total += len(issued)
    return total


@pytest.mark.parametrize("N,kv,ks,seed", [(1500, 40, 60, 5), (2048, 300, 9, 7), (1000, 3, 500, 8)])
def test_vs_expanded_blocks_cover_every_kept_key_once(N, kv, ks, seed):
    """Every kept (q, j) of the oracle's block-expanded mask lies in exactly one needed block of
    its row block or (a column in a block it does not need) in the column tiles."""
    rng = np.random.default_rng(seed)
    v = np.sort(rng.choice(N, size=kv, replace=False))
    s = np.sort(rng.choice(N, size=ks, replace=False))
    D = {0} | {o // 64 for o in s} | {o // 64 + 1 for o in s if o % 64}
    mask = O.vs_expanded_mask_rows(N, np.arange(N), v, s)
    vset = set(v.tolist())
    for q in range(N):
        r = q // 128
        need = _expanded_blocks_brute(r, D)
        for j in np.nonzero(mask[q])[0]:
            in_blocks = (j >> 6) in need
            in_cols = (64 <= j < 128 * r) and (j in vset) and not in_blocks
            assert in_blocks + in_cols == 1, (q, int(j))


@pytest.mark.parametrize("N,kv,ks,seed", [(4096, 300, 7, 0), (8192, 1000, 40, 1), (2112, 50, 0, 2)])
def test_vs_expanded_tile_count_matches_enumeration(N, kv, ks, seed):
    rng = np.random.default_rng(seed)
    v = np.sort(rng.choice(N, size=kv, replace=False))
    s = np.sort(rng.choice(N, size=ks, replace=False)) if ks else np.zeros(0, dtype=np.int64)
    assert F.vs_tiles(N, v, s, expanded=True) == _vs_expanded_tiles_brute(N, v.tolist(), s.tolist())


def test_block_tiles_pairing_covers_each_selection_once():
    """The block-sparse schedule: per 128-row block, blocks both 64-row halves selected
    pair with each other, blocks one half selected pair with the other half's.  Every
    (half, selected block) must be kept in exactly one tile, no tile keeps a block for a
    half that did not select it, and the tile count is the one the bench reports."""
    rng = np.random.default_rng(3)
    for _ in range(200):
        nb = int(rng.integers(2, 80))
        topk = int(rng.integers(1, 40))
        sel = [np.sort(rng.choice(r + 1, size=min(topk, r + 1), replace=False)) for r in range(nb)]
        total = 0
        for r in range(0, nb, 2):
            s0 = set(int(c) for c in sel[r])
            s1 = set(int(c) for c in sel[r + 1]) if r + 1 < nb else set()
            both = sorted(s0 & s1)
            only0, only1 = sorted(s0 - s1), sorted(s1 - s0)
            tiles = [(both[i], both[i + 1] if i + 1 < len(both) else None, True, True)
                     for i in range(0, len(both), 2)]
            for j in range(max(len(only0), len(only1))):
                tiles.append((only0[j] if j < len(only0) else None, only1[j] if j < len(only1) else None,
                              False, False))
            kept = {0: [], 1: []}
            for a, b, common_a, common_b in tiles:
                if common_a:  # a common pair: both halves keep both blocks
                    for h in (0, 1):
                        kept[h] += [a] + ([b] if b is not None else [])
                else:
                    if a is not None:
                        kept[0].append(a)
                    if b is not None:
                        kept[1].append(b)
            assert sorted(kept[0]) == sorted(s0) and sorted(kept[1]) == sorted(s1)
            total += len(tiles)
        assert total == F.block_tiles(sel)


def _offsets_from_gaps(start, gaps, N):
    o = [start]
    for g in gaps:
        if o[-1] + g >= N:
            break
        o.append(o[-1] + g)
    return np.array(o, dtype=np.int64)


@pytest.mark.parametrize("N,seed", [(6000, 0), (200_000, 7)])
def test_windows_on_chain_gap_patterns_match_stabbing_greedy(N, seed):
    """Gaps of 1, 64 and 128 (one run), 129-255 (a run that may continue the chain),
    256 and 300 (a new chain), at sizes with more runs than the index kernel has threads."""
    rng = np.random.default_rng(seed)
    gaps = rng.choice([129, 170, 255, 256, 300, 128, 64, 1], size=3000)
    s = _offsets_from_gaps(int(rng.integers(0, 100)), gaps, N)
    assert F.vs_windows(N, s).tolist() == _windows_brute(N, s.tolist())
