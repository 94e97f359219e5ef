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


def _vs_tiles_brute(N, v, s):
    NT = (N + 127) // 128
    D = {0} | {o >> 7 for o in s} | {(o >> 7) + 1 for o in s if o & 127}
    total = 0
    for r in range(NT):
        contig = {0} | {r - d for d in D if d <= r}
        total += len(contig) + _column_chunks(v, r, contig)
    return total


def _column_chunks(v, r, contig):
    """Column tiles of row block r: 128-entry chunks of the sorted column list, counted
    from the first column past key tile 0, up to the last column before the row block;
    a chunk is issued when it holds a column whose key tile no contiguous tile covers."""
    cols = sorted(v)
    entries = [j for j in cols if 1 <= (j >> 7) < r]
    lo = sum(1 for j in cols if (j >> 7) < 1)
    issued = set()
    for e, j in enumerate(cols):
        if j in entries and (j >> 7) not in contig:
            issued.add((e - lo) // 128)
    return len(issued)


@pytest.mark.parametrize("N,kv,ks,seed", [(4096, 300, 7, 0), (8192, 1000, 40, 1), (2112, 50, 0, 2)])
def test_vs_tile_count_matches_enumeration(N, kv, ks, seed):
    rng = np.random.default_rng(seed)
    v = np.sort(rng.choice(N, size=kv, replace=False))
    s = np.sort(rng.choice(N, size=ks, replace=False)) if ks else np.zeros(0, dtype=np.int64)
    assert F.vs_tiles(N, v, s) == _vs_tiles_brute(N, v.tolist(), s.tolist())


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


def _vs_expanded_tiles_brute(N, v, s):
    """Enumerate: a 128x128 tile (r, t) is issued when one of its four 64x64 blocks is in the
    block-expanded mask's block set, or t = 0, or it holds a residual column."""
    NT = (N + 127) // 128
    D = {0} | {o // 64 for o in s} | {o // 64 + 1 for o in s if o % 64}
    total = 0
    for r in range(NT):
        contig = {0} | {t for t in range(r + 1)
                        if any((2 * r + rh) - (2 * t + kh) in D for rh in (0, 1) for kh in (0, 1))}
        total += len(contig) + _column_chunks(v, r, contig)
    return total


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
