"""GPU parity of the exact vertical-slash kernel on offset patterns that exercise its
key windows (the greedy hitting set of the rows' offset intervals, built by the
index kernel in chains of runs): gaps of exactly 128 (same run), 129 and 255 (a
new run that may continue the chain), 256 and more (a new chain), isolated
diagonals, long dense runs, offsets next to N, windows that reach into tile 0,
and more runs than the index kernel has threads (chains that start in one
thread's range and end in another's).
"""
import numpy as np
import pytest
import torch

import oracle as O
from dynamic_sparse_attention_vertical_gb300 import binding as B
from dynamic_sparse_attention_vertical_gb300 import inputs as I
from tests.parity import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def _offsets_from_gaps(start, gaps, N):
    o = [start]
    for g in gaps:
        if o[-1] + g >= N:
            break
        o.append(o[-1] + g)
    return np.array(o, dtype=np.int64)


def _run(N, sis, vis, rows):
    Hq, Hkv = len(sis), 1
    x = I.literal_inputs(Hq, Hkv, N, n_cols=0, n_offsets=0, seed=N % 97)
    q, k, v = x.q.to(DEV), x.k.to(DEV), x.v.to(DEV)
    ks = max(len(s) for s in sis)
    kv = max(1, max(len(c) for c in vis))
    s_idx = torch.full((Hq, ks), -1, dtype=torch.int32)
    v_idx = torch.full((Hq, kv), -1, dtype=torch.int32)
    for h in range(Hq):
        s_idx[h, : len(sis[h])] = torch.as_tensor(sis[h], dtype=torch.int32)
        v_idx[h, : len(vis[h])] = torch.as_tensor(vis[h], dtype=torch.int32)
    out = B.mi_vs_sparse_attn(q, k, v, v_idx.to(DEV), s_idx.to(DEV))
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    for h in range(Hq):
        ref, _ = O.attention_rows(x.q[h], x.k[0], x.v[0], rows,
                                  lambda r, h=h: O.vs_mask_rows(N, r, vis[h], sis[h]))
        assert_close(o[h][rows], ref, f"windows h{h}")


def test_gap_boundaries_all_rows():
    N = 6000
    gaps = [128, 129, 255, 256, 1, 127, 130, 300, 254, 128, 128, 129, 512, 3, 255, 200, 257, 1000]
    sis = [_offsets_from_gaps(5, gaps, N), _offsets_from_gaps(0, gaps[::-1], N)]
    rng = np.random.default_rng(1)
    vis = [np.sort(rng.choice(N, size=40, replace=False)), np.zeros(0, dtype=np.int64)]
    _run(N, sis, vis, np.arange(N))


def test_isolated_diagonals_and_offsets_next_to_n():
    N = 5000
    sis = [np.array([1, 300, 777, 2000, 2001, 4870, N - 2, N - 1]), np.array([N - 1])]
    vis = [np.array([64, 65, 127, 128, 129, 4999]), np.array([0, 1, 2])]
    _run(N, sis, vis, np.arange(N))


def test_dense_runs_with_unaligned_starts():
    N = 4500
    sis = [np.concatenate([np.arange(70, 900), np.arange(1057, 1500), np.arange(3001, 3003)]),
           np.arange(1, N, 7)]
    vis = [np.arange(200, 4000, 37), np.zeros(0, dtype=np.int64)]
    _run(N, sis, vis, np.arange(N))


def test_more_runs_than_index_threads():
    """Over 512 runs: chains start in one index thread's range and continue past it."""
    N = 200_000
    rng = np.random.default_rng(7)
    gaps = rng.choice([129, 170, 255, 256, 300, 128, 64], size=2000)
    sis = [_offsets_from_gaps(0, gaps, N), _offsets_from_gaps(3, rng.permutation(gaps), N)]
    vis = [np.sort(rng.choice(N, size=500, replace=False)), np.sort(rng.choice(N, size=64, replace=False))]
    # whole row blocks around the middle and the end, and scattered rows
    rows = np.unique(np.concatenate([np.arange(65_536 - 128, 65_536 + 128), np.arange(N - 200, N),
                                     rng.choice(N, size=200, replace=False)]))
    _run(N, sis, vis, rows)


def _run_expanded(N, sis, vis, rows):
    Hq = len(sis)
    x = I.literal_inputs(Hq, 1, N, n_cols=0, n_offsets=0, seed=N % 89)
    q, k, v = x.q.to(DEV), x.k.to(DEV), x.v.to(DEV)
    ks = max(len(s) for s in sis)
    kv = max(1, max(len(c) for c in vis))
    s_idx = torch.full((Hq, ks), -1, dtype=torch.int32)
    v_idx = torch.full((Hq, kv), -1, dtype=torch.int32)
    for h in range(Hq):
        s_idx[h, : len(sis[h])] = torch.as_tensor(sis[h], dtype=torch.int32)
        v_idx[h, : len(vis[h])] = torch.as_tensor(vis[h], dtype=torch.int32)
    out = B.mi_vs_sparse_attn(q, k, v, v_idx.to(DEV), s_idx.to(DEV), expanded=True)
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    for h in range(Hq):
        ref, _ = O.attention_rows(x.q[h], x.k[0], x.v[0], rows,
                                  lambda r, h=h: O.vs_expanded_mask_rows(N, r, vis[h], sis[h]))
        assert_close(o[h][rows], ref, f"expanded h{h}")


def test_expanded_pairs_ragged_n_and_block_one_columns():
    """Block-expanded slashes, whose needed 64-key blocks are paired two per tile: a ragged
    last row block (its second own block lies past N), odd block counts, columns in block 1
    (residual whenever block 1 is not needed), isolated far distances."""
    N = 4000  # 31.25 row blocks
    sis = [np.array([1, 64, 65, 200, 1000, 3900]), np.array([5, 3000])]
    vis = [np.array([64, 70, 127, 128, 500, 3999]), np.array([65, 66, 2000])]
    _run_expanded(N, sis, vis, np.arange(N))


def test_expanded_pairs_dense_band_and_gaps():
    N = 6000
    sis = [np.arange(0, 1500, 3), _offsets_from_gaps(7, [64, 65, 128, 129, 200, 640, 1000], N)]
    rng = np.random.default_rng(3)
    vis = [np.sort(rng.choice(N, size=300, replace=False)), np.zeros(0, dtype=np.int64)]
    _run_expanded(N, sis, vis, np.arange(N))
