"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test ties one oracle function to an independent fact: a hand-worked
fixture in tests/golden/, a library routine (torch fp64 scaled-dot-product
attention, numpy.trace), a closed form on constructed inputs, or an invariant.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from dynamic_sparse_attention_vertical_gb300 import inputs as I
from tests.golden_io import read_cases, read_fixture


def _ints(vals):
    return np.array([int(x) for x in vals], dtype=np.int64)


# ---------------------------------------------------------------- masks ----

@pytest.mark.parametrize("name", ["vs_mask_n8_blk2_a.txt", "vs_mask_n8_blk2_b.txt"])
def test_vs_mask_hand_worked(name):
    fx = read_fixture(name)
    N, blk = int(fx["N"][0]), int(fx["blk"][0])
    got = O.vs_mask_rows(N, np.arange(N), _ints(fx["V"]), _ints(fx["S"]), blk=blk)
    np.testing.assert_array_equal(got, fx["mask"])


def test_vs_expanded_mask_hand_worked():
    fx = read_fixture("vs_expanded_mask_n8_blk2.txt")
    N, blk = int(fx["N"][0]), int(fx["blk"][0])
    got = O.vs_expanded_mask_rows(N, np.arange(N), _ints(fx["V"]), _ints(fx["S"]), blk=blk)
    np.testing.assert_array_equal(got, fx["mask"])


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_vs_expanded_mask_equals_blocks_crossed_by_each_diagonal(seed):
    """Brute force: walk every element (q, q - o) of each selected diagonal and keep
    the whole block pair it lies in; the block-distance rule must give the same mask."""
    rng = np.random.default_rng(seed)
    N, blk = 96, 8
    s = np.sort(rng.choice(N, size=7, replace=False))
    v = np.sort(rng.choice(N, size=5, replace=False))
    pairs = set()
    for o in s:
        for q in range(o, N):
            pairs.add((q // blk, (q - o) // blk))
    want = np.zeros((N, N), dtype=bool)
    for q in range(N):
        for j in range(q + 1):
            want[q, j] = (j < blk or j in set(v.tolist()) or q // blk == j // blk
                          or (q // blk, j // blk) in pairs)
    got = O.vs_expanded_mask_rows(N, np.arange(N), v, s, blk=blk)
    np.testing.assert_array_equal(got, want)
    # the block cover contains the exact diagonals
    exact = O.vs_mask_rows(N, np.arange(N), v, s, blk=blk)
    assert not np.any(exact & ~got)


def test_block_mask_hand_worked():
    fx = read_fixture("block_mask_n8_blk2.txt")
    N, blk = int(fx["N"][0]), int(fx["blk"][0])
    sel = [_ints(fx[f"sel{r}"]) for r in range(N // blk)]
    got = O.block_sparse_mask_rows(N, np.arange(N), sel, blk=blk)
    np.testing.assert_array_equal(got, fx["mask"])


def test_ashape_mask_hand_worked():
    fx = read_fixture("ashape_mask_n8.txt")
    N = int(fx["N"][0])
    got = O.ashape_mask_rows(N, np.arange(N), int(fx["n_init"][0]), int(fx["window"][0]))
    np.testing.assert_array_equal(got, fx["mask"])


# ---------------------------------------------------------------- top-k ----

def test_topk_ties_hand_worked():
    for scores, k, exp in read_cases("topk_ties.txt"):
        assert O.topk_sorted(scores, k).tolist() == exp


def test_topk_matches_python_sorted_on_random_ties():
    rng = np.random.default_rng(7)
    for _ in range(50):
        n = int(rng.integers(1, 200))
        scores = rng.integers(0, 6, size=n).astype(np.float64)
        k = int(rng.integers(0, n + 3))
        ref = sorted(sorted(range(n), key=lambda i: (-scores[i], i))[:min(k, n)])
        assert O.topk_sorted(scores, k).tolist() == ref


def test_topk_decides_in_fp32():
    # 1 + 2^-30 and 1 are different in fp64 but equal in fp32: the lower index wins.
    scores = np.array([1.0, 1.0 + 2.0 ** -30])
    assert O.topk_sorted(scores, 1).tolist() == [0]


# ----------------------------------------------------------- estimation ----

def test_estimate_uniform_hand_worked():
    fx = read_fixture("vs_estimate_uniform_n4.txt")
    N, d, lq = int(fx["N"][0]), int(fx["d"][0]), int(fx["last_q"][0])
    q = np.zeros((N, d))
    k = np.random.default_rng(0).normal(size=(N, d))  # irrelevant: q = 0
    v, s = O.vs_estimate_scores(q, k, lq)
    np.testing.assert_allclose(v, [float(x) for x in fx["v"]], rtol=0, atol=1e-15)
    np.testing.assert_allclose(s, [float(x) for x in fx["s"]], rtol=0, atol=1e-15)
    assert O.topk_sorted(v, 2).tolist() == [int(x) for x in fx["topk_v2"]]
    assert O.topk_sorted(s, 3).tolist() == [int(x) for x in fx["topk_s3"]]


def test_estimate_geometric_hand_worked():
    fx = read_fixture("vs_estimate_geometric_n3.txt")
    N, d, lq = int(fx["N"][0]), int(fx["d"][0]), int(fx["last_q"][0])
    q = np.zeros((N, d))
    q[2, 0] = 2.0
    k = np.zeros((N, d))
    k[:, 0] = [0.0, math.log(2.0), math.log(4.0)]
    v, s = O.vs_estimate_scores(q, k, lq)
    np.testing.assert_allclose(v, [float(x) for x in fx["v"]], rtol=1e-13)
    np.testing.assert_allclose(s, [float(x) for x in fx["s"]], rtol=1e-13)
    # attention of row 2 with V = identity returns the softmax weights
    o, _ = O.masked_attention_rows(q, k, np.eye(3), [2], O.causal_mask_rows(N, [2]))
    np.testing.assert_allclose(o[0], [float(x) for x in fx["v"]], rtol=1e-13)


def _probs_via_torch(q, k):
    """Full causal attention probabilities from torch's fp64 softmax."""
    N, d = q.shape
    logits = torch.from_numpy(q) @ torch.from_numpy(k).T / math.sqrt(d)
    logits = logits.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), float("-inf"))
    return torch.softmax(logits, dim=-1).numpy()


@pytest.mark.parametrize("N,last_q", [(64, 64), (100, 4), (256, 64), (130, 1)])
def test_estimate_matches_trace_brute_force(N, last_q):
    rng = np.random.default_rng(N + last_q)
    d = 16
    q = rng.normal(size=(N, d))
    k = rng.normal(size=(N, d))
    A = _probs_via_torch(q, k)[N - last_q:]          # [last_q, N]
    v_ref = A.sum(axis=0)
    # element (i, p_i - o) of A lies on the diagonal with offset N - last_q - o
    s_ref = np.array([np.trace(A, offset=N - last_q - o) for o in range(N)])
    v, s = O.vs_estimate_scores(q, k, last_q)
    np.testing.assert_allclose(v, v_ref, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(s, s_ref, rtol=1e-12, atol=1e-15)


def test_estimate_mass_invariants():
    rng = np.random.default_rng(3)
    for N, lq in [(512, 64), (300, 17), (64, 64)]:
        q = rng.normal(size=(N, 32)) * 2
        k = rng.normal(size=(N, 32)) * 2
        v, s = O.vs_estimate_scores(q, k, lq)
        assert abs(v.sum() - lq) < 1e-9 and abs(s.sum() - lq) < 1e-9
        assert (v >= 0).all() and (s >= 0).all()
        # no row reaches an offset beyond its own position
        assert np.all(s[N:] == 0) if N < len(s) else True


@pytest.mark.parametrize("N,k_v,k_s", [(1024, 16, 24), (2048, 64, 32)])
def test_margin_inputs_recover_planted_sets(N, k_v, k_s):
    """Closed form: on margin-planted inputs the top-k sets are the planted sets."""
    Hq, Hkv = 4, 2
    x = I.margin_inputs(Hq, Hkv, N, k_v, k_s, seed=11)
    for h in range(Hq):
        g = O.kv_head(h, Hq, Hkv)
        vi, si, v, s = O.vs_estimate(x.q[h], x.k[g], 64, k_v, k_s)
        assert vi.tolist() == x.planted_cols[g].tolist()
        assert si.tolist() == x.planted_offsets[g].tolist()
        for sc, kk in ((v, k_v), (s, k_s)):
            srt = np.sort(sc)[::-1]
            assert srt[kk - 1] >= 1.001 * srt[kk]
    # the two KV heads carry different sets, so a wrong head mapping is caught
    assert x.planted_cols[0].tolist() != x.planted_cols[1].tolist()


# ------------------------------------------------------------ attention ----

def _sdpa(q, k, v):
    qt, kt, vt = (torch.from_numpy(a)[None, None] for a in (q, k, v))
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)[0, 0].numpy()


@pytest.mark.parametrize("N,d", [(200, 128), (64, 32)])
def test_dense_attention_equals_sdpa(N, d):
    rng = np.random.default_rng(N)
    q, k, v = (rng.normal(size=(N, d)) for _ in range(3))
    o, _ = O.attention_rows(q, k, v, np.arange(N), lambda r: O.causal_mask_rows(N, r))
    np.testing.assert_allclose(o, _sdpa(q, k, v), rtol=1e-10, atol=1e-12)


def test_full_budgets_reduce_to_dense():
    N, d = 192, 64
    rng = np.random.default_rng(5)
    q, k, v = (rng.normal(size=(N, d)) for _ in range(3))
    ref = _sdpa(q, k, v)
    vi, si, _, _ = O.vs_estimate(q, k, 64, N, N)
    masks = {
        "vs": lambda r: O.vs_mask_rows(N, r, vi, si),
        "block": lambda r: O.block_sparse_mask_rows(N, r, O.block_sparse_select(q, k, N), 64),
        "ashape": lambda r: O.ashape_mask_rows(N, r, 0, N),
    }
    for name, fn in masks.items():
        np.testing.assert_array_equal(fn(np.arange(N)), O.causal_mask_rows(N, np.arange(N)), err_msg=name)
        o, _ = O.attention_rows(q, k, v, np.arange(N), fn)
        np.testing.assert_allclose(o, ref, rtol=1e-10, atol=1e-12, err_msg=name)


def test_single_key_rows_return_their_value():
    N, d = 96, 16
    rng = np.random.default_rng(9)
    q, k, v = (rng.normal(size=(N, d)) for _ in range(3))
    o, lse = O.attention_rows(q, k, v, np.arange(N), lambda r: O.ashape_mask_rows(N, r, 0, 1))
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, np.einsum("nd,nd->n", q, k) / math.sqrt(d), rtol=1e-12)


def test_weights_sum_to_one_and_lse_counts_keys():
    """V = 1 gives O = 1; q = 0 gives lse = log(number of kept keys)."""
    N, d = 256, 32
    rng = np.random.default_rng(2)
    q, k = rng.normal(size=(N, d)), rng.normal(size=(N, d))
    vi, si, _, _ = O.vs_estimate(q, k, 64, 10, 12)
    fn = lambda r: O.vs_mask_rows(N, r, vi, si)
    o, _ = O.attention_rows(q, k, np.ones((N, d)), np.arange(N), fn)
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-13)
    _, lse = O.attention_rows(np.zeros((N, d)), k, np.ones((N, d)), np.arange(N), fn)
    np.testing.assert_allclose(lse, np.log(fn(np.arange(N)).sum(axis=1)), rtol=1e-13)


def test_attention_is_causal():
    N, d = 160, 16
    rng = np.random.default_rng(4)
    q, k, v = (rng.normal(size=(N, d)) for _ in range(3))
    vi, si, _, _ = O.vs_estimate(q, k, 64, 8, 8)
    fn = lambda r: O.vs_mask_rows(N, r, vi, si)
    o1, _ = O.attention_rows(q, k, v, np.arange(N), fn)
    for qrow in (0, 63, 100):
        v2 = v.copy()
        v2[qrow + 1:] = 1e6
        o2, _ = O.masked_attention_rows(q, k, v2, [qrow], fn(np.array([qrow])))
        np.testing.assert_allclose(o2[0], o1[qrow], rtol=0, atol=1e-12)


# --------------------------------------------------------- block-sparse ----

def test_block_pool_is_block_mean():
    x = np.arange(10 * 3, dtype=np.float64).reshape(10, 3)
    p = O.block_pool(x, 4)
    np.testing.assert_allclose(p, [x[0:4].mean(0), x[4:8].mean(0), x[8:10].mean(0)])


def test_block_selection_closed_form():
    """Block-constant q/k make sigma[r, c] = c (or constant): the selection is known."""
    blk, nb, d = 4, 6, 8
    N = blk * nb
    q = np.zeros((N, d))
    q[:, 0] = 1.0
    k = np.zeros((N, d))
    k[:, 0] = np.repeat(np.arange(nb, dtype=np.float64), blk)   # sigma[r, c] = c
    sel = O.block_sparse_select(q, k, 2, blk)
    assert [s.tolist() for s in sel] == [[0], [0, 1], [1, 2], [2, 3], [3, 4], [4, 5]]
    k[:, 0] = 1.0                                                # all equal: lowest blocks
    sel = O.block_sparse_select(q, k, 2, blk)
    assert [s.tolist() for s in sel] == [[0], [0, 1]] + [[0, 1]] * 4
    k[:, 0] = -np.repeat(np.arange(nb, dtype=np.float64), blk)   # decreasing: earliest blocks
    sel = O.block_sparse_select(q, k, 3, blk)
    assert [s.tolist() for s in sel] == [[0], [0, 1], [0, 1, 2]] + [[0, 1, 2]] * 3


def test_kv_head_mapping():
    assert [O.kv_head(h, 32, 8) for h in (0, 3, 4, 31)] == [0, 0, 1, 7]
    assert [O.kv_head(h, 4, 4) for h in range(4)] == [0, 1, 2, 3]
