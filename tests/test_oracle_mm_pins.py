"""Pins of the multi-modal oracle functions (grid and Q-boundary) against facts other
than themselves: hand-worked masks, the already pinned vertical-slash estimation on a
truncated input, closed forms on planted inputs, a bincount formulation of the lattice
scores, and the probability-mass invariants.  No GPU needed."""
import numpy as np
import pytest
import torch

import oracle as O
from dynamic_sparse_attention_vertical_gb300 import inputs as I
from tests.golden_io import read_fixture


def _ints(vals):
    return np.array([int(x) for x in vals], dtype=np.int64)


def test_grid_mask_hand_worked():
    fx = read_fixture("grid_mask_n8_blk2.txt")
    N, blk = int(fx["N"][0]), int(fx["blk"][0])
    got = O.grid_mask_rows(N, np.arange(N), int(fx["sigma"][0]), int(fx["phi"][0]), blk=blk)
    np.testing.assert_array_equal(got, fx["mask"])


def test_qboundary_mask_hand_worked():
    fx = read_fixture("qboundary_mask_n8_blk2.txt")
    N, blk = int(fx["N"][0]), int(fx["blk"][0])
    sets = [(_ints(fx["V0"]), _ints(fx["S0"])), (_ints(fx["V1"]), _ints(fx["S1"]))]
    got = O.qboundary_mask_rows(N, np.arange(N), _ints(fx["modality"]), sets, blk=blk)
    np.testing.assert_array_equal(got, fx["mask"])


def test_qboundary_mask_with_one_modality_is_the_vertical_slash_mask():
    rng = np.random.default_rng(0)
    N = 300
    v = np.sort(rng.choice(N, 9, replace=False))
    s = np.sort(rng.choice(N, 7, replace=False))
    got = O.qboundary_mask_rows(N, np.arange(N), np.zeros(N, dtype=np.int64), [(v, s)])
    np.testing.assert_array_equal(got, O.vs_mask_rows(N, np.arange(N), v, s))


@pytest.mark.parametrize("R", [64, 100, 257, 300])
def test_window_scores_equal_vertical_slash_scores_of_the_truncated_input(R):
    """Rows ending at R see keys < R only, so the window scores over N keys are the
    (pinned) vertical-slash scores of the first R tokens, padded with zeros."""
    g = torch.Generator().manual_seed(R)
    N, d = 300, 16
    q = torch.randn(N, d, generator=g, dtype=torch.float64)
    k = torch.randn(N, d, generator=g, dtype=torch.float64)
    v, s = O.window_estimate_scores(q, k, R, last_q=64)
    vr, sr = O.vs_estimate_scores(q[:R], k[:R], last_q=64)
    np.testing.assert_allclose(v[:R], vr, rtol=0, atol=1e-12)
    np.testing.assert_allclose(s[:R], sr, rtol=0, atol=1e-12)
    assert np.all(v[R:] == 0) and np.all(s[R:] == 0)
    assert abs(v.sum() - 64) < 1e-9 and abs(s.sum() - 64) < 1e-9


def test_window_before_the_first_64_rows_uses_the_first_64_rows():
    g = torch.Generator().manual_seed(5)
    q = torch.randn(200, 8, generator=g, dtype=torch.float64)
    k = torch.randn(200, 8, generator=g, dtype=torch.float64)
    a = O.window_estimate_scores(q, k, 10, last_q=64)
    b = O.window_estimate_scores(q, k, 64, last_q=64)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_qboundary_estimate_recovers_each_modalitys_planted_sets():
    """Closed form: each modality's window attends only to its own planted columns and
    diagonals (its own dimensions), with a wide margin, so the top-k are the planted sets."""
    runs = [(0, 300), (1, 500), (0, 400), (1, 300)]
    x, mod, planted = I.modality_inputs(1, 1, runs, k_v=12, k_s=8, seed=3)
    got = O.qboundary_estimate(x.q[0], x.k[0], mod.numpy(), 2, 64, 12, 8)
    for m in (0, 1):
        assert got[m][0].tolist() == planted[m][0].tolist()
        assert got[m][1].tolist() == planted[m][1].tolist()


def test_modality_row_end():
    mod = np.array([0, 0, 1, 1, 0, 1, 1, 1])
    assert O.modality_row_end(mod, 0) == 5 and O.modality_row_end(mod, 1) == 8
    assert O.modality_row_end(mod, 2) == 0


@pytest.mark.parametrize("sigma", [3, 7, 16])
def test_grid_scores_equal_a_bincount_of_the_residues(sigma):
    rng = np.random.default_rng(sigma)
    v = rng.random(257)
    v *= 64 / v.sum()
    want = np.bincount(np.arange(v.size) % sigma, weights=v - 64 / v.size, minlength=sigma)
    np.testing.assert_allclose(O.grid_scores(v, sigma), want, rtol=0, atol=1e-12)


def test_grid_fit_closed_forms():
    N = 960
    base = np.full(N, 1.0)
    # a lattice of stride 12 from 5 holds extra mass: it wins over its multiples (24, 36:
    # half and a third of the lines) and its divisors (6, 4: as much mass, more columns)
    v = base.copy()
    v[5::12] += 30.0
    v *= 64 / v.sum()
    assert O.grid_fit(v, 2, 40) == (12, 5)
    # equal lattices at (10, 3) and (10, 7): the smaller phi
    v = base.copy()
    v[3::10] += 20.0
    v[7::10] += 20.0
    v *= 64 / v.sum()
    assert O.grid_fit(v, 8, 12) == (10, 3)
    # a flat profile (exact in binary: 64 / 1024): every E is exactly 0, the smallest
    # sigma and phi win the tie
    v = np.full(1024, 64 / 1024)
    assert O.grid_fit(v, 4, 9) == (4, 0)


@pytest.mark.parametrize("sigma,phi", [(64, 17), (100, 0), (37, 36)])
def test_grid_estimate_recovers_a_planted_lattice(sigma, phi):
    x = I.grid_inputs(1, 1, 4096, sigma, phi, seed=sigma)
    assert O.grid_estimate(x.q[0], x.k[0], 64, 16, 160) == (sigma, phi)


def test_boundary2d_mask_hand_worked():
    fx = read_fixture("boundary2d_mask_n8_blk1.txt")
    N, blk = int(fx["N"][0]), int(fx["blk"][0])
    sets = [(_ints(fx["V0"]), _ints(fx["S0"])), (_ints(fx["V1"]), _ints(fx["S1"]))]
    got = O.boundary2d_mask_rows(N, np.arange(N), _ints(fx["modality"]), sets, blk=blk, min_len=0)
    np.testing.assert_array_equal(got, fx["mask"])


def test_boundary2d_mask_with_one_modality_is_the_vertical_slash_mask():
    rng = np.random.default_rng(1)
    N = 300
    v = np.sort(rng.choice(N, 9, replace=False))
    s = np.sort(rng.choice(N, 7, replace=False))
    got = O.boundary2d_mask_rows(N, np.arange(N), np.zeros(N, dtype=np.int64), [(v, s)])
    np.testing.assert_array_equal(got, O.vs_mask_rows(N, np.arange(N), v, s))


def test_boundary2d_estimate_recovers_sets_planted_in_each_sub_sequence():
    """Closed form: two margin-planted sequences (planted sets in their own positions),
    interleaved by runs into one input, are recovered per modality."""
    a = I.margin_inputs(1, 1, 1024, 16, 12, seed=21)
    b = I.margin_inputs(1, 1, 768, 10, 8, seed=22)
    runs = [(0, 300), (1, 200), (0, 500), (1, 568), (0, 224)]
    mod = np.concatenate([np.full(n, m) for m, n in runs])
    q = torch.empty((1792, 128), dtype=torch.bfloat16)
    k = torch.empty((1792, 128), dtype=torch.bfloat16)
    q[mod == 0], k[mod == 0] = a.q[0], a.k[0]
    q[mod == 1], k[mod == 1] = b.q[0], b.k[0]
    got = O.boundary2d_estimate(q, k, mod, 2, 64, 16, 12)
    assert got[0][0].tolist() == a.planted_cols[0].tolist()
    assert got[0][1].tolist() == a.planted_offsets[0].tolist()
    got = O.boundary2d_estimate(q, k, mod, 2, 64, 10, 8)
    assert got[1][0].tolist() == b.planted_cols[0].tolist()
    assert got[1][1].tolist() == b.planted_offsets[0].tolist()


def test_modality_positions():
    np.testing.assert_array_equal(O.modality_positions(np.array([0, 1, 0, 0, 1, 0, 1, 0])),
                                  [0, 0, 1, 2, 1, 3, 2, 4])
