"""Multi-modal heads on the GPU (grid and Q-boundary) against the oracle, through the C ABI.

- grid estimation: the planted lattice exactly; on unplanted inputs the GPU's lattice scores
  within rounding of the oracle's best;
- grid attention on given (sigma, phi): every row (ragged N) and sampled rows at 32K against
  the oracle's grid mask, the lattice rows included;
- Q-boundary estimation: each modality's planted sets exactly;
- Q-boundary attention: every row against the oracle's per-modality mask, with the GPU's and
  with the oracle's index sets.
"""
import numpy as np
import pytest
import torch

import oracle as O
from dynamic_sparse_attention_vertical_gb300 import binding as B
from dynamic_sparse_attention_vertical_gb300 import inputs as I
from tests.parity import assert_close, band_agree, sample_rows

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def _dev(x):
    return x.q.to(DEV), x.k.to(DEV), x.v.to(DEV)


@pytest.mark.parametrize("N,sigma,phi", [(4096, 64, 17), (4160, 100, 0), (8192, 37, 36)])
def test_grid_estimate_recovers_the_planted_lattice(N, sigma, phi):
    x = I.grid_inputs(4, 2, N, sigma, phi, seed=N + sigma)
    q, k, _ = _dev(x)
    grid = B.mi_grid_estimate(q, k, 16, 160)
    torch.cuda.synchronize()
    assert grid.cpu().tolist() == [[sigma, phi]] * 4
    assert O.grid_estimate(x.q[0], x.k[0], 64, 16, 160) == (sigma, phi)


def test_grid_estimate_unplanted_scores_within_rounding_of_the_best():
    N = 4096
    x = I.literal_inputs(2, 1, N, n_cols=8, n_offsets=4, seed=61)
    q, k, _ = _dev(x)
    grid = B.mi_grid_estimate(q, k, 8, 96).cpu().numpy()
    for h in range(2):
        v, _ = O.window_estimate_scores(x.q[h], x.k[0], N, 64)
        best = max(O.grid_scores(v, s).max() for s in range(8, 97))
        got = O.grid_scores(v, int(grid[h, 0]))[int(grid[h, 1])]
        assert got >= best - 1e-4 * abs(best) - 1e-6, (grid[h], got, best)


@pytest.mark.parametrize("N,sigma,phi", [(2112, 48, 5), (1000, 7, 6), (640, 64, 63)])
def test_grid_attention_every_row(N, sigma, phi):
    x = I.literal_inputs(4, 2, N, n_cols=4, n_offsets=2, seed=N)
    q, k, v = _dev(x)
    grid = torch.tensor([[sigma, phi]] * 4, dtype=torch.int32, device=DEV)
    lse = torch.full((4, N), float("nan"), dtype=torch.float32, device=DEV)
    out = B.mi_grid_attn(q, k, v, grid, max(1, -(-N // B.MI_MAX_KV)), lse=lse)
    torch.cuda.synchronize()
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    for h in range(4):
        g = O.kv_head(h, 4, 2)
        ref, ref_lse = O.attention_rows(x.q[h], x.k[g], x.v[g], np.arange(N),
                                        lambda r: O.grid_mask_rows(N, r, sigma, phi))
        assert_close(o[h], ref, f"grid head {h}")
        np.testing.assert_allclose(l[h], ref_lse, atol=2e-2)


def test_grid_attention_32k_sampled_and_lattice_rows():
    N, sigma, phi = 32768, 100, 37
    x = I.literal_inputs(2, 1, N, n_cols=8, n_offsets=4, seed=77)
    q, k, v = _dev(x)
    grid = torch.tensor([[sigma, phi], [sigma + 3, 2]], dtype=torch.int32, device=DEV)
    out = B.mi_grid_attn(q, k, v, grid, 16)
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    rng = np.random.default_rng(3)
    for h, (s, p) in enumerate([(sigma, phi), (sigma + 3, 2)]):
        lattice_rows = np.arange(p, N, s)[rng.integers(0, (N - p) // s, 24)]
        rows = np.unique(np.concatenate([sample_rows(N, rng, n_random=24, blocks=1), lattice_rows,
                                         [p, N - 1]]))
        ref, _ = O.attention_rows(x.q[h], x.k[0], x.v[0], rows, lambda r: O.grid_mask_rows(N, r, s, p), chunk=32)
        assert_close(o[h][rows], ref, f"grid 32K head {h}")


def test_grid_attention_rejects_bad_lattices():
    N = 1024
    x = I.literal_inputs(2, 1, N, n_cols=2, n_offsets=1, seed=5)
    q, k, v = _dev(x)
    with pytest.raises(B.MIError):  # sigma_min below N / MI_MAX_KV is refused at launch
        B.mi_grid_attn(q, k, v, torch.tensor([[64, 0]] * 2, dtype=torch.int32, device=DEV), 0)
    ws = torch.empty(B.mi_workspace_bytes(B.MI_OP_GRID_ATTN, 2, 1, N), dtype=torch.uint8, device=DEV)
    bad = torch.tensor([[8, 9], [4, 1]], dtype=torch.int32, device=DEV)  # phi >= sigma; sigma < sigma_min
    out = B.mi_grid_attn(q, k, v, bad, 6, workspace=ws)
    assert B.mi_read_status(ws) == B.MI_ERR_INDEX
    # a rejected head keeps only the first block and its own block (no lattice columns, no lattice rows)
    o = out.float().cpu().numpy()
    for h in range(2):
        ref, _ = O.attention_rows(x.q[h], x.k[0], x.v[0], np.arange(N),
                                  lambda r: O.vs_mask_rows(N, r, np.zeros(0, np.int64), np.zeros(0, np.int64)))
        assert_close(o[h], ref, f"rejected grid head {h}")


def test_qboundary_estimate_recovers_each_modalitys_planted_sets():
    runs = [(0, 700), (1, 900), (0, 500), (1, 2048)]
    x, mod, planted = I.modality_inputs(4, 2, runs, k_v=40, k_s=24, seed=9)
    q, k, _ = _dev(x)
    vi, si = B.mi_qboundary_estimate(q, k, mod.to(DEV), 2, k_v=40, k_s=24)
    torch.cuda.synchronize()
    vi, si = vi.cpu().numpy(), si.cpu().numpy()
    for m in (0, 1):
        for h in range(4):
            assert vi[m, h].tolist() == planted[m][0].tolist(), (m, h)
            assert si[m, h].tolist() == planted[m][1].tolist(), (m, h)


@pytest.mark.parametrize("runs", [[(0, 700), (1, 900), (0, 500), (1, 300)], [(1, 100), (0, 1900), (1, 37)]])
def test_qboundary_attention_every_row(runs):
    N = sum(n for _, n in runs)
    mod = torch.cat([torch.full((n,), m, dtype=torch.int32) for m, n in runs])
    x = I.literal_inputs(2, 1, N, n_cols=6, n_offsets=3, seed=N)
    q, k, v = _dev(x)
    k_v, k_s = 64, 48
    vi, si = B.mi_qboundary_estimate(q, k, mod.to(DEV), 2, k_v=k_v, k_s=k_s)
    out = B.mi_qboundary_attn(q, k, v, mod.to(DEV), 2, vi, si)
    torch.cuda.synchronize()
    vi_n, si_n, o = vi.cpu().numpy(), si.cpu().numpy(), out.float().cpu().numpy()
    for h in range(2):
        ref_sets = O.qboundary_estimate(x.q[h], x.k[0], mod.numpy(), 2, 64, k_v, k_s)
        sets = []
        for m in (0, 1):
            vv, ss = O.window_estimate_scores(x.q[h], x.k[0], O.modality_row_end(mod.numpy(), m), 64)
            band_agree(vi_n[m, h], ref_sets[m][0], vv, k_v)
            band_agree(si_n[m, h], ref_sets[m][1], ss, k_s)
            sets.append((vi_n[m, h][vi_n[m, h] >= 0], si_n[m, h][si_n[m, h] >= 0]))
        ref, _ = O.attention_rows(x.q[h], x.k[0], x.v[0], np.arange(N),
                                  lambda r: O.qboundary_mask_rows(N, r, mod.numpy(), sets))
        assert_close(o[h], ref, f"q-boundary head {h}")
    # the attention on the oracle's own sets (index-given path)
    given_v = np.full((2, 2, k_v), -1, dtype=np.int32)
    given_s = np.full((2, 2, k_s), -1, dtype=np.int32)
    refs = []
    for h in range(2):
        rs = O.qboundary_estimate(x.q[h], x.k[0], mod.numpy(), 2, 64, k_v, k_s)
        refs.append(rs)
        for m in (0, 1):
            given_v[m, h, :len(rs[m][0])] = rs[m][0]
            given_s[m, h, :len(rs[m][1])] = rs[m][1]
    out2 = B.mi_qboundary_attn(q, k, v, mod.to(DEV), 2, torch.tensor(given_v, device=DEV),
                               torch.tensor(given_s, device=DEV))
    o2 = out2.float().cpu().numpy()
    for h in range(2):
        ref, _ = O.attention_rows(x.q[h], x.k[0], x.v[0], np.arange(N),
                                  lambda r: O.qboundary_mask_rows(N, r, mod.numpy(), refs[h]))
        assert_close(o2[h], ref, f"q-boundary given head {h}")


def test_qboundary_rejects_unknown_modalities():
    N = 512
    x = I.literal_inputs(2, 1, N, n_cols=2, n_offsets=1, seed=8)
    q, k, v = _dev(x)
    mod = torch.zeros(N, dtype=torch.int32, device=DEV)
    mod[100] = 5
    ws = torch.empty(B.mi_workspace_bytes(B.MI_OP_QBOUNDARY_ESTIMATE, 2, 1, N), dtype=torch.uint8, device=DEV)
    B.mi_qboundary_estimate(q, k, mod, 2, k_v=8, k_s=8, workspace=ws)
    assert B.mi_read_status(ws) == B.MI_ERR_INDEX
    with pytest.raises(B.MIError):
        B.mi_qboundary_estimate(q, k, mod, B.MI_MAX_MODALITIES + 1, k_v=8, k_s=8)


def _runs_modality(runs):
    return np.concatenate([np.full(n, m, dtype=np.int64) for m, n in runs])


@pytest.mark.parametrize("runs", [[(0, 700), (1, 900), (0, 500), (1, 300)],
                                  [(1, 40), (0, 1500), (1, 100), (0, 333)],
                                  [(0, 1000), (1, 50), (0, 500)],
                                  [(0, 2048)]])
def test_boundary2d_attention_every_row(runs):
    N = sum(n for _, n in runs)
    mod = _runs_modality(runs)
    x = I.literal_inputs(4, 2, N, n_cols=6, n_offsets=3, seed=N + len(runs))
    q, k, v = _dev(x)
    k_v, k_s = 48, 40
    lse = torch.full((4, N), float("nan"), dtype=torch.float32, device=DEV)
    out, vi, si = B.mi_boundary2d_attn(q, k, v, runs, k_v=k_v, k_s=k_s, lse=lse)
    torch.cuda.synchronize()
    vi_n, si_n, o, l = vi.cpu().numpy(), si.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy()
    for h in range(4):
        g = O.kv_head(h, 4, 2)
        ref_sets = O.boundary2d_estimate(x.q[h], x.k[g], mod, 2, 64, k_v, k_s)
        sets = []
        for m in (0, 1):
            idx = np.nonzero(mod == m)[0]
            if idx.size >= 64:
                vv, ss = O.vs_estimate_scores(x.q[h][torch.as_tensor(idx)], x.k[g][torch.as_tensor(idx)], 64)
                band_agree(vi_n[m, h], ref_sets[m][0], vv, k_v)
                band_agree(si_n[m, h], ref_sets[m][1], ss, k_s)
            sets.append((vi_n[m, h][vi_n[m, h] >= 0], si_n[m, h][si_n[m, h] >= 0]))
        ref, ref_lse = O.attention_rows(x.q[h], x.k[g], x.v[g], np.arange(N),
                                        lambda r: O.boundary2d_mask_rows(N, r, mod, sets))
        assert_close(o[h], ref, f"2D-boundary head {h}")
        np.testing.assert_allclose(l[h], ref_lse, atol=2e-2)


def test_boundary2d_attention_on_oracle_sets():
    runs = [(0, 600), (1, 800), (0, 400), (1, 248)]
    N = sum(n for _, n in runs)
    mod = _runs_modality(runs)
    x = I.literal_inputs(2, 1, N, n_cols=4, n_offsets=2, seed=99)
    q, k, v = _dev(x)
    k_v, k_s = 32, 24
    gv = np.full((2, 2, k_v), -1, dtype=np.int32)
    gs = np.full((2, 2, k_s), -1, dtype=np.int32)
    refs = []
    for h in range(2):
        rs = O.boundary2d_estimate(x.q[h], x.k[0], mod, 2, 64, k_v, k_s)
        refs.append(rs)
        for m in (0, 1):
            gv[m, h, :len(rs[m][0])] = rs[m][0]
            gs[m, h, :len(rs[m][1])] = rs[m][1]
    out, _, _ = B.mi_boundary2d_attn(q, k, v, runs, v_idx=torch.tensor(gv, device=DEV),
                                     s_idx=torch.tensor(gs, device=DEV), given=True)
    o = out.float().cpu().numpy()
    for h in range(2):
        ref, _ = O.attention_rows(x.q[h], x.k[0], x.v[0], np.arange(N),
                                  lambda r: O.boundary2d_mask_rows(N, r, mod, refs[h]))
        assert_close(o[h], ref, f"2D-boundary given head {h}")


def test_boundary2d_rejects_malformed_runs():
    N = 256
    x = I.literal_inputs(2, 1, N, n_cols=2, n_offsets=1, seed=3)
    q, k, v = _dev(x)
    for runs in ([(0, 100), (1, 100)], [(2, 256)], [(0, 0), (1, 256)]):
        with pytest.raises(B.MIError):
            B.mi_boundary2d_attn(q, k, v, runs, k_v=8, k_s=8)


def test_mm_heads_128k_sampled():
    """The three multi-modal calls at 128K tokens (the size bench.py --mm times): sampled rows
    against the oracle, with the GPU's estimated lattice and index sets (the sets checked against
    the oracle's within the top-k band)."""
    N = 131072
    runs = [(0, 8192), (1, 98304), (0, 24576)]
    mod = _runs_modality(runs)
    rng = np.random.default_rng(17)
    # grid: a planted lattice, estimated, then attended
    x = I.grid_inputs(2, 1, N, 256, 37, seed=71)
    q, k, v = _dev(x)
    grid = B.mi_grid_estimate(q, k, 64, 1024)
    out = B.mi_grid_attn(q, k, v, grid, 64)
    torch.cuda.synchronize()
    assert grid.cpu().tolist() == [[256, 37]] * 2
    rows = np.unique(np.concatenate([sample_rows(N, rng, n_random=16, blocks=1), np.arange(37, N, 256)[:8]]))
    ref, _ = O.attention_rows(x.q[1], x.k[0], x.v[0], rows, lambda r: O.grid_mask_rows(N, r, 256, 37), chunk=32)
    assert_close(out[1][torch.as_tensor(rows, device=DEV)].float().cpu().numpy(), ref, "grid 128K")
    del x, q, k, v, out
    torch.cuda.empty_cache()
    # Q-boundary and 2D-boundary on literal inputs
    x = I.literal_inputs(2, 1, N, n_cols=8, n_offsets=4, seed=72)
    q, k, v = _dev(x)
    dmod = torch.as_tensor(mod, dtype=torch.int32, device=DEV)
    vi, si = B.mi_qboundary_estimate(q, k, dmod, 2, k_v=1000, k_s=6096)
    out = B.mi_qboundary_attn(q, k, v, dmod, 2, vi, si)
    torch.cuda.synchronize()
    vi_n, si_n = vi.cpu().numpy(), si.cpu().numpy()
    h = 1
    sets = []
    for m in (0, 1):
        vv, ss = O.window_estimate_scores(x.q[h], x.k[0], O.modality_row_end(mod, m), 64)
        band_agree(vi_n[m, h], O.topk_sorted(vv, 1000), vv, 1000)
        band_agree(si_n[m, h], O.topk_sorted(ss, 6096), ss, 6096)
        sets.append((vi_n[m, h][vi_n[m, h] >= 0], si_n[m, h][si_n[m, h] >= 0]))
    rows = sample_rows(N, rng, n_random=24, blocks=1)
    ref, _ = O.attention_rows(x.q[h], x.k[0], x.v[0], rows, lambda r: O.qboundary_mask_rows(N, r, mod, sets),
                              chunk=32)
    assert_close(out[h][torch.as_tensor(rows, device=DEV)].float().cpu().numpy(), ref, "q-boundary 128K")
    out2, vi2, si2 = B.mi_boundary2d_attn(q, k, v, runs, k_v=1000, k_s=6096)
    torch.cuda.synchronize()
    vi2_n, si2_n = vi2.cpu().numpy(), si2.cpu().numpy()
    sets2 = [(vi2_n[m, h][vi2_n[m, h] >= 0], si2_n[m, h][si2_n[m, h] >= 0]) for m in (0, 1)]
    idx1 = torch.as_tensor(np.nonzero(mod == 1)[0])
    vv, ss = O.vs_estimate_scores(x.q[h][idx1], x.k[0][idx1], 64)
    band_agree(vi2_n[1, h], O.topk_sorted(vv, 1000), vv, 1000)
    band_agree(si2_n[1, h], O.topk_sorted(ss, 6096), ss, 6096)
    ref, _ = O.attention_rows(x.q[h], x.k[0], x.v[0], rows, lambda r: O.boundary2d_mask_rows(N, r, mod, sets2),
                              chunk=32)
    assert_close(out2[h][torch.as_tensor(rows, device=DEV)].float().cpu().numpy(), ref, "2D-boundary 128K")
