"""Parity at the configurations' full sizes, in the launch configuration bench.py times.

The oracle cannot evaluate whole layers at 32K-1M tokens, so these tests check
exactly what it can compute one by one:
- every index set on margin-planted inputs (bit-exact);
- estimation of sampled heads on literal inputs (up to top-k boundary ties);
- the attention output of sampled rows (the first, the last and a random
  128-row block plus random rows) against the oracle's masked softmax, using
  the indices the GPU selected.
"""
import os
import sys

import numpy as np
import pytest
import torch

import oracle as O
from dynamic_sparse_attention_vertical_gb300 import binding as B
from dynamic_sparse_attention_vertical_gb300 import inputs as I
from tests.parity import assert_close, band_agree, sample_rows

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()
    yield
    torch.cuda.empty_cache()


def _free(*xs):
    for x in xs:
        del x
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _check_vs_rows(x, h, vi, si, rows, what):
    Hq, N = x.q.shape[0], x.q.shape[1]
    g = O.kv_head(h, Hq, x.k.shape[0])
    vi = vi[vi >= 0]
    si = si[si >= 0]
    return O.attention_rows(x.q[h], x.k[g], x.v[g], rows, lambda r: O.vs_mask_rows(N, r, vi, si), chunk=32)[0]


@pytest.mark.parametrize("N,k_v,k_s", [(32768, 1000, 6096), (131072, 1000, 6096), (16384, 500, 2048),
                                       (65536, 2000, 6096)])
def test_margin_planted_indices_exact_full_layer(N, k_v, k_s):
    """32 q / 8 KV heads: every head's index sets equal the planted sets bit for bit."""
    x = I.margin_inputs(32, 8, N, k_v, k_s, seed=N % 1000 + 102, device=DEV)
    v_idx, s_idx = B.mi_vs_estimate(x.q, x.k, k_v=k_v, k_s=k_s)
    vi, si = v_idx.cpu().numpy(), s_idx.cpu().numpy()
    for h in range(32):
        assert vi[h].tolist() == x.planted_cols[h // 4].tolist(), f"head {h}"
        assert si[h].tolist() == x.planted_offsets[h // 4].tolist(), f"head {h}"
    _free(x, v_idx, s_idx)


def test_margin_planted_indices_exact_1m():
    N = 1 << 20
    x = I.margin_inputs(32, 8, N, 1000, 6096, seed=104, device=DEV)
    v_idx, s_idx = B.mi_vs_estimate(x.q, x.k, k_v=1000, k_s=6096)
    vi, si = v_idx.cpu().numpy(), s_idx.cpu().numpy()
    for h in range(32):
        assert vi[h].tolist() == x.planted_cols[h // 4].tolist(), f"head {h}"
        assert si[h].tolist() == x.planted_offsets[h // 4].tolist(), f"head {h}"
    _free(x, v_idx, s_idx)


def _layer(workload):
    w = bench.WORKLOADS[workload]
    x = bench.make_inputs(w, "literal", torch.device(DEV))
    L = bench.Layer(B, w, x.q, x.k, x.v)
    L.step()
    torch.cuda.synchronize()
    L.check_status()
    return w, x, L


@pytest.mark.parametrize("workload,heads_checked", [("vs-32k", 3), ("vs-1m", 3)])
def test_vs_layer_sampled(workload, heads_checked):
    w, x, L = _layer(workload)
    N = w["N"]
    rng = np.random.default_rng(N)
    vi_all, si_all = L.v_idx.cpu().numpy(), L.s_idx.cpu().numpy()
    out = L.out
    for n in np.linspace(0, len(L.vs) - 1, heads_checked).astype(int):
        h = L.vs[n]
        g = O.kv_head(h, w["Hq"], w["Hkv"])
        vi_ref, si_ref, v, s = O.vs_estimate(x.q[h], x.k[g], 64, w["k_v"], w["k_s"])
        band_agree(vi_all[n], vi_ref, v, w["k_v"])
        band_agree(si_all[n], si_ref, s, w["k_s"])
        if N > 200000:  # the fp64 oracle costs N*d per row: a smaller sample at 1M (first rows,
            # the last 128-row block, one random block and random rows)
            b = int(rng.integers(1, N // 128 - 1))
            rows = np.unique(np.concatenate([np.arange(16), np.arange(N - 128, N), np.arange(128 * b, 128 * b + 128),
                                             rng.integers(0, N, 32)]))
        else:
            rows = sample_rows(N, rng, n_random=32, blocks=4)
        ref = _check_vs_rows(x, h, vi_all[n], si_all[n], rows, workload)
        got = out[h][torch.as_tensor(rows, device=DEV)].float().cpu().numpy()
        assert_close(got, ref, f"{workload} head {h}")
    _free(x, L)


def test_mixed_layer_128k_sampled():
    """The benchmark's default layer: 24 vertical-slash, 4 block-sparse, 4 A-shape heads."""
    w, x, L = _layer("mixed-128k")
    N = w["N"]
    rng = np.random.default_rng(7)
    out = L.out
    vi_all, si_all = L.v_idx.cpu().numpy(), L.s_idx.cpu().numpy()
    for n in (0, len(L.vs) - 1):
        h = L.vs[n]
        g = O.kv_head(h, w["Hq"], w["Hkv"])
        vi_ref, si_ref, v, s = O.vs_estimate(x.q[h], x.k[g], 64, w["k_v"], w["k_s"])
        band_agree(vi_all[n], vi_ref, v, w["k_v"])
        band_agree(si_all[n], si_ref, s, w["k_s"])
        rows = sample_rows(N, rng, n_random=32, blocks=2)
        ref = _check_vs_rows(x, h, vi_all[n], si_all[n], rows, "mixed vs")
        assert_close(out[h][torch.as_tensor(rows, device=DEV)].float().cpu().numpy(), ref, f"vs head {h}")
    bl = L.blk_idx.cpu().numpy()
    for n, h in enumerate(L.blk[:2]):
        g = O.kv_head(h, w["Hq"], w["Hkv"])
        sig = O.block_scores(x.q[h], x.k[g])
        for r in rng.integers(0, N // 64, size=64):
            got = bl[n, r][bl[n, r] >= 0]
            ref_sel = O.topk_sorted(sig[r, : r + 1], min(w["topk"], r + 1))
            band_agree(got, ref_sel, sig[r, : r + 1], min(w["topk"], r + 1), rel_band=1e-4)
        sel = [row[row >= 0] for row in bl[n]]
        rows = sample_rows(N, rng, n_random=32, blocks=2)
        ref, _ = O.attention_rows(x.q[h], x.k[g], x.v[g], rows,
                                  lambda r: O.block_sparse_mask_rows(N, r, sel), chunk=32)
        assert_close(out[h][torch.as_tensor(rows, device=DEV)].float().cpu().numpy(), ref, f"block head {h}")
    for h in L.ash[:2]:
        g = O.kv_head(h, w["Hq"], w["Hkv"])
        rows = sample_rows(N, rng, n_random=32, blocks=2)
        ref, _ = O.attention_rows(x.q[h], x.k[g], x.v[g], rows,
                                  lambda r: O.ashape_mask_rows(N, r, w["n_init"], w["window"]), chunk=32)
        assert_close(out[h][torch.as_tensor(rows, device=DEV)].float().cpu().numpy(), ref, f"ashape head {h}")
    _free(x, L)


@pytest.mark.parametrize("N,k_v,k_s", [(16384, 500, 2048), (65536, 2000, 6096), (131072, 1000, 2048),
                                       (262144, 2000, 6096), (524288, 500, 2048)])
def test_sweep_points_sampled(N, k_v, k_s):
    """Sweep points (one at every sweep length): one vertical-slash layer, sampled rows of
    one head, and our dense kernel on the same inputs."""
    x = I.literal_inputs(32, 8, N, n_cols=16, n_offsets=8, seed=5, device=DEV)
    v_idx, s_idx = B.mi_vs_estimate(x.q, x.k, k_v=k_v, k_s=k_s)
    out = B.mi_vs_sparse_attn(x.q, x.k, x.v, v_idx, s_idx)
    dense = B.mi_dense_causal_attn(x.q, x.k, x.v)
    torch.cuda.synchronize()
    h = 17
    vi, si = v_idx[h].cpu().numpy(), s_idx[h].cpu().numpy()
    rows = sample_rows(N, np.random.default_rng(N), n_random=32, blocks=2)
    ref = _check_vs_rows(x, h, vi, si, rows, "sweep")
    ridx = torch.as_tensor(rows, device=DEV)
    assert_close(out[h][ridx].float().cpu().numpy(), ref, f"sweep vs N={N}")
    g = O.kv_head(h, 32, 8)
    dref, _ = O.attention_rows(x.q[h], x.k[g], x.v[g], rows, lambda r: O.causal_mask_rows(N, r), chunk=32)
    assert_close(dense[h][ridx].float().cpu().numpy(), dref, f"sweep dense N={N}")
    _free(x, v_idx, s_idx, out, dense)


def test_vs_block_expanded_32k_sampled():
    """Block-expanded mode on a full 32K layer (32 q / 8 KV heads, estimated indices):
    sampled rows of three heads against the oracle's block-expanded mask."""
    N = 32768
    x = I.literal_inputs(32, 8, N, n_cols=16, n_offsets=8, seed=2, device=DEV)
    v_idx, s_idx = B.mi_vs_estimate(x.q, x.k, k_v=1000, k_s=6096)
    out = B.mi_vs_sparse_attn(x.q, x.k, x.v, v_idx, s_idx, expanded=True)
    torch.cuda.synchronize()
    vi_all, si_all = v_idx.cpu().numpy(), s_idx.cpu().numpy()
    rng = np.random.default_rng(9)
    for h in (0, 13, 31):
        g = O.kv_head(h, 32, 8)
        vi, si = vi_all[h][vi_all[h] >= 0], si_all[h][si_all[h] >= 0]
        rows = sample_rows(N, rng, n_random=32, blocks=2)
        ref, _ = O.attention_rows(x.q[h], x.k[g], x.v[g], rows,
                                  lambda r: O.vs_expanded_mask_rows(N, r, vi, si), chunk=32)
        assert_close(out[h][torch.as_tensor(rows, device=DEV)].float().cpu().numpy(), ref,
                     f"expanded head {h}")
    _free(x, v_idx, s_idx, out)


def test_largest_accepted_length_2m():
    """N = 2^21, the largest length the ABI accepts: margin-planted indices bit-exact,
    and sampled rows of the vertical-slash attention against the oracle."""
    N = 1 << 21
    x = I.margin_inputs(4, 1, N, 500, 2048, seed=211, device=DEV)
    v_idx, s_idx = B.mi_vs_estimate(x.q, x.k, k_v=500, k_s=2048)
    vi, si = v_idx.cpu().numpy(), s_idx.cpu().numpy()
    for h in range(4):
        assert vi[h].tolist() == x.planted_cols[0].tolist(), f"head {h}"
        assert si[h].tolist() == x.planted_offsets[0].tolist(), f"head {h}"
    out = B.mi_vs_sparse_attn(x.q, x.k, x.v, v_idx, s_idx, heads=[0])
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(8), np.arange(N - 8, N),
                                     np.random.default_rng(5).integers(0, N, 8)]))
    ref = _check_vs_rows(x, 0, vi[0], si[0], rows, "2m")
    assert_close(out[0][torch.as_tensor(rows, device=DEV)].float().cpu().numpy(), ref, "vs 2M head 0")
    _free(x, v_idx, s_idx, out)


def test_block_sparse_largest_topk_128k_sampled():
    """Block-sparse at the largest accepted top-k (MI_MAX_KV / 2 blocks per 64-row
    block) on 128K tokens: a late row block's two halves select up to 2048 blocks, so
    the CTA's list can hold every 128-key tile below the diagonal.  Sampled selections
    (up to ties at the top-k boundary) and sampled rows against the oracle."""
    N, Hq, Hkv, topk = 131072, 2, 1, B.MI_MAX_KV // 2
    x = I.literal_inputs(Hq, Hkv, N, n_cols=8, n_offsets=4, seed=91)
    q, k, v = x.q.to(DEV), x.k.to(DEV), x.v.to(DEV)
    out, blk = B.mi_block_sparse_attn(q, k, v, topk=topk)
    torch.cuda.synchronize()
    bl = blk.cpu().numpy()
    o = out.float().cpu().numpy()
    rng = np.random.default_rng(9)
    for h in range(Hq):
        sig = O.block_scores(x.q[h], x.k[0])
        for r in list(rng.integers(0, N // 64, size=24)) + [N // 64 - 1, N // 64 - 2]:
            got = bl[h, r][bl[h, r] >= 0]
            kk = min(topk, r + 1)
            band_agree(got, O.topk_sorted(sig[r, : r + 1], kk), sig[r, : r + 1], kk, rel_band=1e-4)
        sel = [row[row >= 0] for row in bl[h]]
        rows = sample_rows(N, rng, n_random=16, blocks=1)
        ref, _ = O.attention_rows(x.q[h], x.k[0], x.v[0], rows,
                                  lambda r: O.block_sparse_mask_rows(N, r, sel), chunk=32)
        assert_close(o[h][rows], ref, f"block head {h} topk {topk}")
    _free(x, q, k, v, out, blk)


@pytest.mark.parametrize("expanded", [False, True])
def test_vs_largest_vertical_budget_128k_sampled(expanded):
    """The largest accepted vertical budget (MI_MAX_KV columns) with 8192 diagonals on
    128K tokens: a late row block carries up to 16 gathered column tiles after its
    contiguous ones.  Sampled rows against the oracle with the selected indices."""
    N, Hq, Hkv = 131072, 2, 1
    k_v, k_s = B.MI_MAX_KV, 8192
    x = I.literal_inputs(Hq, Hkv, N, n_cols=24, n_offsets=8, seed=93)
    q, k, v = x.q.to(DEV), x.k.to(DEV), x.v.to(DEV)
    vi, si = B.mi_vs_estimate(q, k, k_v=k_v, k_s=k_s)
    out = B.mi_vs_sparse_attn(q, k, v, vi, si, expanded=expanded)
    torch.cuda.synchronize()
    vi_all, si_all = vi.cpu().numpy(), si.cpu().numpy()
    o = out.float().cpu().numpy()
    rng = np.random.default_rng(11)
    for h in range(Hq):
        rows = sample_rows(N, rng, n_random=16, blocks=1)
        vv, ss = vi_all[h][vi_all[h] >= 0], si_all[h][si_all[h] >= 0]
        mask = (lambda r: O.vs_expanded_mask_rows(N, r, vv, ss)) if expanded else \
            (lambda r: O.vs_mask_rows(N, r, vv, ss))
        ref, _ = O.attention_rows(x.q[h], x.k[0], x.v[0], rows, mask, chunk=32)
        assert_close(o[h][rows], ref, f"vs head {h} k_v {k_v} expanded {expanded}")
    _free(x, q, k, v, out, vi, si)
