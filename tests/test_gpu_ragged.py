"""GPU: lengths that are not a multiple of 64 (a partial last block of rows and keys),
down to a single token, for every call, against the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from dynamic_sparse_attention_vertical_gb300 import binding as B
from dynamic_sparse_attention_vertical_gb300 import inputs as I
from tests.parity import assert_close, band_agree

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def _inputs(Hq, Hkv, N, seed):
    x = I.literal_inputs(Hq, Hkv, N, n_cols=0, n_offsets=0, seed=seed)
    return x, x.q.to(DEV), x.k.to(DEV), x.v.to(DEV)


@pytest.mark.parametrize("N", [1, 17, 63, 100, 1000, 2111])
def test_dense_ashape_and_given_vs_at_ragged_lengths(N):
    Hq, Hkv = 2, 1
    x, q, k, v = _inputs(Hq, Hkv, N, seed=N + 3)
    rows = np.arange(N)
    dense = B.mi_dense_causal_attn(q, k, v).float().cpu().numpy()
    ash = B.mi_ashape_attn(q, k, v, n_init=5, window=40).float().cpu().numpy()
    vi = np.array(sorted({0, N // 3, N - 1}))
    si = np.array(sorted({0, min(1, N - 1), N // 2, N - 1}))
    v_idx = torch.tensor(np.stack([vi, vi]), dtype=torch.int32, device=DEV)
    s_idx = torch.tensor(np.stack([si, si]), dtype=torch.int32, device=DEV)
    vs = B.mi_vs_sparse_attn(q, k, v, v_idx, s_idx).float().cpu().numpy()
    for h in range(Hq):
        ref, _ = O.attention_rows(x.q[h], x.k[0], x.v[0], rows, lambda r: O.causal_mask_rows(N, r))
        assert_close(dense[h], ref, f"dense N={N}")
        ref, _ = O.attention_rows(x.q[h], x.k[0], x.v[0], rows, lambda r: O.ashape_mask_rows(N, r, 5, 40))
        assert_close(ash[h], ref, f"ashape N={N}")
        ref, _ = O.attention_rows(x.q[h], x.k[0], x.v[0], rows, lambda r: O.vs_mask_rows(N, r, vi, si))
        assert_close(vs[h], ref, f"vs given N={N}")


@pytest.mark.parametrize("N", [64, 65, 1000, 4097])
def test_estimate_and_vs_attention_at_ragged_lengths(N):
    Hq, Hkv = 2, 1
    x = I.literal_inputs(Hq, Hkv, N, n_cols=4, n_offsets=2, seed=N)
    q, k, v = x.q.to(DEV), x.k.to(DEV), x.v.to(DEV)
    v_idx, s_idx = B.mi_vs_estimate(q, k, k_v=40, k_s=30)
    out = B.mi_vs_sparse_attn(q, k, v, v_idx, s_idx).float().cpu().numpy()
    vi_all, si_all = v_idx.cpu().numpy(), s_idx.cpu().numpy()
    for h in range(Hq):
        vi_ref, si_ref, vsc, ssc = O.vs_estimate(x.q[h], x.k[0], 64, 40, 30)
        band_agree(vi_all[h], vi_ref, vsc, 40)
        band_agree(si_all[h], si_ref, ssc, 30)
        vi, si = vi_all[h][vi_all[h] >= 0], si_all[h][si_all[h] >= 0]
        ref, _ = O.attention_rows(x.q[h], x.k[0], x.v[0], np.arange(N), lambda r: O.vs_mask_rows(N, r, vi, si))
        assert_close(out[h], ref, f"vs N={N}")


def test_estimate_needs_64_rows():
    x, q, k, v = _inputs(1, 1, 63, seed=1)
    with pytest.raises(B.MIError) as e:
        B.mi_vs_estimate(q, k, k_v=4, k_s=4)
    assert e.value.code == B.MI_ERR_SHAPE


@pytest.mark.parametrize("N,topk", [(17, 4), (100, 2), (1000, 5), (2111, 8)])
def test_block_sparse_partial_last_block(N, topk):
    """The last 64-block holds N % 64 rows and keys: pooled as the mean of its rows,
    selectable, and its query rows get their own block lists."""
    Hq, Hkv = 2, 1
    planted = 4 if N > 256 else 0
    x = I.literal_inputs(Hq, Hkv, N, n_cols=planted, n_offsets=planted // 2, seed=N + 9)
    q, k, v = x.q.to(DEV), x.k.to(DEV), x.v.to(DEV)
    NB = (N + 63) // 64
    out, blk = B.mi_block_sparse_attn(q, k, v, topk=topk)
    assert tuple(blk.shape) == (Hq, NB, topk)
    bl = blk.cpu().numpy()
    o = out.float().cpu().numpy()
    for h in range(Hq):
        sig = O.block_scores(x.q[h], x.k[0])
        ref_sel = O.block_sparse_select(x.q[h], x.k[0], topk)
        assert sig.shape == (NB, NB)
        for r in range(NB):
            got = bl[h, r][bl[h, r] >= 0]
            band_agree(got, ref_sel[r], sig[r, : r + 1], min(topk, r + 1), rel_band=1e-3)
        sel = [row[row >= 0] for row in bl[h]]
        ref, _ = O.attention_rows(x.q[h], x.k[0], x.v[0], np.arange(N),
                                  lambda r: O.block_sparse_mask_rows(N, r, sel))
        assert_close(o[h], ref, f"block N={N}")


def test_layer_call_at_a_ragged_length():
    N, Hq, Hkv = 3001, 4, 2
    x = I.literal_inputs(Hq, Hkv, N, n_cols=8, n_offsets=4, seed=5, device=DEV)
    H = B.HeadCfg
    cfg = [H.vs(64, 32), H.block(8), H.ashape(128, 512), H.dense()]
    out = B.mi_layer_attn(x.q, x.k, x.v, cfg)
    ref = torch.zeros_like(x.q)
    vi, si = B.mi_vs_estimate(x.q, x.k, heads=[0], k_v=64, k_s=32)
    B.mi_vs_sparse_attn(x.q, x.k, x.v, vi, si, heads=[0], out=ref)
    B.mi_block_sparse_attn(x.q, x.k, x.v, topk=8, heads=[1], out=ref)
    B.mi_ashape_attn(x.q, x.k, x.v, n_init=128, window=512, heads=[2], out=ref)
    B.mi_dense_causal_attn(x.q, x.k, x.v, heads=[3], out=ref)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
