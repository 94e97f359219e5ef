"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Outputs: max-abs <= 2e-2, mean-abs <= 2e-3 and relative Frobenius <= 1e-2 per
head, bf16 GPU against the fp64 oracle.  Indices: bit-exact on margin-planted
inputs; elsewhere equal up to elements scoring at the top-k boundary.
"""
import numpy as np
import pytest
import torch

import oracle as O
from dynamic_sparse_attention_vertical_gb300 import binding as B
from dynamic_sparse_attention_vertical_gb300 import inputs as I
from tests.parity import REL_FRO, assert_close, band_agree, rel_fro

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def _dev(x):
    return x.q.to(DEV), x.k.to(DEV), x.v.to(DEV)


def _rand_inputs(Hq, Hkv, N, seed):
    return I.literal_inputs(Hq, Hkv, N, n_cols=0, n_offsets=0, seed=seed)


# ----------------------------------------------------------------- dense ----

@pytest.mark.parametrize("N", [128, 320, 1024])
def test_dense_matches_oracle(N):
    Hq, Hkv = 2, 1
    x = _rand_inputs(Hq, Hkv, N, seed=N)
    q, k, v = _dev(x)
    lse = torch.full((Hq, N), float("nan"), device=DEV)
    out = B.mi_dense_causal_attn(q, k, v, lse=lse)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    rows = np.arange(N)
    for h in range(Hq):
        g = O.kv_head(h, Hq, Hkv)
        ref, rl = O.attention_rows(x.q[h], x.k[g], x.v[g], rows,
                                   lambda r: O.causal_mask_rows(N, r))
        assert_close(o[h], ref, f"dense h{h}")
        assert np.abs(l[h] - rl).max() < 1e-3


def test_dense_writes_only_listed_heads():
    Hq, Hkv, N = 4, 2, 256
    x = _rand_inputs(Hq, Hkv, N, seed=3)
    q, k, v = _dev(x)
    out = torch.full_like(q, 7.0)
    B.mi_dense_causal_attn(q, k, v, heads=[3, 0], out=out)
    o = out.float().cpu().numpy()
    assert np.all(o[1] == 7.0) and np.all(o[2] == 7.0)
    for h in (3, 0):
        g = O.kv_head(h, Hq, Hkv)
        ref, _ = O.attention_rows(x.q[h], x.k[g], x.v[g], np.arange(N),
                                  lambda r: O.causal_mask_rows(N, r))
        assert_close(o[h], ref, f"dense subset h{h}")


# --------------------------------------------------------------- A-shape ----

@pytest.mark.parametrize("N,n_init,window",
                         [(640, 128, 256), (2048, 100, 300), (1024, 0, 1), (512, 64, 4096)])
def test_ashape_matches_oracle(N, n_init, window):
    Hq, Hkv = 2, 2
    x = _rand_inputs(Hq, Hkv, N, seed=N + window)
    q, k, v = _dev(x)
    out = B.mi_ashape_attn(q, k, v, n_init=n_init, window=window)
    o = out.float().cpu().numpy()
    for h in range(Hq):
        ref, _ = O.attention_rows(x.q[h], x.k[h], x.v[h], np.arange(N),
                                  lambda r: O.ashape_mask_rows(N, r, n_init, window))
        assert_close(o[h], ref, f"ashape h{h}")
    if n_init == 0 and window == 1:  # every row keeps only itself
        assert torch.equal(out.cpu(), x.v)


# ------------------------------------------------------- vertical-slash ----

def _vs_check(x, heads, v_idx, s_idx, out, rows=None):
    Hq, N = x.q.shape[0], x.q.shape[1]
    Hkv = x.k.shape[0]
    o = out.float().cpu().numpy()
    rows = np.arange(N) if rows is None else rows
    for n, h in enumerate(heads):
        g = O.kv_head(h, Hq, Hkv)
        vi = np.asarray(v_idx[n])
        vi = vi[vi >= 0]
        si = np.asarray(s_idx[n])
        si = si[si >= 0]
        ref, _ = O.attention_rows(x.q[h], x.k[g], x.v[g], rows,
                                  lambda r: O.vs_mask_rows(N, r, vi, si))
        assert_close(o[h][rows], ref, f"vs h{h}")


@pytest.mark.parametrize("N", [2112, 4096])
def test_vs_attention_with_oracle_indices(N):
    Hq, Hkv = 2, 1
    x = I.literal_inputs(Hq, Hkv, N, n_cols=8, n_offsets=4, seed=N)
    vis, sis = [], []
    for h in range(Hq):
        vi, si, _, _ = O.vs_estimate(x.q[h], x.k[0], 64, 64, 32)
        vis.append(vi)
        sis.append(si)
    q, k, v = _dev(x)
    v_idx = torch.tensor(np.stack(vis), dtype=torch.int32, device=DEV)
    s_idx = torch.tensor(np.stack(sis), dtype=torch.int32, device=DEV)
    out = B.mi_vs_sparse_attn(q, k, v, v_idx, s_idx)
    _vs_check(x, range(Hq), vis, sis, out)


def test_vs_attention_gathered_columns():
    """Many columns outside the diagonal tiles: several gathered column tiles per block."""
    N, Hq, Hkv = 4096, 2, 1
    x = _rand_inputs(Hq, Hkv, N, seed=11)
    rng = np.random.default_rng(5)
    vis = [np.sort(rng.choice(np.arange(N), size=300, replace=False)) for _ in range(Hq)]
    sis = [np.array([5, 700, 2000]), np.array([0, 1, 2, 3, 129, 4000])]
    q, k, v = _dev(x)
    v_idx = torch.tensor(np.stack(vis), dtype=torch.int32, device=DEV)
    s_idx = torch.full((Hq, 6), -1, dtype=torch.int32)
    for h in range(Hq):
        s_idx[h, : len(sis[h])] = torch.tensor(sis[h])
    out = B.mi_vs_sparse_attn(q, k, v, v_idx, s_idx.to(DEV))
    _vs_check(x, range(Hq), vis, sis, out)


def _vs_expanded_check(x, heads, v_idx, s_idx, out, rows=None):
    Hq, N = x.q.shape[0], x.q.shape[1]
    Hkv = x.k.shape[0]
    o = out.float().cpu().numpy()
    rows = np.arange(N) if rows is None else rows
    for n, h in enumerate(heads):
        g = O.kv_head(h, Hq, Hkv)
        vi = np.asarray(v_idx[n])
        vi = vi[vi >= 0]
        si = np.asarray(s_idx[n])
        si = si[si >= 0]
        ref, _ = O.attention_rows(x.q[h], x.k[g], x.v[g], rows,
                                  lambda r: O.vs_expanded_mask_rows(N, r, vi, si))
        assert_close(o[h][rows], ref, f"vs expanded h{h}")


@pytest.mark.parametrize("N,seed", [(1024, 21), (2112, 22), (4096, 23)])
def test_vs_block_expanded_matches_oracle(N, seed):
    """Block-expanded diagonals: sparse offsets (partial tiles, the 64x64 sub-block
    mask), runs of offsets (tiles kept whole), offset 0 and the last offset,
    columns inside and outside the covered tiles (gathered tiles)."""
    Hq, Hkv = 3, 1
    x = _rand_inputs(Hq, Hkv, N, seed=seed)
    rng = np.random.default_rng(seed)
    sis = [np.array(sorted({0, 70, 300, N // 2 + 5, N - 1})),
           np.arange(200, 520),                                    # a run: whole tiles
           np.sort(rng.choice(np.arange(N), size=40, replace=False))]
    vis = [np.sort(rng.choice(np.arange(N), size=k, replace=False)) for k in (10, 200, 130)]
    k_s = max(len(si) for si in sis)
    k_v = max(len(vi) for vi in vis)
    s_idx = torch.full((Hq, k_s), -1, dtype=torch.int32)
    v_idx = torch.full((Hq, k_v), -1, dtype=torch.int32)
    for h in range(Hq):
        s_idx[h, : len(sis[h])] = torch.tensor(sis[h])
        v_idx[h, : len(vis[h])] = torch.tensor(vis[h])
    q, k, v = _dev(x)
    out = B.mi_vs_sparse_attn(q, k, v, v_idx.to(DEV), s_idx.to(DEV), expanded=True)
    _vs_expanded_check(x, range(Hq), vis, sis, out)


def test_vs_block_expanded_estimated_indices_and_exact_differ():
    """With estimated indices the expanded mode keeps a superset of the exact mask:
    both match their own oracle mask, and on these inputs they differ."""
    N, Hq, Hkv = 2048, 2, 1
    x = I.literal_inputs(Hq, Hkv, N, n_cols=8, n_offsets=4, seed=31)
    q, k, v = _dev(x)
    v_idx, s_idx = B.mi_vs_estimate(q, k, k_v=64, k_s=32)
    exp = B.mi_vs_sparse_attn(q, k, v, v_idx, s_idx, expanded=True)
    ex = B.mi_vs_sparse_attn(q, k, v, v_idx, s_idx)
    vi, si = v_idx.cpu().numpy(), s_idx.cpu().numpy()
    _vs_expanded_check(x, range(Hq), vi, si, exp)
    _vs_check(x, range(Hq), vi, si, ex)
    assert (exp.float() - ex.float()).abs().max().item() > 1e-3


def test_vs_unknown_flag_is_refused():
    N, Hq, Hkv = 256, 1, 1
    x = _rand_inputs(Hq, Hkv, N, seed=4)
    q, k, v = _dev(x)
    v_idx = torch.tensor([[3]], dtype=torch.int32, device=DEV)
    s_idx = torch.tensor([[5]], dtype=torch.int32, device=DEV)
    out = torch.zeros_like(q)
    ws = torch.empty(B.mi_workspace_bytes(B.MI_OP_VS_SPARSE_ATTN, 1, Hkv, N), dtype=torch.uint8, device=DEV)
    lib = B.load()
    rc = lib.mi_vs_sparse_attn(q.data_ptr(), k.data_ptr(), v.data_ptr(), Hq, Hkv, N, 128, None, 1,
                               v_idx.data_ptr(), 1, s_idx.data_ptr(), 1, 2, out.data_ptr(), None,
                               ws.data_ptr(), ws.numel(), None)
    assert rc == B.MI_ERR_UNIMPLEMENTED


def test_vs_full_budget_is_dense():
    N, Hq, Hkv = 384, 1, 1
    x = _rand_inputs(Hq, Hkv, N, seed=2)
    q, k, v = _dev(x)
    v_idx, s_idx = B.mi_vs_estimate(q, k, k_v=N, k_s=N)
    assert v_idx.cpu().tolist() == [list(range(N))] and s_idx.cpu().tolist() == [list(range(N))]
    out = B.mi_vs_sparse_attn(q, k, v, v_idx, s_idx)
    dense = B.mi_dense_causal_attn(q, k, v)
    ref, _ = O.attention_rows(x.q[0], x.k[0], x.v[0], np.arange(N),
                              lambda r: O.causal_mask_rows(N, r))
    assert_close(out.float().cpu().numpy()[0], ref, "vs full budget")
    assert_close(dense.float().cpu().numpy()[0], ref, "dense")


@pytest.mark.parametrize("Hq,Hkv,N,k_v,k_s",
                         [(4, 2, 2048, 64, 32), (2, 1, 4160, 100, 50), (1, 1, 4096, 64, 32)])
def test_vs_estimate_margin_planted_exact(Hq, Hkv, N, k_v, k_s):
    x = I.margin_inputs(Hq, Hkv, N, k_v, k_s, seed=N + k_v)
    q, k, _ = _dev(x)
    v_idx, s_idx = B.mi_vs_estimate(q, k, k_v=k_v, k_s=k_s)
    vi, si = v_idx.cpu().numpy(), s_idx.cpu().numpy()
    for h in range(Hq):
        g = O.kv_head(h, Hq, Hkv)
        assert vi[h].tolist() == x.planted_cols[g].tolist()
        assert si[h].tolist() == x.planted_offsets[g].tolist()


def test_vs_estimate_literal_band():
    """The single-head 4K configuration: planted indices found, the rest up to boundary ties."""
    N = 4096
    x = I.literal_inputs(1, 1, N, n_cols=8, n_offsets=4, seed=1)
    q, k, _ = _dev(x)
    v_idx, s_idx = B.mi_vs_estimate(q, k, k_v=64, k_s=32)
    vi_ref, si_ref, v, s = O.vs_estimate(x.q[0], x.k[0], 64, 64, 32)
    # literal planting does not force every planted index into the top-k (the
    # oracle ranks some planted columns in the hundreds); the ones the oracle
    # keeps must be kept by the GPU too
    pc = [c for c in x.planted_cols[0].tolist() if c in set(vi_ref.tolist())]
    po = [o for o in x.planted_offsets[0].tolist() if o in set(si_ref.tolist())]
    assert len(po) == len(x.planted_offsets[0])  # planted diagonals do rank first here
    band_agree(v_idx.cpu().numpy()[0], vi_ref, v, 64, must_have=pc)
    band_agree(s_idx.cpu().numpy()[0], si_ref, s, 32, must_have=po)


def test_vs_estimate_budget_edges():
    N = 256
    x = _rand_inputs(2, 1, N, seed=9)
    q, k, _ = _dev(x)
    v_idx, s_idx = B.mi_vs_estimate(q, k, k_v=0, k_s=5)
    assert v_idx.shape == (2, 0) and s_idx.shape == (2, 5)
    v_idx, s_idx = B.mi_vs_estimate(q, k, k_v=N + 10, k_s=3)
    vi = v_idx.cpu().numpy()
    assert vi[:, :N].tolist() == [list(range(N))] * 2 and np.all(vi[:, N:] == -1)
    for h in range(2):
        _, si_ref, _, s = O.vs_estimate(x.q[h], x.k[0], 64, 0, 3)
        band_agree(s_idx.cpu().numpy()[h], si_ref, s, 3)


def test_vs_end_to_end_and_mutation():
    """Estimate + attention; removing one selected column must break the tolerance."""
    N, Hq, Hkv = 4096, 2, 1
    x = I.literal_inputs(Hq, Hkv, N, n_cols=8, n_offsets=4, seed=21)
    g = torch.Generator().manual_seed(77)
    x.v = torch.randn(x.v.shape, generator=g).to(torch.bfloat16)  # V ~ N(0, 1)
    q, k, v = _dev(x)
    v_idx, s_idx = B.mi_vs_estimate(q, k, k_v=64, k_s=32)
    out = B.mi_vs_sparse_attn(q, k, v, v_idx, s_idx)
    vi, si = v_idx.cpu().numpy(), s_idx.cpu().numpy()
    _vs_check(x, range(Hq), vi, si, out)
    # mutation: drop a planted column from head 0's list
    col = int(x.planted_cols[0][0])
    keep = vi[0][vi[0] != col]
    assert len(keep) == len(vi[0]) - 1
    mut = torch.full_like(v_idx[:1], -1)
    mut[0, : len(keep)] = torch.tensor(keep, dtype=torch.int32, device=DEV)
    out_m = B.mi_vs_sparse_attn(q, k, v, mut, s_idx[:1].contiguous(), heads=[0])
    rows = np.arange(((col // 128) + 1) * 128, N)
    ref, _ = O.attention_rows(x.q[0], x.k[0], x.v[0], rows,
                              lambda r: O.vs_mask_rows(N, r, vi[0], si[0]))
    assert rel_fro(out_m.float().cpu().numpy()[0][rows], ref) > REL_FRO


# ----------------------------------------------------------- block-sparse ----

def test_block_sparse_select_and_attention():
    N, Hq, Hkv, topk = 2048, 2, 1, 8
    x = I.literal_inputs(Hq, Hkv, N, n_cols=4, n_offsets=2, seed=31)
    q, k, v = _dev(x)
    out, blk = B.mi_block_sparse_attn(q, k, v, topk=topk)
    bl = blk.cpu().numpy()
    o = out.float().cpu().numpy()
    for h in range(Hq):
        sig = O.block_scores(x.q[h], x.k[0])
        ref_sel = O.block_sparse_select(x.q[h], x.k[0], topk)
        for r in range(N // 64):
            got = bl[h, r][bl[h, r] >= 0]
            assert np.all(np.diff(got) > 0) and got.max() <= r
            band_agree(got, ref_sel[r], sig[r, : r + 1], min(topk, r + 1), rel_band=1e-4)
        sel = [row[row >= 0] for row in bl[h]]
        ref, _ = O.attention_rows(x.q[h], x.k[0], x.v[0], np.arange(N),
                                  lambda r: O.block_sparse_mask_rows(N, r, sel))
        assert_close(o[h], ref, f"block h{h}")
    # the same with the oracle's own selection passed in
    given = np.full((Hq, N // 64, topk), -1, dtype=np.int32)
    refs = []
    for h in range(Hq):
        ref_sel = O.block_sparse_select(x.q[h], x.k[0], topk)
        refs.append(ref_sel)
        for r, s in enumerate(ref_sel):
            given[h, r, : len(s)] = s
    out2, _ = B.mi_block_sparse_attn(q, k, v, topk=topk, blk_idx=torch.tensor(given, device=DEV),
                                     given=True)
    for h in range(Hq):
        ref, _ = O.attention_rows(x.q[h], x.k[0], x.v[0], np.arange(N),
                                  lambda r: O.block_sparse_mask_rows(N, r, refs[h]))
        assert_close(out2.float().cpu().numpy()[h], ref, f"block given h{h}")


def test_block_select_many_candidates():
    """Up to 256 candidate blocks per query block and top-100, against the oracle's ranking."""
    N, Hq, Hkv, topk = 16384, 1, 1, 100
    x = I.literal_inputs(Hq, Hkv, N, n_cols=4, n_offsets=2, seed=41)
    q, k, v = _dev(x)
    _, blk = B.mi_block_sparse_attn(q, k, v, topk=topk)
    bl = blk.cpu().numpy()[0]
    sig = O.block_scores(x.q[0], x.k[0])
    ref_sel = O.block_sparse_select(x.q[0], x.k[0], topk)
    diffs = 0
    for r in range(N // 64):
        got = bl[r][bl[r] >= 0]
        assert len(got) == min(topk, r + 1) and np.all(np.diff(got) > 0) and got.max() <= r
        assert np.all(bl[r][len(got):] == -1)
        diffs += band_agree(got, ref_sel[r], sig[r, : r + 1], min(topk, r + 1), rel_band=1e-4)
    assert diffs <= N // 64  # near-ties only


# ----------------------------------------------------------------- errors ----

def test_argument_and_index_errors():
    N = 256
    x = _rand_inputs(2, 1, N, seed=4)
    q, k, v = _dev(x)
    # a length beyond 2^21 is refused before any work (the tensors are not read)
    out = torch.empty_like(q)
    ws0 = torch.empty(256, dtype=torch.uint8, device=DEV)
    rc = B.load().mi_dense_causal_attn(q.data_ptr(), k.data_ptr(), v.data_ptr(), 2, 1, (1 << 21) + 64, 128,
                                       None, 2, out.data_ptr(), None, ws0.data_ptr(), 256, None)
    assert rc == B.MI_ERR_SHAPE
    with pytest.raises(B.MIError) as e:
        B.mi_dense_causal_attn(q, k, v, heads=[0, 0])
    assert e.value.code == B.MI_ERR_ARG
    ws = torch.empty(1024, dtype=torch.uint8, device=DEV)
    with pytest.raises(B.MIError) as e:
        B.mi_dense_causal_attn(q, k, v, workspace=ws[1:257])
    assert e.value.code == B.MI_ERR_WORKSPACE
    # unsorted / out-of-range indices: reported through the status word, no fault
    bad_v = torch.tensor([[5, 3, 9], [1, 2, 3]], dtype=torch.int32, device=DEV)
    s_idx = torch.tensor([[0, 7], [1, N + 5]], dtype=torch.int32, device=DEV)
    ws = torch.empty(B.mi_workspace_bytes(B.MI_OP_VS_SPARSE_ATTN, 2, 1, N), dtype=torch.uint8,
                     device=DEV)
    B.mi_vs_sparse_attn(q, k, v, bad_v, s_idx, workspace=ws)
    assert B.mi_read_status(ws) == B.MI_ERR_INDEX
    good_v = torch.tensor([[3, 5, 9], [1, 2, 3]], dtype=torch.int32, device=DEV)
    good_s = torch.tensor([[0, 7], [1, -1]], dtype=torch.int32, device=DEV)
    B.mi_vs_sparse_attn(q, k, v, good_v, good_s, workspace=ws)
    assert B.mi_read_status(ws) == B.MI_OK


def test_bounded_wait_expiry_reports_timeout():
    """A wait that nothing completes expires, the call reports MI_ERR_TIMEOUT, the context stays usable."""
    N = 256
    x = _rand_inputs(2, 1, N, seed=12)
    q, k, v = _dev(x)
    ws = torch.empty(256, dtype=torch.uint8, device=DEV)
    assert B.mi_debug_inject(B.MI_FAULT_SKIP_Q_LOAD, 2_000_000) == B.MI_OK  # 2 ms
    try:
        B.mi_dense_causal_attn(q, k, v, workspace=ws)
        assert B.mi_read_status(ws) == B.MI_ERR_TIMEOUT
    finally:
        assert B.mi_debug_inject(B.MI_FAULT_NONE) == B.MI_OK
    out = B.mi_dense_causal_attn(q, k, v, workspace=ws)
    assert B.mi_read_status(ws) == B.MI_OK
    ref, _ = O.attention_rows(x.q[0], x.k[0], x.v[0], np.arange(N), lambda r: O.causal_mask_rows(N, r))
    assert_close(out.float().cpu().numpy()[0], ref, "after timeout")


@pytest.mark.parametrize("where", ["spread", "first_half", "second_half"])
def test_topk_ties_across_the_pair_halves(where):
    """1500 identical key rows along the direction of the last 64 queries: their
    vertical scores tie exactly (the same column sums in the same order) and lie
    far above every other column, so the top 1000 are the 1000 lowest-indexed of
    them.  Each score row is selected by two CTAs, one per half of the row (the
    boundary is N / 2 here): spread over both halves, the tied keys taken make
    the second CTA's output start after the first's, and the tie cut falls in the
    second half; in one half, the other CTA holds no tied key."""
    N, Hq, Hkv, d = 32768, 2, 1, 128
    g = torch.Generator().manual_seed(17)
    rng = np.random.default_rng(17)
    lo, hi = {"spread": (0, N - 64), "first_half": (0, N // 2), "second_half": (N // 2, N - 64)}[where]
    T = np.sort(rng.choice(np.arange(lo, hi), size=1500, replace=False))
    u = torch.randn(d, generator=g)
    u = u / u.norm()
    k = torch.randn(Hkv, N, d, generator=g)
    k[0, torch.from_numpy(T)] = 16.0 * u
    q = torch.randn(Hq, N, d, generator=g)
    q[:, N - 64:] = 16.0 * u + 0.01 * torch.randn(Hq, 64, d, generator=g)
    q, k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    v_idx, s_idx = B.mi_vs_estimate(q.to(DEV), k.to(DEV), k_v=1000, k_s=256)
    want = T[:1000]
    for h in range(Hq):
        vi_ref, si_ref, _, sc = O.vs_estimate(q[h], k[0], 64, 1000, 256)
        assert vi_ref.tolist() == want.tolist()  # the construction, checked on the oracle
        assert v_idx[h].cpu().tolist() == want.tolist()
        band_agree(s_idx[h].cpu().numpy(), si_ref, sc, 256)


def test_estimate_all_ties_takes_lowest_indices():
    """Zero queries: every query weighs its keys uniformly, so the column scores tie
    (each column summed over the same rows in the same order) and the selection must
    keep the lowest indices, also at large N where the sampled-threshold path sees
    every score reach the threshold and the full selection runs.  The slash scores
    also tie in exact arithmetic, but the GPU sums each diagonal in fp32 across tiles
    in its own order, so they are compared with the tie band."""
    N, Hq, Hkv = 32768, 2, 1
    x = _rand_inputs(Hq, Hkv, N, seed=6)
    q = torch.zeros_like(x.q).to(DEV)
    k = x.k.to(DEV)
    v_idx, s_idx = B.mi_vs_estimate(q, k, k_v=1000, k_s=2048)
    for h in range(Hq):
        vi_ref, si_ref, _, sc = O.vs_estimate(torch.zeros_like(x.q[h]), x.k[0], 64, 1000, 2048)
        assert v_idx[h].cpu().tolist() == vi_ref.tolist()
        band_agree(s_idx[h].cpu().numpy(), si_ref, sc, 2048)
