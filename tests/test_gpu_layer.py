"""GPU: the layer call (every head of every pattern in one attention launch)."""
import numpy as np
import pytest
import torch

import oracle as O
from dynamic_sparse_attention_vertical_gb300 import binding as B
from dynamic_sparse_attention_vertical_gb300 import inputs as I
from tests.parity import assert_close, sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
H = B.HeadCfg


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def _per_head(q, k, v, cfg):
    """The same layer through the per-pattern calls, one head at a time."""
    Hq, N, _ = q.shape
    out = torch.full_like(q, 3.0)
    lse = torch.full((Hq, N), float("nan"), device=DEV)
    for h, c in enumerate(cfg):
        if c.pattern == B.MI_PAT_DENSE:
            B.mi_dense_causal_attn(q, k, v, heads=[h], out=out, lse=lse)
        elif c.pattern == B.MI_PAT_VS:
            vi, si = B.mi_vs_estimate(q, k, heads=[h], k_v=c.k_v, k_s=c.k_s)
            B.mi_vs_sparse_attn(q, k, v, vi, si, heads=[h], out=out, lse=lse,
                                expanded=bool(c.vs_flags & B.MI_VS_BLOCK_EXPANDED))
        elif c.pattern == B.MI_PAT_BLOCK:
            B.mi_block_sparse_attn(q, k, v, topk=c.topk, heads=[h], out=out, lse=lse)
        elif c.pattern == B.MI_PAT_ASHAPE:
            B.mi_ashape_attn(q, k, v, n_init=c.n_init, window=c.window, heads=[h], out=out, lse=lse)
    return out, lse


@pytest.mark.parametrize("N,expanded", [(2048, False), (4160, False), (2048, True)])
def test_layer_call_equals_per_pattern_calls(N, expanded):
    """Mixed patterns and budgets (two vertical-slash groups, two block groups, two
    A-shape sizes, a dense head, a skipped head): outputs and log-sum-exps equal the
    per-pattern calls bit for bit; the skipped head's rows stay untouched."""
    Hq, Hkv = 8, 2
    x = I.literal_inputs(Hq, Hkv, N, n_cols=8, n_offsets=4, seed=N + 1, device=DEV)
    cfg = [H.vs(64, 32, expanded), H.block(8), H.ashape(128, 512), H.dense(),
           H.vs(128, 16, expanded), H.skip(), H.block(16), H.ashape(64, 1024)]
    out = torch.full_like(x.q, 3.0)
    lse = torch.full((Hq, N), float("nan"), device=DEV)
    B.mi_layer_attn(x.q, x.k, x.v, cfg, out=out, lse=lse)
    ref_out, ref_lse = _per_head(x.q, x.k, x.v, cfg)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    assert torch.equal(lse[[0, 1, 2, 3, 4, 6, 7]], ref_lse[[0, 1, 2, 3, 4, 6, 7]])
    assert bool((out[5] == 3.0).all()) and bool(torch.isnan(lse[5]).all())


def test_layer_call_matches_oracle_on_sampled_rows():
    N, Hq, Hkv = 4096, 4, 1
    x = I.literal_inputs(Hq, Hkv, N, n_cols=8, n_offsets=4, seed=17, device=DEV)
    cfg = [H.vs(64, 32), H.block(8), H.ashape(128, 1024), H.dense()]
    out = B.mi_layer_attn(x.q, x.k, x.v, cfg)
    torch.cuda.synchronize()
    xc = type(x)(x.q.cpu(), x.k.cpu(), x.v.cpu(), x.planted_cols, x.planted_offsets, x.seed, x.kind)
    rows = sample_rows(N, np.random.default_rng(3), n_random=32, blocks=2)
    vi, si = B.mi_vs_estimate(x.q, x.k, heads=[0], k_v=64, k_s=32)
    vi, si = vi[0].cpu().numpy(), si[0].cpu().numpy()
    _, bl = B.mi_block_sparse_attn(x.q, x.k, x.v, topk=8, heads=[1])
    sel = [r_[r_ >= 0] for r_ in bl[0].cpu().numpy()]
    masks = {0: lambda r: O.vs_mask_rows(N, r, vi[vi >= 0], si[si >= 0]),
             1: lambda r: O.block_sparse_mask_rows(N, r, sel),
             2: lambda r: O.ashape_mask_rows(N, r, 128, 1024),
             3: lambda r: O.causal_mask_rows(N, r)}
    got = out.float().cpu().numpy()
    for h in range(Hq):
        ref, _ = O.attention_rows(xc.q[h], xc.k[0], xc.v[0], rows, masks[h], chunk=64)
        assert_close(got[h][rows], ref, f"layer head {h}")


def test_layer_call_errors():
    N, Hq, Hkv = 1024, 2, 1
    x = I.literal_inputs(Hq, Hkv, N, n_cols=0, n_offsets=0, seed=2, device=DEV)
    with pytest.raises(ValueError):
        B.mi_layer_attn(x.q, x.k, x.v, [H.dense()])
    with pytest.raises(B.MIError) as e:
        B.mi_layer_attn(x.q, x.k, x.v, [H.dense(), B.HeadCfg(9, 0, 0, 0, 0, 0, 0)])
    assert e.value.code == B.MI_ERR_ARG
    with pytest.raises(B.MIError):
        B.mi_layer_attn(x.q, x.k, x.v, [H.vs(64, 16), H.vs(64, 16, expanded=True)])


def test_layer_call_replays_in_a_cuda_graph():
    """The layer call only enqueues stream work (no allocation, no host wait), so a
    caller can capture it once in a CUDA graph and replay it on new inputs in the
    same buffers: each replay equals a direct call on those inputs."""
    Hq, Hkv, N = 8, 2, 2048
    cfg = [H.vs(64, 32), H.block(8), H.ashape(128, 512), H.dense(),
           H.vs(128, 16), H.skip(), H.block(16), H.ashape(64, 1024)]
    xs = [I.literal_inputs(Hq, Hkv, N, n_cols=8, n_offsets=4, seed=s, device=DEV) for s in (71, 72)]
    q, k, v = xs[0].q.clone(), xs[0].k.clone(), xs[0].v.clone()
    out = torch.zeros_like(q)
    ws = torch.empty(B.mi_layer_workspace_bytes(Hq, Hkv, N, cfg), dtype=torch.uint8, device=DEV)
    B.mi_layer_attn(q, k, v, cfg, out=out, workspace=ws)  # first-call setup outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.mi_layer_attn(q, k, v, cfg, out=out, workspace=ws)
    for x in (xs[1], xs[0], xs[1]):
        q.copy_(x.q)
        k.copy_(x.k)
        v.copy_(x.v)
        g.replay()
        ref = torch.zeros_like(q)
        B.mi_layer_attn(x.q, x.k, x.v, cfg, out=ref)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
