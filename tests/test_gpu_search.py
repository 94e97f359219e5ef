"""GPU: the kernel-aware pattern search measures recall correctly and recovers planted head types."""
import numpy as np
import pytest
import torch

import oracle as O
from dynamic_sparse_attention_vertical_gb300 import binding as B
from dynamic_sparse_attention_vertical_gb300 import inputs as I
from dynamic_sparse_attention_vertical_gb300 import search as S

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def _kept_mass(x, h, N, mask_rows):
    """Oracle: mean over rows of the causal softmax mass on the kept keys."""
    qh, kh = O.as_f64(x.q[h]), O.as_f64(x.k[h])
    rows = np.arange(N)
    logits = (qh @ kh.T) / np.sqrt(qh.shape[1])
    logits = np.where(O.causal_mask_rows(N, rows), logits, -np.inf)
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return (p * mask_rows(rows)).sum(axis=1).mean()


def test_recall_from_lse_equals_oracle_kept_mass():
    N = 2048
    x = I.pattern_head_inputs(N, seed=3, window=256, offsets=(300, 900))
    q, k, v = x.q.to(DEV), x.k.to(DEV), x.v.to(DEV)
    heads = [0, 1, 2]
    lse_d = torch.empty((3, N), dtype=torch.float32, device=DEV)
    B.mi_dense_causal_attn(q, k, v, lse=lse_d)
    for cand in (S.Candidate.make("ashape", n_init=128, window=512), S.Candidate.make("vs", k_v=64, k_s=16),
                 S.Candidate.make("block", topk=8)):
        lse_c = torch.empty_like(lse_d)
        out = torch.empty_like(q)
        if cand.pattern == "ashape":
            B.mi_ashape_attn(q, k, v, n_init=128, window=512, out=out, lse=lse_c)
            masks = [lambda r: O.ashape_mask_rows(N, r, 128, 512)] * 3
        elif cand.pattern == "vs":
            vi, si = B.mi_vs_estimate(q, k, k_v=64, k_s=16)
            B.mi_vs_sparse_attn(q, k, v, vi, si, out=out, lse=lse_c)
            vi, si = vi.cpu().numpy(), si.cpu().numpy()
            masks = [lambda r, a=vi[h][vi[h] >= 0], b=si[h][si[h] >= 0]: O.vs_mask_rows(N, r, a, b)
                     for h in heads]
        else:
            _, bl = B.mi_block_sparse_attn(q, k, v, topk=8, out=out, lse=lse_c)
            bl = bl.cpu().numpy()
            masks = [lambda r, s=[row[row >= 0] for row in bl[h]]: O.block_sparse_mask_rows(N, r, s)
                     for h in heads]
        got = torch.exp(lse_c - lse_d).double().mean(dim=1).cpu().numpy()
        for h in heads:
            want = _kept_mass(x, h, N, masks[h])
            assert abs(got[h] - want) < 2e-3, (str(cand), h, got[h], want)


def test_search_recovers_planted_pattern_types():
    """Head 0 is a sink + local-window head, head 1 a vertical-slash head, head 2 a
    block-topic head: the search must give head 1 a vertical-slash pattern and head 2
    a block-sparse one; head 0 must be covered almost fully by a pattern that is not
    vertical-slash (A-shape or blocks both fit a sink plus a window)."""
    N = 32768
    x = I.pattern_head_inputs(N, seed=5, device=DEV)
    choices = S.search(x.q, x.k, x.v, budget_frac=0.4, reps=2)
    by_head = {c.head: c for c in choices}
    table = {c.head: [(str(e.candidate), round(e.recall, 4), round(e.cost_ms, 4)) for e in c.evaluations]
             + [("dense", 1.0, round(c.dense_ms, 4))] for c in choices}
    for c in choices:
        assert c.choice.cost_ms <= c.budget_ms, table
    assert by_head[1].choice.candidate.pattern == "vs", table[1]
    assert by_head[2].choice.candidate.pattern == "block", table[2]
    assert by_head[0].choice.candidate.pattern in ("ashape", "block"), table[0]
    assert by_head[0].choice.recall > 0.99
    assert by_head[1].choice.recall > 0.8 and by_head[2].choice.recall > 0.7
    # the choice is the best recall in the budget for every head
    for c in choices:
        fit = [e.recall for e in c.evaluations if e.cost_ms <= c.budget_ms]
        assert c.choice.recall >= max(fit) - 0.005
    # the chosen configuration runs as one layer call and keeps the recall it was chosen for
    cfg = S.layer_config(choices, 3)
    lse_d = torch.empty((3, N), dtype=torch.float32, device=DEV)
    lse = torch.empty_like(lse_d)
    B.mi_dense_causal_attn(x.q, x.k, x.v, lse=lse_d)
    B.mi_layer_attn(x.q, x.k, x.v, cfg, lse=lse)
    got = torch.exp(lse - lse_d).double().mean(dim=1).cpu().numpy()
    for c in choices:
        assert abs(got[c.head] - c.choice.recall) < 1e-6
