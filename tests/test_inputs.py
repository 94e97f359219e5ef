"""Seeded input generators: determinism, shapes and planted ranges (no GPU)."""
import torch

from dynamic_sparse_attention_vertical_gb300 import inputs as I


def test_literal_is_seeded_and_shaped():
    a = I.literal_inputs(4, 2, 512, n_cols=8, n_offsets=4, seed=3)
    b = I.literal_inputs(4, 2, 512, n_cols=8, n_offsets=4, seed=3)
    c = I.literal_inputs(4, 2, 512, n_cols=8, n_offsets=4, seed=4)
    assert a.q.shape == (4, 512, 128) and a.k.shape == (2, 512, 128) and a.q.dtype == torch.bfloat16
    assert torch.equal(a.q, b.q) and torch.equal(a.k, b.k) and torch.equal(a.v, b.v)
    assert not torch.equal(a.q, c.q)
    for g in range(2):
        cols, offs = a.planted_cols[g], a.planted_offsets[g]
        assert len(cols) == 8 and len(offs) == 4
        assert cols.min() >= 64 and cols.max() < 512 - 64
        assert offs.min() >= 64 and offs.max() <= 512 - 64
        assert torch.all(cols[1:] > cols[:-1]) and torch.all(offs[1:] > offs[:-1])


def test_literal_column_is_visible_in_keys():
    x = I.literal_inputs(1, 1, 1024, n_cols=4, n_offsets=0, seed=5)
    norms = x.k[0].float().norm(dim=1)
    planted = norms[x.planted_cols[0]]
    assert planted.min() > 2.0 * norms.median()   # K[c] += 4u makes planted rows stand out


def test_margin_inputs_structure():
    x = I.margin_inputs(2, 1, 512, k_v=5, k_s=7, seed=2)
    lastq = x.q[0, -64:, :64].float()
    assert torch.equal(lastq, 8.0 * torch.eye(64))
    assert torch.all(x.q[0, -64:, 64:] == 0)
    assert len(x.planted_cols[0]) == 5 and len(x.planted_offsets[0]) == 7
    assert x.planted_offsets[0].max() <= 512 - 64


def test_local_inputs_rotary_pair():
    x = I.local_inputs(2, 1, 256, n_cols=2, n_offsets=1, seed=1)
    r = x.q[0, :, 126:].float().norm(dim=1)
    assert torch.allclose(r, r[0].expand_as(r), rtol=2e-2)
