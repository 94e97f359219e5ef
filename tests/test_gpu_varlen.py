"""GPU: packed batches of sequences of any lengths (cu_seqlens) through one layer call."""
import numpy as np
import pytest
import torch

from dynamic_sparse_attention_vertical_gb300 import binding as B
from dynamic_sparse_attention_vertical_gb300 import inputs as I

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
H = B.HeadCfg


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def _packed(Hq, Hkv, lens, seed):
    """Sequences drawn one by one, packed along the token dimension."""
    seqs = [I.literal_inputs(Hq, Hkv, n, n_cols=4 if n > 256 else 0, n_offsets=2 if n > 256 else 0,
                             seed=seed + i, device=DEV) if n else None for i, n in enumerate(lens)]
    cat = lambda name: torch.cat([getattr(s, name) for s in seqs if s is not None], dim=1).contiguous()
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    return seqs, cat("q"), cat("k"), cat("v"), cu


def test_varlen_equals_the_layer_call_per_sequence():
    """Lengths 1000, 81, 2500, 0 (skipped), 40 (too short to estimate: its
    vertical-slash head runs dense) and 3001: outputs and log-sum-exps equal the layer
    call on each sequence on its own, bit for bit."""
    Hq, Hkv = 4, 2
    lens = [1000, 81, 2500, 0, 40, 3001]
    seqs, q, k, v, cu = _packed(Hq, Hkv, lens, seed=20)
    cfg = [H.vs(64, 32), H.block(8), H.ashape(128, 512), H.dense()]
    total = cu[-1]
    out = torch.full_like(q, 5.0)
    lse = torch.full((Hq, total), float("nan"), device=DEV)
    B.mi_layer_attn_varlen(q, k, v, cu, cfg, out=out, lse=lse)
    torch.cuda.synchronize()
    for b, n in enumerate(lens):
        if n == 0:
            continue
        s = seqs[b]
        c = list(cfg) if n >= 64 else [H.dense() if x.pattern == B.MI_PAT_VS else x for x in cfg]
        ro = torch.full_like(s.q, 5.0)
        rl = torch.full((Hq, n), float("nan"), device=DEV)
        B.mi_layer_attn(s.q, s.k, s.v, c, out=ro, lse=rl)
        torch.cuda.synchronize()
        lo, hi = cu[b], cu[b + 1]
        assert torch.equal(out[:, lo:hi], ro), f"sequence {b}"
        assert torch.equal(lse[:, lo:hi], rl), f"sequence {b} lse"


def test_varlen_block_expanded_equals_the_layer_call_per_sequence():
    """The block-expanded slash mode (needed 64-key blocks paired per tile) over ragged
    packed lengths: each sequence's rows equal its own layer call, bit for bit."""
    Hq, Hkv = 2, 1
    lens = [1500, 130, 2100]
    seqs, q, k, v, cu = _packed(Hq, Hkv, lens, seed=60)
    cfg = [H.vs(48, 24, expanded=True), H.vs(16, 64, expanded=True)]  # one slash mode per layer
    out = B.mi_layer_attn_varlen(q, k, v, cu, cfg)
    torch.cuda.synchronize()
    for b, n in enumerate(lens):
        s = seqs[b]
        ro = B.mi_layer_attn(s.q, s.k, s.v, cfg)
        torch.cuda.synchronize()
        assert torch.equal(out[:, cu[b]:cu[b + 1]], ro), f"sequence {b}"


def test_varlen_sequences_do_not_see_each_other():
    Hq, Hkv = 2, 1
    lens = [700, 1300]
    seqs, q, k, v, cu = _packed(Hq, Hkv, lens, seed=40)
    cfg = [H.vs(32, 16), H.dense()]
    a = B.mi_layer_attn_varlen(q, k, v, cu, cfg)
    k2, v2 = k.clone(), v.clone()
    k2[:, :700] = -k2[:, :700]
    v2[:, :700] = 3.0 * v2[:, :700]
    b = B.mi_layer_attn_varlen(q, k2, v2, cu, cfg)
    torch.cuda.synchronize()
    assert torch.equal(a[:, 700:], b[:, 700:])
    assert not torch.equal(a[:, :700], b[:, :700])


def test_varlen_rejects_malformed_offsets():
    Hq, Hkv = 2, 1
    seqs, q, k, v, cu = _packed(Hq, Hkv, [100, 200], seed=1)
    cfg = [H.dense(), H.ashape(16, 64)]
    for bad in ([0, 100, 250], [1, 100, 300], [0, 200, 100, 300]):
        with pytest.raises(B.MIError) as e:
            B.mi_layer_attn_varlen(q, k, v, bad, cfg)
        assert e.value.code == B.MI_ERR_ARG
