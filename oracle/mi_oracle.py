"""Plain fp64 restatement of dynamic sparse prefill attention (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use this module.  It shares nothing with the CUDA path.

What it restates, step by step, in the order the method takes them:

1. Online estimation of a vertical-slash head's indices
   (MInference talk slides, boteman.cn, "Step 2: Online Estimation of Sparsity
   Indices"; MInference README mirror, gittoolsai.com, "TL;DR": the pattern of
   each head is fixed offline, its sparse indices are approximated online).
   The last ``last_q`` queries are scored against every key with a causal
   softmax; the probabilities are summed per key column (vertical) and per
   diagonal offset q - j (slash); the top-k of each are kept.
2. A boolean mask per pattern (the same slides, "A-shape, Vertical-Slash and
   block-sparse patterns"; README mirror, "Kernel-only usage":
   ``vertical_slash_sparse_attention(q, k, v, vertical_topk, slash)``,
   ``block_sparse_attention(q, k, v, topk)``,
   ``streaming_forward(q, k, v, init_num, local_window_num)``).
3. Masked dense softmax attention with the 1/sqrt(d) scale.

Readings taken where the pages are silent (each listed in the design notes):
the vertical-slash mask also keeps the first ``blk`` keys and the keys of the
query's own aligned ``blk``-block; offsets are q - j; top-k ranks by larger
score then lower index, on scores rounded to fp32 (the precision the GPU
decides in), and returns indices in ascending order; offsets whose diagonal
meets fewer than ``last_q`` rows keep their raw sum; block-sparse ranks
mean-pooled Q.K (no scale) over blocks c <= r with no forced blocks; A-shape
keeps j < n_init or 0 <= q - j < window; GQA maps q-head h to KV head
h // (Hq / Hkv).
"""
from __future__ import annotations

import math
from typing import Callable, List, Optional, Sequence

import numpy as np

__all__ = [
    "BLK",
    "as_f64",
    "kv_head",
    "vs_estimate_scores",
    "topk_sorted",
    "vs_estimate",
    "vs_mask_rows",
    "vs_expanded_mask_rows",
    "block_pool",
    "block_scores",
    "block_sparse_select",
    "block_sparse_mask_rows",
    "ashape_mask_rows",
    "causal_mask_rows",
    "masked_attention_rows",
    "attention_rows",
]

BLK = 64


def as_f64(x) -> np.ndarray:
    """Exact upcast of a bf16/fp32 tensor or array to a float64 numpy array."""
    if hasattr(x, "detach"):  # a torch tensor: go through fp32, exact for bf16
        x = x.detach().to("cpu").float().numpy()
    return np.asarray(x, dtype=np.float64)


def kv_head(h: int, Hq: int, Hkv: int) -> int:
    """KV head of q-head ``h`` under grouped-query attention (consecutive groups)."""
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return h // (Hq // Hkv)


# ---------------------------------------------------------------------------
# 1. Online estimation (vertical-slash heads)
# ---------------------------------------------------------------------------

def vs_estimate_scores(q_h: np.ndarray, k_g: np.ndarray, last_q: int = 64):
    """Vertical and slash scores of one head.

    ``q_h``: [N, d] queries of the head, ``k_g``: [N, d] keys of its KV head.
    For the query rows p_i = N - last_q + i (i < last_q):
      l_ij = <q_{p_i}, k_j> / sqrt(d) for j <= p_i (causal),
      a_ij = exp(l_ij - max_j l_ij) / sum_j exp(l_ij - max_j l_ij),
      v[j] = sum_i a_ij                     (column, "vertical" score),
      s[o] = sum_i a_{i, p_i - o}, o >= 0   (diagonal offset, "slash" score).
    Returns (v, s), each float64 [N].
    """
    q_h = as_f64(q_h)
    k_g = as_f64(k_g)
    N, d = q_h.shape
    last_q = min(last_q, N)
    p = np.arange(N - last_q, N)
    logits = (q_h[p] @ k_g.T) / math.sqrt(d)
    keep = np.arange(N)[None, :] <= p[:, None]
    logits = np.where(keep, logits, -np.inf)
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    a = e / e.sum(axis=1, keepdims=True)
    v = a.sum(axis=0)
    s = np.zeros(N, dtype=np.float64)
    for i in range(last_q):
        keys = np.arange(p[i] + 1)
        s[p[i] - keys] += a[i, keys]      # one key per offset within a row
    return v, s


def topk_sorted(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices of the ``k`` largest scores, returned in ascending index order.

    Ranking: larger score first, equal scores by lower index.  The scores are
    rounded to fp32 first, the precision in which the GPU takes the same
    decision.  ``k`` is clipped to [0, len(scores)].
    """
    scores = np.asarray(scores)
    n = scores.shape[0]
    k = max(0, min(int(k), n))
    key = scores.astype(np.float32).astype(np.float64)
    order = np.lexsort((np.arange(n), -key))   # primary: -score, then index
    return np.sort(order[:k]).astype(np.int64)


def vs_estimate(q_h, k_g, last_q: int, k_v: int, k_s: int):
    """(v_idx, s_idx, v, s) for one vertical-slash head."""
    v, s = vs_estimate_scores(q_h, k_g, last_q)
    return topk_sorted(v, k_v), topk_sorted(s, k_s), v, s


# ---------------------------------------------------------------------------
# 2. Masks (one boolean row per query)
# ---------------------------------------------------------------------------

def causal_mask_rows(N: int, rows: Sequence[int]) -> np.ndarray:
    r = np.asarray(rows, dtype=np.int64)[:, None]
    return np.arange(N)[None, :] <= r


def vs_mask_rows(N: int, rows, v_idx, s_idx, blk: int = BLK) -> np.ndarray:
    """M[q, j] = j <= q and (j < blk or j//blk == q//blk or j in V or q-j in S)."""
    r = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.arange(N, dtype=np.int64)[None, :]
    col = np.zeros(N, dtype=bool)
    col[np.asarray(v_idx, dtype=np.int64)] = True
    sl = np.zeros(N, dtype=bool)
    sl[np.asarray(s_idx, dtype=np.int64)] = True
    off = r - j
    slash = np.where(off >= 0, sl[np.clip(off, 0, N - 1)], False)
    keep = (j < blk) | ((j // blk) == (r // blk)) | col[None, :] | slash
    return (j <= r) & keep


def vs_expanded_mask_rows(N: int, rows, v_idx, s_idx, blk: int = BLK) -> np.ndarray:
    """Block-expanded vertical-slash mask: every blk x blk block a selected diagonal crosses.

    The block kernels the MInference pages build on (PIT and the block-sparse
    FlashAttention of the talk slides, "Dynamic Sparse Attention Calculation
    with PIT, FlashAttention") cover the diagonals with whole blocks.  A diagonal
    o = blk*a + b crosses the blocks at block distance a and, when b > 0, a + 1;
    distance 0 (the query's own block) is always kept.
    M[q, j] = j <= q and (j < blk or j in V or q//blk - j//blk in D).
    """
    r = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.arange(N, dtype=np.int64)[None, :]
    col = np.zeros(N, dtype=bool)
    col[np.asarray(v_idx, dtype=np.int64)] = True
    dist = np.zeros(N // blk + 2, dtype=bool)
    dist[0] = True
    for o in np.asarray(s_idx, dtype=np.int64):
        dist[o // blk] = True
        if o % blk:
            dist[o // blk + 1] = True
    bd = r // blk - j // blk
    crossed = np.where(bd >= 0, dist[np.clip(bd, 0, dist.size - 1)], False)
    keep = (j < blk) | col[None, :] | crossed
    return (j <= r) & keep


def block_pool(x, blk: int = BLK) -> np.ndarray:
    """Mean of each run of ``blk`` consecutive rows (a partial last run: its own mean)."""
    x = as_f64(x)
    N = x.shape[0]
    nb = (N + blk - 1) // blk
    out = np.empty((nb, x.shape[1]), dtype=np.float64)
    for b in range(nb):
        out[b] = x[b * blk:(b + 1) * blk].mean(axis=0)
    return out


def block_scores(q_h, k_g, blk: int = BLK) -> np.ndarray:
    """sigma[r, c] = <mean-pooled q block r, mean-pooled k block c> (no scale)."""
    return block_pool(q_h, blk) @ block_pool(k_g, blk).T


def block_sparse_select(q_h, k_g, topk: int, blk: int = BLK) -> List[np.ndarray]:
    """Per query block r: top-min(topk, r+1) key blocks c <= r, ascending."""
    sig = block_scores(q_h, k_g, blk)
    return [topk_sorted(sig[r, : r + 1], min(topk, r + 1)) for r in range(sig.shape[0])]


def block_sparse_mask_rows(N: int, rows, sel: List[np.ndarray], blk: int = BLK) -> np.ndarray:
    r = np.asarray(rows, dtype=np.int64)
    j = np.arange(N, dtype=np.int64)
    out = np.zeros((r.shape[0], N), dtype=bool)
    for n, q in enumerate(r):
        chosen = np.zeros((N + blk - 1) // blk, dtype=bool)
        chosen[np.asarray(sel[q // blk], dtype=np.int64)] = True
        out[n] = (j <= q) & chosen[j // blk]
    return out


def ashape_mask_rows(N: int, rows, n_init: int, window: int) -> np.ndarray:
    """Sink keys j < n_init plus the local window 0 <= q - j < window, causal."""
    r = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.arange(N, dtype=np.int64)[None, :]
    return (j <= r) & ((j < n_init) | ((r - j) < window))


# ---------------------------------------------------------------------------
# 3. Masked softmax attention
# ---------------------------------------------------------------------------

def masked_attention_rows(q_h, k_g, v_g, rows, mask: np.ndarray):
    """O[q] = sum_j softmax_j(<q, k_j>/sqrt(d) over kept j) v_j for q in ``rows``.

    Returns (O [len(rows), d], lse [len(rows)]) in float64, lse being the
    natural log of sum_j exp(<q, k_j>/sqrt(d)) over kept j.
    """
    q_h = as_f64(q_h)
    k_g = as_f64(k_g)
    v_g = as_f64(v_g)
    d = q_h.shape[1]
    rows = np.asarray(rows, dtype=np.int64)
    logits = (q_h[rows] @ k_g.T) / math.sqrt(d)
    logits = np.where(mask, logits, -np.inf)
    m = logits.max(axis=1, keepdims=True)
    if not np.all(np.isfinite(m)):
        raise ValueError("a query row keeps no key")
    e = np.exp(logits - m)
    l = e.sum(axis=1, keepdims=True)
    o = (e / l) @ v_g
    return o, (m + np.log(l))[:, 0]


def attention_rows(q_h, k_g, v_g, rows, mask_fn: Callable[[np.ndarray], np.ndarray],
                   chunk: int = 256):
    """``masked_attention_rows`` over ``rows`` in chunks; ``mask_fn(rows)`` gives the mask."""
    q_h = as_f64(q_h)
    k_g = as_f64(k_g)
    v_g = as_f64(v_g)
    rows = np.asarray(rows, dtype=np.int64)
    outs, lses = [], []
    for c in range(0, rows.shape[0], chunk):
        rr = rows[c:c + chunk]
        o, l = masked_attention_rows(q_h, k_g, v_g, rr, mask_fn(rr))
        outs.append(o)
        lses.append(l)
    if not outs:
        return np.zeros((0, q_h.shape[1])), np.zeros((0,))
    return np.concatenate(outs), np.concatenate(lses)
