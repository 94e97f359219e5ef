"""Kernel-aware sparse pattern search: the offline step that assigns each head its pattern.

The MInference talk slides ("Step 1: Kernel-Aware Sparse Pattern Search") fix each
head's pattern offline: among the A-shape, vertical-slash and block-sparse patterns
and their budgets, a head gets the one that keeps the most attention for a given
cost, where the cost is that of the actual kernels.  Here both sides are measured
with this library's own kernels on a calibration input:

* recall of a candidate for a head: the attention mass its mask keeps, averaged
  over the rows.  For row q it is exp(lse_pattern(q) - lse_dense(q)), the ratio
  of the two log-sum-exps over the kept and over all causal keys (both written by
  the attention calls);
* cost: the measured time of the candidate's calls per copy of that head, on
  ``copies`` copies of it at once so that the GPU is full (one head alone is one
  wave of CTAs and measures the slowest row block, not throughput); CUDA
  events, best of ``reps``; the online index step included (estimation for
  vertical-slash heads, pooling and selection for block-sparse heads).

The head gets the highest-recall candidate whose cost fits the budget; among the
candidates within ``recall_tol`` of that recall, the cheapest.  With nothing in the
budget it gets the cheapest candidate.  This module only orchestrates calls
through ``binding``; every step runs in the library's kernels.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence, Tuple

import torch

from . import binding as B

__all__ = ["Candidate", "Evaluation", "HeadChoice", "default_candidates", "choose", "search", "layer_config"]


@dataclasses.dataclass(frozen=True)
class Candidate:
    pattern: str                        # "ashape" | "vs" | "block"
    params: Tuple[Tuple[str, int], ...]  # sorted (name, value) pairs

    @staticmethod
    def make(pattern: str, **params) -> "Candidate":
        if pattern not in ("ashape", "vs", "block"):
            raise ValueError(f"unknown pattern {pattern!r}")
        return Candidate(pattern, tuple(sorted(params.items())))

    @property
    def p(self) -> Dict[str, int]:
        return dict(self.params)

    def __str__(self) -> str:
        return self.pattern + "(" + ", ".join(f"{k}={v}" for k, v in self.params) + ")"


@dataclasses.dataclass
class Evaluation:
    candidate: Candidate
    recall: float    # mean kept attention mass over the rows
    cost_ms: float   # measured latency for this head


@dataclasses.dataclass
class HeadChoice:
    head: int
    choice: Evaluation
    dense_ms: float
    budget_ms: float
    evaluations: List[Evaluation]


def default_candidates() -> List[Candidate]:
    """Budgets around the ones the pages use (A-shape 128 + window, vertical-slash
    1000 / 6096 at 128K, block-sparse top 100) and smaller ones."""
    c = [Candidate.make("ashape", n_init=128, window=w) for w in (1024, 2048, 4096)]
    c += [Candidate.make("vs", k_v=kv, k_s=ks) for kv, ks in ((64, 16), (128, 64), (256, 256), (1000, 1024))]
    c += [Candidate.make("block", topk=t) for t in (16, 32, 64, 100)]
    return c


def choose(evals: Sequence[Evaluation], budget_ms: float, recall_tol: float = 0.005) -> Evaluation:
    """Highest recall within the budget; the cheapest within ``recall_tol`` of it.

    With nothing within the budget, the cheapest evaluation overall.
    """
    if not evals:
        raise ValueError("no candidates")
    fit = [e for e in evals if e.cost_ms <= budget_ms]
    if not fit:
        return min(evals, key=lambda e: (e.cost_ms, -e.recall))
    best = max(e.recall for e in fit)
    near = [e for e in fit if e.recall >= best - recall_tol]
    return min(near, key=lambda e: (e.cost_ms, -e.recall))


def _run(cand: Candidate, q, k, v, heads, out, lse):
    """Run one candidate's calls (index step + attention) for ``heads``."""
    p = cand.p
    if cand.pattern == "ashape":
        B.mi_ashape_attn(q, k, v, n_init=p["n_init"], window=p["window"], heads=heads, out=out, lse=lse)
    elif cand.pattern == "vs":
        vi, si = B.mi_vs_estimate(q, k, heads=heads, k_v=p["k_v"], k_s=p["k_s"])
        B.mi_vs_sparse_attn(q, k, v, vi, si, heads=heads, out=out, lse=lse)
    else:
        B.mi_block_sparse_attn(q, k, v, topk=p["topk"], heads=heads, out=out, lse=lse)


def _time(fn, reps: int) -> float:
    best = math.inf
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        best = min(best, a.elapsed_time(b))
    return best


def search(q, k, v, heads: Optional[Sequence[int]] = None, candidates: Optional[Sequence[Candidate]] = None,
           budget_frac: float = 0.4, recall_tol: float = 0.005, reps: int = 3,
           rows: Optional[slice] = None, copies: int = 16) -> List[HeadChoice]:
    """Evaluate every candidate on every listed head and choose per head.

    q, k, v: ``[H, N, 128]`` bf16 CUDA tensors with one KV head per q-head (a
    calibration input).  The budget of a head is ``budget_frac`` times its
    measured dense causal time.  ``rows`` restricts the recall average (default:
    all rows).
    """
    if not q.is_cuda:
        raise ValueError("the pattern search runs the CUDA kernels: pass CUDA tensors")
    Hq, N, _ = q.shape
    heads = list(range(Hq)) if heads is None else [int(h) for h in heads]
    candidates = list(default_candidates() if candidates is None else candidates)
    rows = slice(None) if rows is None else rows
    out = torch.empty_like(q)
    lse_d = torch.full((Hq, N), float("nan"), dtype=torch.float32, device=q.device)
    B.mi_dense_causal_attn(q, k, v, heads=heads, out=out, lse=lse_d)
    recalls: Dict[Candidate, torch.Tensor] = {}
    for cand in candidates:
        lse_c = torch.full_like(lse_d, float("nan"))
        _run(cand, q, k, v, heads, out, lse_c)
        r = torch.exp(lse_c - lse_d)[:, rows].double().mean(dim=1)
        recalls[cand] = r.cpu()
    torch.cuda.synchronize()
    choices = []
    for h in heads:
        qr, kr, vr = (t[h:h + 1].expand(copies, -1, -1).contiguous() for t in (q, k, v))
        outr = torch.empty_like(qr)
        B.mi_dense_causal_attn(qr, kr, vr, out=outr)
        dense_ms = _time(lambda: B.mi_dense_causal_attn(qr, kr, vr, out=outr), reps) / copies
        evals = []
        for cand in candidates:
            _run(cand, qr, kr, vr, None, outr, None)  # warm-up of this shape
            ms = _time(lambda: _run(cand, qr, kr, vr, None, outr, None), reps) / copies
            evals.append(Evaluation(cand, float(recalls[cand][h]), ms))
        budget = budget_frac * dense_ms
        choices.append(HeadChoice(h, choose(evals, budget, recall_tol), dense_ms, budget, evals))
        del qr, kr, vr, outr
    return choices


def layer_config(choices: Sequence[HeadChoice], Hq: int) -> List["B.HeadCfg"]:
    """The per-head configuration of ``mi_layer_attn`` for the chosen patterns
    (heads without a choice are computed dense)."""
    cfg = [B.HeadCfg.dense() for _ in range(Hq)]
    for c in choices:
        p = c.choice.candidate.p
        pat = c.choice.candidate.pattern
        if pat == "vs":
            cfg[c.head] = B.HeadCfg.vs(p["k_v"], p["k_s"])
        elif pat == "block":
            cfg[c.head] = B.HeadCfg.block(p["topk"])
        else:
            cfg[c.head] = B.HeadCfg.ashape(p["n_init"], p["window"])
    return cfg


def _main(argv=None) -> None:
    """Run the search on the synthetic pattern heads and print one JSON line per head."""
    import argparse
    import json

    from . import inputs as I

    ap = argparse.ArgumentParser(description="kernel-aware pattern search on synthetic heads")
    ap.add_argument("--seqlen", type=int, default=32768)
    ap.add_argument("--seed", type=int, default=5)
    ap.add_argument("--budget-frac", type=float, default=0.4)
    args = ap.parse_args(argv)
    x = I.pattern_head_inputs(args.seqlen, seed=args.seed, device="cuda")
    for c in search(x.q, x.k, x.v, budget_frac=args.budget_frac):
        print(json.dumps({
            "head": c.head, "choice": str(c.choice.candidate), "recall": c.choice.recall,
            "cost_ms": c.choice.cost_ms, "dense_ms": c.dense_ms, "budget_ms": c.budget_ms,
            "candidates": [{"candidate": str(e.candidate), "recall": e.recall, "cost_ms": e.cost_ms}
                           for e in c.evaluations]}))


if __name__ == "__main__":
    _main()
