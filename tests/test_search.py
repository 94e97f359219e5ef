"""Host logic of the kernel-aware pattern search (no GPU)."""
import pytest

from dynamic_sparse_attention_vertical_gb300 import search as S


def _e(pat, recall, cost, **p):
    return S.Evaluation(S.Candidate.make(pat, **p), recall, cost)


def test_choose_takes_best_recall_within_budget():
    evals = [_e("ashape", 0.70, 1.0, n_init=128, window=1024), _e("vs", 0.95, 2.0, k_v=64, k_s=16),
             _e("block", 0.99, 5.0, topk=32)]
    assert S.choose(evals, budget_ms=3.0).candidate.pattern == "vs"
    assert S.choose(evals, budget_ms=10.0).candidate.pattern == "block"


def test_choose_prefers_cheapest_among_near_ties():
    evals = [_e("block", 0.998, 1.2, topk=16), _e("ashape", 0.996, 0.9, n_init=128, window=1024),
             _e("ashape", 0.999, 2.0, n_init=128, window=4096)]
    got = S.choose(evals, budget_ms=5.0, recall_tol=0.005)
    assert got.candidate == S.Candidate.make("ashape", n_init=128, window=1024)
    # with a tight tolerance only the best recall counts
    assert S.choose(evals, budget_ms=5.0, recall_tol=0.0).recall == 0.999


def test_choose_falls_back_to_cheapest_when_nothing_fits():
    evals = [_e("vs", 0.9, 3.0, k_v=64, k_s=16), _e("block", 0.95, 2.5, topk=16)]
    assert S.choose(evals, budget_ms=1.0).candidate.pattern == "block"


def test_candidates_and_errors():
    c = S.default_candidates()
    assert {x.pattern for x in c} == {"ashape", "vs", "block"}
    assert len(set(c)) == len(c)
    assert str(S.Candidate.make("vs", k_s=16, k_v=64)) == "vs(k_s=16, k_v=64)"
    with pytest.raises(ValueError):
        S.Candidate.make("dense")
    with pytest.raises(ValueError):
        S.choose([], 1.0)
