"""Comparison helpers shared by the GPU parity tests."""
import numpy as np

MAX_ABS = 2e-2   # bf16 outputs against the fp64 oracle
MEAN_ABS = 2e-3
REL_FRO = 1e-2   # per head: guards rows whose |O| is far below MAX_ABS


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert err.max() <= MAX_ABS, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean abs err {err.mean():.3e}"
    assert rel <= REL_FRO, f"{what}: relative Frobenius err {rel:.3e}"
    return err.max(), err.mean(), rel


def rel_fro(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)


def band_agree(gpu_idx, ref_idx, scores, k, rel_band=1e-4, must_have=()):
    """Index sets may differ only on elements whose score sits at the top-k boundary.

    tau = the oracle's k-th largest score (fp32-rounded); every index in the
    symmetric difference must score within rel_band * tau of tau.  Planted
    indices (must_have) must be in the GPU set.  Returns the disagreement count.
    """
    g = set(int(i) for i in np.asarray(gpu_idx) if i >= 0)
    r = set(int(i) for i in np.asarray(ref_idx) if i >= 0)
    assert len(g) == len(r), f"set sizes {len(g)} vs {len(r)}"
    sc = np.asarray(scores, dtype=np.float32).astype(np.float64)
    kk = min(k, len(sc))
    if kk == 0:
        return 0
    tau = np.sort(sc)[::-1][kk - 1]
    diff = g ^ r
    for i in diff:
        assert abs(sc[i] - tau) <= rel_band * abs(tau) + 1e-12, (
            f"index {i} score {sc[i]:.9g} outside the band around tau={tau:.9g}")
    for i in must_have:
        assert int(i) in g, f"planted index {int(i)} missing"
    return len(diff)


def sample_rows(N, rng, n_random=64, blocks=4):
    """All rows of the first, last and a few random 128-row blocks plus random rows."""
    nb = (N + 127) // 128
    pick = {0, nb - 1} | set(int(b) for b in rng.integers(0, nb, size=blocks))
    rows = set()
    for b in pick:
        rows |= set(range(b * 128, min(N, b * 128 + 128)))
    rows |= set(int(r) for r in rng.integers(0, N, size=n_random))
    return np.array(sorted(rows))
