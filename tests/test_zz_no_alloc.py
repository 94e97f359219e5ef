"""The allocation-free estimation entry point against the workspace one (GPU).

mi_vs_estimate_noalloc serves callers that cannot allocate device memory when
they call in (an engine whose pool owns the device, a plugin where cudaMalloc is
off limits): it runs the same estimation in a fixed scratch array that libmi.so
owns.  Its indices must equal those of mi_vs_estimate on the same inputs, call
after call, even though every call reuses the array the previous one left
behind.  This file is collected last so that a failure here cannot hide the
other GPU tests.
"""
import ctypes

import pytest
import torch

from dynamic_sparse_attention_vertical_gb300 import binding as B
from dynamic_sparse_attention_vertical_gb300 import inputs as I

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def test_noalloc_matches_workspace_call_twice_in_a_row():
    cases = [
        (I.margin_inputs(4, 2, 2048, 64, 32, seed=17), 64, 32),  # exact planted sets
        (I.literal_inputs(2, 1, 4160, n_cols=8, n_offsets=4, seed=23), 100, 50),  # ragged N
    ]
    for x, k_v, k_s in cases:  # second call runs over the first call's leftovers
        q, k = x.q.to(DEV), x.k.to(DEV)
        ref_v, ref_s = B.mi_vs_estimate(q, k, k_v=k_v, k_s=k_s)
        got_v, got_s = B.mi_vs_estimate_noalloc(q, k, k_v=k_v, k_s=k_s)
        torch.cuda.synchronize()
        assert torch.equal(got_v, ref_v) and torch.equal(got_s, ref_s)
        if x.kind == "margin":
            for h in range(4):
                assert got_v[h].cpu().tolist() == x.planted_cols[h // 2].tolist()
                assert got_s[h].cpu().tolist() == x.planted_offsets[h // 2].tolist()


def _raw_call(q, k, Hq, Hkv, N, n_heads, last_q=64, k_v=1, k_s=1, out=None):
    p = ctypes.c_void_p
    return B.load().mi_vs_estimate_noalloc(p(q.data_ptr()), p(k.data_ptr()), Hq, Hkv, N, 128, None,
                                           n_heads, last_q, k_v, k_s, p(out.data_ptr()), p(out.data_ptr()),
                                           p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_largest_documented_job_runs_and_the_next_size_is_refused():
    # The header documents that a whole 32-head layer fits the 36 MiB array up to
    # N = 138686 tokens.  That job must run and equal the workspace call; one more
    # token must be refused with MI_ERR_WORKSPACE before any work is queued.
    N = 138686
    assert B.mi_workspace_bytes(B.MI_OP_VS_ESTIMATE, 32, 8, N) <= 36 << 20
    assert B.mi_workspace_bytes(B.MI_OP_VS_ESTIMATE, 32, 8, N + 1) > 36 << 20
    g = torch.Generator(device=DEV).manual_seed(31)
    q = (torch.randn((32, N + 1, 128), generator=g, device=DEV) / 128 ** 0.5).to(torch.bfloat16)
    k = (torch.randn((8, N + 1, 128), generator=g, device=DEV) / 128 ** 0.5).to(torch.bfloat16)
    qn, kn = q[:, :N].contiguous(), k[:, :N].contiguous()
    ref_v, ref_s = B.mi_vs_estimate(qn, kn, k_v=1000, k_s=2048)
    got_v, got_s = B.mi_vs_estimate_noalloc(qn, kn, k_v=1000, k_s=2048)
    torch.cuda.synchronize()
    assert torch.equal(got_v, ref_v) and torch.equal(got_s, ref_s)
    del qn, kn
    out = torch.zeros(64, dtype=torch.int32, device=DEV)
    assert _raw_call(q, k, 32, 8, N + 1, 32, out=out) == B.MI_ERR_WORKSPACE
    torch.cuda.synchronize()


def test_noalloc_checks_arguments_before_its_size_limit():
    # A job too large for the array but with a bad argument reports the argument
    # error, as mi_vs_estimate would (its checks come first).
    buf = torch.zeros(1024, dtype=torch.bfloat16, device=DEV)
    out = torch.zeros(64, dtype=torch.int32, device=DEV)
    assert _raw_call(buf, buf, 32, 8, 1 << 20, 32, last_q=32, out=out) == B.MI_ERR_SHAPE
    assert _raw_call(buf, buf, 32, 7, 1 << 20, 32, out=out) == B.MI_ERR_SHAPE
    assert _raw_call(buf, buf, 32, 8, 1 << 20, 32, k_v=-1, out=out) == B.MI_ERR_ARG
    torch.cuda.synchronize()


def test_noalloc_rejects_jobs_larger_than_its_array():
    # 32 heads x 1M tokens need 8 * 32 * 2^20 bytes of scratch, far above the fixed
    # array; the call must refuse before queueing any work (the small buffers
    # below are never read).
    buf = torch.zeros(1024, dtype=torch.bfloat16, device=DEV)
    out = torch.zeros(64, dtype=torch.int32, device=DEV)
    assert _raw_call(buf, buf, 32, 8, 1 << 20, 32, out=out) == B.MI_ERR_WORKSPACE
    torch.cuda.synchronize()
