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


def test_noalloc_rejects_jobs_larger_than_its_array():
    # 32 heads x 1M tokens need 8 * 32 * 2^20 bytes of scratch, far above the fixed
    # array; the call must refuse before queueing any work (the small buffers
    # below are never read).
    buf = torch.zeros(1024, dtype=torch.bfloat16, device=DEV)
    out = torch.zeros(64, dtype=torch.int32, device=DEV)
    p = ctypes.c_void_p
    rc = B.load().mi_vs_estimate_noalloc(p(buf.data_ptr()), p(buf.data_ptr()), 32, 8, 1 << 20, 128,
                                         None, 32, 64, 1, 1, p(out.data_ptr()), p(out.data_ptr()),
                                         p(torch.cuda.current_stream().cuda_stream))
    assert rc == B.MI_ERR_WORKSPACE
    torch.cuda.synchronize()
