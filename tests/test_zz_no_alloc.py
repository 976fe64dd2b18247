"""rlk_logprob_noalloc: the allocation-free entry point for callers that cannot
allocate device memory (engines with a pre-reserved memory pool, decode loops
that must not block on the allocator).

Called through the C ABI with ctypes, twice in a row with different inputs, and
compared with rlk_logprob (the existing entry point) under the parity
tolerances of the other tests -- the two paths run the same kernels, so the
bits are expected to be identical as well.  Also checks that a problem larger
than the fixed scratch is refused before anything runs.

The file name sorts last so that a run stopping at the first failure has
already run every other test; it needs no state from them.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import LOGP_ATOL, LSE_RTOL
from invariant_token_logprob_gb300.inputs import lm_head_inputs

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    import invariant_token_logprob_gb300 as rlk
    L = rlk.lib()
    f = L.rlk_logprob_noalloc
    P, i64 = ctypes.c_void_p, ctypes.c_int64
    f.restype = ctypes.c_int
    f.argtypes = [P, P, P, i64, i64, i64, ctypes.c_float, P, P, P, P]
    return f


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _call_noalloc(f, h, W, tg, inv_temp):
    T, H = h.shape
    V = W.shape[0]
    lp = torch.full((T,), float("nan"), device=h.device)
    lse = torch.full((T,), float("nan"), device=h.device)
    am = torch.full((T,), -7, device=h.device, dtype=torch.int32)
    st = f(_ptr(h), _ptr(W), _ptr(tg), T, H, V, ctypes.c_float(inv_temp), _ptr(lp), _ptr(lse),
           _ptr(am), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, (lp, lse, am)


@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")
def test_noalloc_matches_logprob_on_two_calls_in_a_row():
    import invariant_token_logprob_gb300 as rlk
    f = _noalloc_fn()
    cases = [  # (T, H, V, inv_temp, seed): the second call is smaller, so stale
               # scratch from the first call would show up if it leaked
        (1000, 4096, 151936, 1.0, 41),
        (37, 256, 5000, float(np.float32(1 / 0.7)), 42),
    ]
    for T, H, V, it, seed in cases:
        d = lm_head_inputs(T, H, V, seed=seed, device="cuda")
        st, got = _call_noalloc(f, d["h"], d["W"], d["targets"], it)
        assert st == 0, rlk.lib().rlk_status_string(st).decode()
        rlk.check_device_error()
        ref = rlk.logprob(d["h"], d["W"], d["targets"], it)
        torch.cuda.synchronize()
        g = [x.cpu().numpy() for x in got]
        r = [x.cpu().numpy() for x in ref]
        assert np.all(np.isfinite(g[0])) and np.all(np.isfinite(g[1]))
        assert np.max(np.abs(g[0].astype(np.float64) - r[0])) <= LOGP_ATOL
        assert np.all(np.abs(g[1].astype(np.float64) - r[1]) <= LSE_RTOL * np.maximum(1, np.abs(r[1])))
        assert np.array_equal(g[2], r[2])
        assert np.array_equal(g[0].view(np.uint32), r[0].view(np.uint32))
        assert np.array_equal(g[1].view(np.uint32), r[1].view(np.uint32))


@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")
def test_noalloc_refuses_problems_beyond_its_scratch():
    f = _noalloc_fn()
    V = 151936
    limit = (16 << 20) // (((V + 255) // 256) * 16)   # 1765 rows at this V
    h = torch.zeros(limit + 1, 64, device="cuda", dtype=torch.bfloat16)
    W = torch.zeros(V, 64, device="cuda", dtype=torch.bfloat16)
    tg = torch.zeros(limit + 1, device="cuda", dtype=torch.int32)
    st, (lp, _, _) = _call_noalloc(f, h, W, tg, 1.0)
    assert st == 5  # RLK_ERR_WORKSPACE, returned before any launch
    assert torch.isnan(lp).all()  # outputs untouched
    st, _ = _call_noalloc(f, h[:limit], W, tg[:limit], 1.0)
    assert st == 0
    torch.cuda.synchronize()
