"""Failure detection and execution-context tests on the GPU.

* A device-side wait that nothing will ever complete runs out after its time
  limit; the kernel records it, frees its tensor memory and returns, the host
  reads RLK_ERR_TIMEOUT, and the CUDA context stays usable (no fault, no hang).
  Single-CTA shape: the self-test issues no copy at all.  CTA-pair shape: the
  same (mode 1), and a run whose MMA issuer consumes nothing (mode 2), so both
  CTAs' copies fill their rings and the pair's teardown hand-shake must drain
  them before the CTAs leave.
* rlk_logprob_ws captured in a CUDA graph and replayed with new inputs gives
  the eager bits (decode loops run under CUDA graphs).
* Concurrent calls on two streams (each with its own cached workspace) give
  the same bits as sequential calls.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bitwise, assert_parity, gpu_logprob, to_dev
from invariant_token_logprob_gb300.inputs import lm_head_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import invariant_token_logprob_gb300 as rlk
    rlk.lib()


def _np(xs):
    return tuple(x.cpu().numpy() for x in xs)


def test_bounded_wait_runs_out_and_context_survives(olib):
    import invariant_token_logprob_gb300 as rlk
    L = rlk.lib()
    h = torch.zeros(1, 64, device="cuda", dtype=torch.bfloat16)
    W = torch.zeros(256, 64, device="cuda", dtype=torch.bfloat16)
    tg = torch.zeros(1, device="cuda", dtype=torch.int32)
    part = torch.full((4,), 7.0, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rlk.check_device_error()  # start from a clear error word
    t0 = time.time()
    st = L.rlk_selftest_wait_timeout(ctypes.c_void_p(h.data_ptr()), ctypes.c_void_p(W.data_ptr()),
                                     ctypes.c_void_p(tg.data_ptr()),
                                     ctypes.c_void_p(part.data_ptr()), stream)
    assert st == 0
    with pytest.raises(rlk.RlkError) as e:
        rlk.check_device_error()
    elapsed = time.time() - t0
    assert e.value.status == 6  # RLK_ERR_TIMEOUT
    assert 1.0 < elapsed < 30.0, elapsed
    assert torch.all(part == 7.0)  # nothing was written
    rlk.check_device_error()  # the word was cleared by the read
    # the context is still usable: a normal call is correct
    d = lm_head_inputs(20, 128, 900, seed=3)
    dd = to_dev(d)
    gpu = gpu_logprob(dd["h"], dd["W"], dd["targets"])
    assert_parity(gpu, oracle.logprob(d["h"], d["W"], d["targets"], lib=olib), what="after timeout")


@pytest.mark.parametrize("mode", [1, 2])
def test_pair_shape_bounded_wait_runs_out_and_context_survives(olib, mode):
    import invariant_token_logprob_gb300 as rlk
    L = rlk.lib()
    g = torch.Generator("cuda").manual_seed(mode)
    h = torch.randn(256, 512, device="cuda", generator=g).to(torch.bfloat16)
    W = torch.randn(256, 512, device="cuda", generator=g).to(torch.bfloat16)
    tg = torch.zeros(256, device="cuda", dtype=torch.int32)
    part = torch.full((256 * 4,), 7.0, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rlk.check_device_error()
    assert L.rlk_selftest_wait_timeout_pair(ctypes.c_void_p(h.data_ptr()),
                                            ctypes.c_void_p(W.data_ptr()),
                                            ctypes.c_void_p(tg.data_ptr()),
                                            ctypes.c_void_p(part.data_ptr()), 3, stream) == 1
    t0 = time.time()
    st = L.rlk_selftest_wait_timeout_pair(ctypes.c_void_p(h.data_ptr()),
                                          ctypes.c_void_p(W.data_ptr()),
                                          ctypes.c_void_p(tg.data_ptr()),
                                          ctypes.c_void_p(part.data_ptr()), mode, stream)
    assert st == 0
    bits, rows = rlk.take_device_errors()
    elapsed = time.time() - t0
    assert bits & 1, bits  # a wait ran out
    assert not bits & 2, bits  # and every teardown wait (the hand-shake, the drains) ended in time
    assert 1.0 < elapsed < 30.0, elapsed
    assert torch.all(part == 7.0)  # nothing was written
    rlk.check_device_error()
    # the context is still usable: CTA-pair and single-CTA calls are correct
    for T in (300, 20):
        d = lm_head_inputs(T, 128, 900, seed=T)
        dd = to_dev(d)
        gpu = gpu_logprob(dd["h"], dd["W"], dd["targets"])
        assert_parity(gpu, oracle.logprob(d["h"], d["W"], d["targets"], lib=olib),
                      what=f"after pair timeout, T={T}")


@pytest.mark.parametrize("T", [1, 37, 300])  # 300: CTA-pair clusters, ragged last unit
def test_cuda_graph_capture_and_replay(T):
    import invariant_token_logprob_gb300 as rlk
    H, V = 256, 3000
    a = to_dev(lm_head_inputs(T, H, V, seed=40))
    b = to_dev(lm_head_inputs(T, H, V, seed=41))
    W = a["W"]
    h_s, tg_s = a["h"].clone(), a["targets"].clone()
    ws = torch.empty(rlk.workspace_size(T, H, V), dtype=torch.uint8, device="cuda")
    outs = [torch.empty(T, device="cuda", dtype=dt) for dt in (torch.float32, torch.float32, torch.int32)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        rlk.logprob_ws(h_s, W, tg_s, ws, out=outs)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        rlk.logprob_ws(h_s, W, tg_s, ws, out=outs)
    for src in (b, a, b):
        h_s.copy_(src["h"])
        tg_s.copy_(src["targets"])
        g.replay()
        torch.cuda.synchronize()
        ref = _np(rlk.logprob(src["h"], W, src["targets"]))
        assert_bitwise(ref, _np(outs), f"graph replay T={T}")
    rlk.check_device_error()


def test_concurrent_streams_match_sequential():
    import invariant_token_logprob_gb300 as rlk
    ds = [to_dev(lm_head_inputs(T, 512, 20000, seed=50 + T)) for T in (300, 7)]
    seq = [_np(rlk.logprob(d["h"], d["W"], d["targets"])) for d in ds]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    res = [None, None]
    for _ in range(3):
        for i, (d, s) in enumerate(zip(ds, streams)):
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                res[i] = rlk.logprob(d["h"], d["W"], d["targets"])
        torch.cuda.synchronize()
        for i in range(2):
            assert_bitwise(seq[i], _np(res[i]), f"stream {i}")
    rlk.check_device_error()
