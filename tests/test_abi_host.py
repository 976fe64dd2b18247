"""Host-only checks of the C-ABI library (no GPU needed, no compute calls):
it loads, exports every function include/rlk.h declares, reports its tile
shape and workspace size, and rejects bad arguments on the host before touching
a device."""
import ctypes

import pytest

import invariant_token_logprob_gb300 as rlk


@pytest.fixture(scope="module")
def L():
    from invariant_token_logprob_gb300 import _build
    _build.build()
    return rlk.lib()


def test_exports_every_header_function(L):
    names = rlk.header_functions()
    assert len(names) >= 12, names
    for n in names:
        assert hasattr(L, n), f"librlk.so does not export {n}"


def test_abi_version_and_tiles(L):
    assert L.rlk_abi_version() == 1
    assert L.rlk_row_tile() == 128
    assert L.rlk_vocab_tile() == 256
    for s in range(8):
        assert L.rlk_status_string(s).decode().startswith("RLK_")
    assert L.rlk_status_string(99) == b"unknown rlk_status"


def test_workspace_size(L):
    assert L.rlk_logprob_workspace_size(0, 64, 10) == 0
    assert L.rlk_logprob_workspace_size(5, 64, 0) == 0
    assert L.rlk_logprob_workspace_size(5, 0, 10) == 0
    assert L.rlk_logprob_workspace_size(4096, 4096, 151936) == 4096 * 594 * 16
    assert L.rlk_logprob_workspace_size(16, 4096, 151936) == 16 * 594 * 16
    # the partials alone, whatever T (no staging copy of h)
    assert L.rlk_logprob_workspace_size(1, 4096, 151936) == 594 * 16
    assert L.rlk_logprob_workspace_size(3, 64, 257) == 3 * 2 * 16


A16 = ctypes.c_void_p(1 << 20)       # a 16-byte-aligned dummy address (never dereferenced)
A4 = ctypes.c_void_p((1 << 20) + 4)  # 4-byte aligned only


def _lp(L, h=A16, W=A16, tg=A16, T=4, H=64, V=100, it=1.0, out=A16):
    return L.rlk_logprob(h, W, tg, T, H, V, ctypes.c_float(it), out, out, out, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(T=-1), 1), (dict(H=0), 1), (dict(V=0), 1), (dict(V=1 << 31), 1),
    (dict(it=0.0), 1), (dict(it=-1.0), 1), (dict(it=float("nan")), 1), (dict(it=float("inf")), 1),
    (dict(h=None), 1), (dict(W=None), 1), (dict(tg=None), 1), (dict(out=None), 1),
    (dict(H=60), 2), (dict(h=A4), 2), (dict(W=A4), 2),
])
def test_argument_errors_detected_on_host(L, kw, expect):
    assert _lp(L, **kw) == expect


def test_zero_rows_is_a_no_op(L):
    # T == 0 returns OK without touching any pointer or device
    assert _lp(L, T=0, h=None, W=None, tg=None, out=None) == 0
    assert L.rlk_logprob_ws(None, None, None, 0, 64, 10, ctypes.c_float(1.0), None, None, None,
                            None, 0, None) == 0
    assert L.rlk_lse_merge(None, None, 0, 10, None, None, None, None) == 0


def test_ws_and_partials_errors(L):
    f = ctypes.c_float(1.0)
    # workspace missing / too small / misaligned
    assert L.rlk_logprob_ws(A16, A16, A16, 4, 64, 100, f, A16, A16, A16, None, 0, None) == 5
    assert L.rlk_logprob_ws(A16, A16, A16, 4, 64, 100, f, A16, A16, A16, A16, 16, None) == 5
    assert L.rlk_logprob_ws(A16, A16, A16, 4, 64, 100, f, A16, A16, A16, A4, 1 << 20, None) == 2
    assert L.rlk_logprob_partials(A16, A16, A16, 4, 64, 100, f, A16, 16, None) == 5
    assert L.rlk_logprob_partials(A16, A16, A16, 4, 64, 100, f, None, 1 << 20, None) == 1
    assert L.rlk_lse_merge(A16, A16, -1, 10, A16, A16, A16, None) == 1
    assert L.rlk_lse_merge(A4, A16, 3, 10, A16, A16, A16, None) == 2


def test_stats_host_paths(L):
    out = (ctypes.c_double * 8)()
    assert L.rlk_consistency_stats(A16, A16, None, -1, out, None) == 1
    assert L.rlk_consistency_stats(A16, A16, None, 5, None, None) == 1
    assert L.rlk_consistency_stats(None, A16, None, 5, out, None) == 1
    # n == 0: answered on the host, nothing valid
    assert L.rlk_consistency_stats(None, None, None, 0, out, None) == 0
    assert list(out) == [0.0] * 7 + [-1.0]


def test_stats_async_host_checks(L):
    L.rlk_consistency_stats_workspace_size.restype = ctypes.c_size_t
    L.rlk_consistency_stats_workspace_size.argtypes = [ctypes.c_int64]
    f = L.rlk_consistency_stats_async
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_size_t, ctypes.c_void_p]
    # one 64-byte block record per 256 elements, none for n <= 0
    assert L.rlk_consistency_stats_workspace_size(0) == 0
    assert L.rlk_consistency_stats_workspace_size(-3) == 0
    assert L.rlk_consistency_stats_workspace_size(1) == 64
    assert L.rlk_consistency_stats_workspace_size(256) == 64
    assert L.rlk_consistency_stats_workspace_size(257) == 128
    assert f(A16, A16, None, -1, A16, A16, 1 << 20, None) == 1          # n < 0
    assert f(A16, A16, None, 5, None, A16, 1 << 20, None) == 1          # no output
    assert f(A16, A16, None, 5, A4, A16, 1 << 20, None) == 2            # output not 8-aligned
    assert f(None, A16, None, 5, A16, A16, 1 << 20, None) == 1          # no input
    assert f(A16, A16, None, 5, A16, None, 1 << 20, None) == 5          # no workspace
    assert f(A16, A16, None, 5, A16, A16, 8, None) == 5                 # workspace too small
    assert f(A16, A16, None, 5, A16, A4, 1 << 20, None) == 2            # workspace misaligned


def test_valid_call_without_gpu_reports_device_error(L):
    """On a machine without a GB300 a well-formed call fails with a status,
    never silently computes on the CPU."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the gpu tests")
    assert _lp(L) == 3  # RLK_ERR_UNSUPPORTED_DEVICE
    f = ctypes.c_float(1.0)
    assert L.rlk_logprob_noalloc(A16, A16, A16, 4, 64, 100, f, A16, A16, A16, None) == 3
    assert L.rlk_check_device_error(None) == 3
    bits, rows = ctypes.c_uint32(5), ctypes.c_uint64(5)
    assert L.rlk_take_device_errors(None, ctypes.byref(bits), ctypes.byref(rows)) == 3
    assert (bits.value, rows.value) == (5, 5)  # left untouched


def test_binding_refuses_cpu_tensors():
    import torch
    h = torch.zeros(2, 8, dtype=torch.bfloat16)
    W = torch.zeros(4, 8, dtype=torch.bfloat16)
    tg = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        rlk.logprob(h, W, tg)
