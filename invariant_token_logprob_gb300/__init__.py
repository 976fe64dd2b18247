"""Batch-invariant selected-token logprob for GB300 (sm_103a).

Thin ctypes binding over the C ABI of ``librlk.so`` (declared in
``include/rlk.h``).  Functions here only marshal torch tensors into pointers,
sizes and the current CUDA stream; every step of the computation runs in the
library's CUDA kernels.  There is no CPU fallback: if the library is missing or
the device is not compute capability 10.3 the calls raise.

The library is loaded on first use, so ``invariant_token_logprob_gb300.inputs``
(synthetic data) can be imported without it.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

__all__ = ["RlkError", "lib", "logprob", "logprob_ws", "logprob_partials", "lse_merge",
           "consistency_stats", "workspace_size", "check_device_error", "take_device_errors", "vocab_tile", "row_tile",
           "logprob_backward", "backward_workspace_size", "backward_dz", "selected_token_logprob",
           "logprob_entropy", "entropy_workspace_size", "logprob_partials_shard",
           "lse_merge_sharded", "quantize_fp8_rows", "logprob_fp8", "fp8_workspace_size",
           "quantize_fp8_weight", "unpack_fp8_weight", "quantize_fp8_row_blocks",
           "quantize_fp8_weight_blocks", "logprob_fp8_block", "fp8_block_workspace_size", "consistency_stats_async",
           "stats_workspace_size", "stats_dict",
           "header_functions", "STAT_NAMES", "LIB_PATH", "HEADER_PATH"]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "librlk.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "rlk.h")

STAT_NAMES = ("max_abs", "mean_abs", "std_abs", "k3_mean", "sum_delta", "n_valid",
              "n_bit_mismatch", "first_mismatch")

_STATUS = {0: "RLK_OK", 1: "RLK_ERR_INVALID_ARG", 2: "RLK_ERR_ALIGNMENT",
           3: "RLK_ERR_UNSUPPORTED_DEVICE", 4: "RLK_ERR_CUDA", 5: "RLK_ERR_WORKSPACE",
           6: "RLK_ERR_TIMEOUT", 7: "RLK_ERR_TARGET_RANGE"}


class RlkError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        msg = _lib.rlk_status_string(int(status)).decode() if _lib is not None else _STATUS.get(status)
        super().__init__(f"{where}: {msg} (status {status})")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C-ABI library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (no CPU fallback exists)")
        L = ctypes.CDLL(LIB_PATH)
        P, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
        f32, st = ctypes.c_float, ctypes.c_int
        L.rlk_abi_version.restype = ctypes.c_int
        L.rlk_abi_version.argtypes = []
        L.rlk_status_string.restype = ctypes.c_char_p
        L.rlk_status_string.argtypes = [ctypes.c_int]
        L.rlk_row_tile.restype = ctypes.c_int
        L.rlk_row_tile.argtypes = []
        L.rlk_vocab_tile.restype = ctypes.c_int
        L.rlk_vocab_tile.argtypes = []
        L.rlk_logprob_workspace_size.restype = sz
        L.rlk_logprob_workspace_size.argtypes = [i64, i64, i64]
        L.rlk_logprob.restype = st
        L.rlk_logprob.argtypes = [P, P, P, i64, i64, i64, f32, P, P, P, P]
        L.rlk_logprob_ws.restype = st
        L.rlk_logprob_ws.argtypes = [P, P, P, i64, i64, i64, f32, P, P, P, P, sz, P]
        L.rlk_logprob_partials.restype = st
        L.rlk_logprob_partials.argtypes = [P, P, P, i64, i64, i64, f32, P, sz, P]
        L.rlk_lse_merge.restype = st
        L.rlk_lse_merge.argtypes = [P, P, i64, i64, P, P, P, P]
        L.rlk_consistency_stats.restype = st
        L.rlk_consistency_stats.argtypes = [P, P, P, i64, P, P]
        L.rlk_consistency_stats_workspace_size.restype = sz
        L.rlk_consistency_stats_workspace_size.argtypes = [i64]
        L.rlk_consistency_stats_async.restype = st
        L.rlk_consistency_stats_async.argtypes = [P, P, P, i64, P, P, sz, P]
        L.rlk_selftest_wait_timeout.restype = st
        L.rlk_selftest_wait_timeout.argtypes = [P, P, P, P, P]
        L.rlk_selftest_wait_timeout_pair.restype = st
        L.rlk_selftest_wait_timeout_pair.argtypes = [P, P, P, P, ctypes.c_int, P]
        L.rlk_check_device_error.restype = st
        L.rlk_check_device_error.argtypes = [P]
        L.rlk_take_device_errors.restype = st
        L.rlk_take_device_errors.argtypes = [P, P, P]
        L.rlk_shutdown.restype = st
        L.rlk_shutdown.argtypes = []
        L.rlk_logprob_partials_shard.restype = st
        L.rlk_logprob_partials_shard.argtypes = [P, P, P, i64, i64, i64, i64, i64, f32, P, sz, P]
        L.rlk_lse_merge_sharded.restype = st
        L.rlk_lse_merge_sharded.argtypes = [P, i64, i64, P, i64, i64, P, P, P, P]
        L.rlk_quantize_fp8_rows.restype = st
        L.rlk_quantize_fp8_rows.argtypes = [P, i64, i64, P, P, P]
        L.rlk_fp8_weight_bytes.restype = sz
        L.rlk_fp8_weight_bytes.argtypes = [i64, i64]
        L.rlk_quantize_fp8_weight.restype = st
        L.rlk_quantize_fp8_weight.argtypes = [P, i64, i64, P, P, P]
        L.rlk_logprob_fp8_workspace_size.restype = sz
        L.rlk_logprob_fp8_workspace_size.argtypes = [i64, i64, i64]
        L.rlk_logprob_fp8.restype = st
        L.rlk_logprob_fp8.argtypes = [P, P, P, P, i64, i64, i64, f32, P, P, P, P, sz, P]
        L.rlk_fp8_block_weight_scale_count.restype = sz
        L.rlk_fp8_block_weight_scale_count.argtypes = [i64, i64]
        L.rlk_quantize_fp8_row_blocks.restype = st
        L.rlk_quantize_fp8_row_blocks.argtypes = [P, i64, i64, P, P, P]
        L.rlk_quantize_fp8_weight_blocks.restype = st
        L.rlk_quantize_fp8_weight_blocks.argtypes = [P, i64, i64, P, P, P]
        L.rlk_logprob_fp8_block_workspace_size.restype = sz
        L.rlk_logprob_fp8_block_workspace_size.argtypes = [i64, i64, i64]
        L.rlk_logprob_fp8_block.restype = st
        L.rlk_logprob_fp8_block.argtypes = [P, P, P, P, i64, i64, i64, f32, P, P, P, P, sz, P]
        L.rlk_logprob_entropy_workspace_size.restype = sz
        L.rlk_logprob_entropy_workspace_size.argtypes = [i64, i64, i64]
        L.rlk_logprob_entropy.restype = st
        L.rlk_logprob_entropy.argtypes = [P, P, P, i64, i64, i64, f32, P, P, P, P, P, sz, P]
        L.rlk_logprob_backward_workspace_size.restype = sz
        L.rlk_logprob_backward_workspace_size.argtypes = [i64, i64, i64]
        L.rlk_logprob_backward_dz_ld.restype = sz
        L.rlk_logprob_backward_dz_ld.argtypes = [i64]
        L.rlk_logprob_backward.restype = st
        L.rlk_logprob_backward.argtypes = [P, P, P, P, P, i64, i64, i64, f32, P, P, ctypes.c_int,
                                           P, sz, P]
        _lib = L
    return _lib


def header_functions(path: str = HEADER_PATH) -> list:
    """Names of the functions include/rlk.h declares."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rlk_[a-z_0-9]+)\s*\(", text)))


def _check(status: int, where: str):
    if status != 0:
        raise RlkError(status, where)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name, ndim=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device (no CPU path exists)")
    if t.device.index != torch.cuda.current_device():
        # the library launches on the current device; a tensor elsewhere would be
        # read through a pointer that device cannot use
        raise ValueError(f"{name} is on {t.device}, not on the current device "
                         f"cuda:{torch.cuda.current_device()} (use torch.cuda.set_device)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")


def row_tile() -> int:
    return lib().rlk_row_tile()


def vocab_tile() -> int:
    return lib().rlk_vocab_tile()


def workspace_size(T: int, H: int, V: int) -> int:
    return lib().rlk_logprob_workspace_size(int(T), int(H), int(V))


def _check_inputs(h, W, targets):
    import torch
    _need(h, torch.bfloat16, "h", 2)
    _need(W, torch.bfloat16, "W", 2)
    _need(targets, torch.int32, "targets", 1)
    T, H = h.shape
    V, H2 = W.shape
    if H != H2 or targets.shape[0] != T:
        raise ValueError("shape mismatch: h [T,H], W [V,H], targets [T]")
    return T, H, V


def _outputs(T, device, out):
    import torch
    if out is None:
        return (torch.empty(T, dtype=torch.float32, device=device),
                torch.empty(T, dtype=torch.float32, device=device),
                torch.empty(T, dtype=torch.int32, device=device))
    lp, lse, am = out
    _need(lp, torch.float32, "out[0]", 1)
    _need(lse, torch.float32, "out[1]", 1)
    _need(am, torch.int32, "out[2]", 1)
    return lp, lse, am


def logprob(h, W, targets, inv_temp: float = 1.0, out=None, stream=None):
    """rlk_logprob: returns (logp f32[T], lse f32[T], argmax i32[T]) on h's device."""
    T, H, V = _check_inputs(h, W, targets)
    lp, lse, am = _outputs(T, h.device, out)
    _check(lib().rlk_logprob(_ptr(h), _ptr(W), _ptr(targets), T, H, V, ctypes.c_float(inv_temp),
                             _ptr(lp), _ptr(lse), _ptr(am), _stream(stream)), "rlk_logprob")
    return lp, lse, am


def logprob_ws(h, W, targets, workspace, inv_temp: float = 1.0, out=None, stream=None):
    """rlk_logprob_ws with a caller-owned uint8 CUDA workspace tensor."""
    import torch
    T, H, V = _check_inputs(h, W, targets)
    _need(workspace, torch.uint8, "workspace", 1)
    lp, lse, am = _outputs(T, h.device, out)
    _check(lib().rlk_logprob_ws(_ptr(h), _ptr(W), _ptr(targets), T, H, V, ctypes.c_float(inv_temp),
                                _ptr(lp), _ptr(lse), _ptr(am), _ptr(workspace),
                                workspace.numel(), _stream(stream)), "rlk_logprob_ws")
    return lp, lse, am


def logprob_partials(h, W, targets, inv_temp: float = 1.0, out=None, stream=None):
    """rlk_logprob_partials: returns a float32 tensor [T, NVT, 4] of {m, s, a-bits, zt}
    (view column 2 as int32 for the argmax)."""
    import torch
    T, H, V = _check_inputs(h, W, targets)
    nvt = (V + vocab_tile() - 1) // vocab_tile()
    if out is None:
        out = torch.empty((T, nvt, 4), dtype=torch.float32, device=h.device)
    _need(out, torch.float32, "out")
    _check(lib().rlk_logprob_partials(_ptr(h), _ptr(W), _ptr(targets), T, H, V,
                                      ctypes.c_float(inv_temp), _ptr(out),
                                      out.numel() * 4, _stream(stream)), "rlk_logprob_partials")
    return out


def lse_merge(partials, targets, V: int, out=None, stream=None):
    """rlk_lse_merge over a [T, NVT, 4] float32 partial tensor."""
    import torch
    _need(partials, torch.float32, "partials", 3)
    _need(targets, torch.int32, "targets", 1)
    T = partials.shape[0]
    nvt = (V + vocab_tile() - 1) // vocab_tile()
    if partials.shape[1] != nvt or partials.shape[2] != 4 or targets.shape[0] != T:
        raise ValueError("partials must be [T, ceil(V/vocab_tile), 4] and targets [T]")
    lp, lse, am = _outputs(T, partials.device, out)
    _check(lib().rlk_lse_merge(_ptr(partials), _ptr(targets), T, int(V), _ptr(lp), _ptr(lse),
                               _ptr(am), _stream(stream)), "rlk_lse_merge")
    return lp, lse, am


def consistency_stats(a, b, mask=None, stream=None):
    """rlk_consistency_stats (synchronous): a = train logp, b = rollout logp (f32 CUDA
    tensors), optional int8 mask; returns a dict keyed by STAT_NAMES."""
    import torch
    _need(a, torch.float32, "a", 1)
    _need(b, torch.float32, "b", 1)
    if a.shape != b.shape:
        raise ValueError("a and b must have the same shape")
    mp = None
    if mask is not None:
        _need(mask, torch.int8, "mask", 1)
        if mask.shape != a.shape:
            raise ValueError("mask must match a")
        mp = _ptr(mask)
    out = (ctypes.c_double * 8)()
    _check(lib().rlk_consistency_stats(_ptr(a), _ptr(b), mp, a.shape[0], out, _stream(stream)),
           "rlk_consistency_stats")
    return dict(zip(STAT_NAMES, list(out)))


def consistency_stats_async(a, b, mask=None, out=None, workspace=None, stream=None):
    """rlk_consistency_stats_async: the same statistics written, stream-ordered, into a
    float64 CUDA tensor of 8 (returned; pass `out` to reuse one).  No host sync and no
    allocation inside the library; read it with stats_dict() when needed."""
    import torch
    _need(a, torch.float32, "a", 1)
    _need(b, torch.float32, "b", 1)
    if a.shape != b.shape:
        raise ValueError("a and b must have the same shape")
    mp = None
    if mask is not None:
        _need(mask, torch.int8, "mask", 1)
        if mask.shape != a.shape:
            raise ValueError("mask must match a")
        mp = _ptr(mask)
    n = a.shape[0]
    if out is None:
        out = torch.empty(8, dtype=torch.float64, device=a.device)
    _need(out, torch.float64, "out", 1)
    if out.numel() < 8:
        raise ValueError("out must hold 8 doubles")
    need = lib().rlk_consistency_stats_workspace_size(n)
    if workspace is None:
        workspace = torch.empty(max(16, need), dtype=torch.uint8, device=a.device)
    _need(workspace, torch.uint8, "workspace", 1)
    _check(lib().rlk_consistency_stats_async(_ptr(a), _ptr(b), mp, n, _ptr(out), _ptr(workspace),
                                             workspace.numel(), _stream(stream)),
           "rlk_consistency_stats_async")
    return out


def stats_workspace_size(n: int) -> int:
    return lib().rlk_consistency_stats_workspace_size(int(n))


def stats_dict(out):
    """The 8 statistics of a consistency_stats_async result as a dict (synchronises)."""
    return dict(zip(STAT_NAMES, out.cpu().tolist()))


def check_device_error(stream=None):
    """Raise RlkError(RLK_ERR_TIMEOUT) if a device-side bounded wait ran out, or
    RlkError(RLK_ERR_TARGET_RANGE) if a merge saw a target >= V (synchronises)."""
    _check(lib().rlk_check_device_error(_stream(stream)), "rlk_check_device_error")


def take_device_errors(stream=None):
    """rlk_take_device_errors: read and clear the device's error records; returns
    (wait_error_bits, target_range_rows) (synchronises)."""
    bits = ctypes.c_uint32(0)
    rows = ctypes.c_uint64(0)
    _check(lib().rlk_take_device_errors(_stream(stream), ctypes.byref(bits), ctypes.byref(rows)),
           "rlk_take_device_errors")
    return int(bits.value), int(rows.value)


def backward_workspace_size(T: int, H: int, V: int) -> int:
    return lib().rlk_logprob_backward_workspace_size(int(T), int(H), int(V))


def backward_dz(workspace, T: int, V: int):
    """The bf16 [T, V] view of dz inside a backward workspace (row stride
    rlk_logprob_backward_dz_ld(V) elements)."""
    import torch
    ld = lib().rlk_logprob_backward_dz_ld(int(V))
    return workspace[:T * ld * 2].view(torch.bfloat16).view(T, ld)[:, :V]


def logprob_backward(h, W, targets, lse, grad_logp, inv_temp: float = 1.0, need_h: bool = True,
                     need_W: bool = True, grad_W=None, workspace=None, stream=None):
    """rlk_logprob_backward: returns (grad_h f32 [T,H] or None, grad_W f32 [V,H] or None,
    workspace).  Pass grad_W to accumulate into it.  dz (bf16 [T,V]) is left in the
    workspace afterwards: backward_dz(workspace, T, V)."""
    import torch
    T, H, V = _check_inputs(h, W, targets)
    _need(lse, torch.float32, "lse", 1)
    _need(grad_logp, torch.float32, "grad_logp", 1)
    gh = torch.empty((T, H), dtype=torch.float32, device=h.device) if need_h else None
    accumulate = grad_W is not None
    if need_W and grad_W is None:
        grad_W = torch.empty((V, H), dtype=torch.float32, device=h.device)
    if grad_W is not None:
        _need(grad_W, torch.float32, "grad_W", 2)
    if workspace is None:
        workspace = torch.empty(backward_workspace_size(T, H, V), dtype=torch.uint8, device=h.device)
    _need(workspace, torch.uint8, "workspace", 1)
    _check(lib().rlk_logprob_backward(
        _ptr(h), _ptr(W), _ptr(targets), _ptr(lse), _ptr(grad_logp), T, H, V,
        ctypes.c_float(inv_temp), _ptr(gh) if gh is not None else None,
        _ptr(grad_W) if (need_W or accumulate) else None, 1 if accumulate else 0,
        _ptr(workspace), workspace.numel(), _stream(stream)), "rlk_logprob_backward")
    return gh, (grad_W if (need_W or accumulate) else None), workspace


def _autograd_function():
    import torch

    class SelectedTokenLogprob(torch.autograd.Function):
        """logp = selected-token logprob; forward values from rlk_logprob (the
        batch-invariant kernel), gradients from rlk_logprob_backward."""

        @staticmethod
        def forward(ctx, h, W, targets, inv_temp):
            lp, lse, am = logprob(h, W, targets, inv_temp)
            ctx.save_for_backward(h, W, targets, lse)
            ctx.inv_temp = inv_temp
            return lp

        @staticmethod
        def backward(ctx, grad_lp):
            h, W, targets, lse = ctx.saved_tensors
            need_h, need_W = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
            if not (need_h or need_W):
                return None, None, None, None
            gh, gW, _ = logprob_backward(h, W, targets, lse, grad_lp.contiguous().float(),
                                         ctx.inv_temp, need_h=need_h, need_W=need_W)
            return (gh.to(h.dtype) if need_h else None, gW.to(W.dtype) if need_W else None,
                    None, None)

    return SelectedTokenLogprob


_SelectedTokenLogprob = None


def selected_token_logprob(h, W, targets, inv_temp: float = 1.0):
    """Differentiable selected-token logprob (torch autograd): the forward is the
    batch-invariant kernel, the backward recomputes the logits on the same tiles."""
    global _SelectedTokenLogprob
    if _SelectedTokenLogprob is None:
        _SelectedTokenLogprob = _autograd_function()
    return _SelectedTokenLogprob.apply(h, W, targets, inv_temp)


def entropy_workspace_size(T: int, H: int, V: int) -> int:
    return lib().rlk_logprob_entropy_workspace_size(int(T), int(H), int(V))


def logprob_entropy(h, W, targets, inv_temp: float = 1.0, workspace=None, stream=None):
    """rlk_logprob_entropy: returns (logp, lse, argmax, entropy)."""
    import torch
    T, H, V = _check_inputs(h, W, targets)
    lp, lse, am = _outputs(T, h.device, None)
    ent = torch.empty(T, dtype=torch.float32, device=h.device)
    if workspace is None:
        workspace = torch.empty(max(1, entropy_workspace_size(T, H, V)), dtype=torch.uint8,
                                device=h.device)
    _need(workspace, torch.uint8, "workspace", 1)
    _check(lib().rlk_logprob_entropy(_ptr(h), _ptr(W), _ptr(targets), T, H, V,
                                     ctypes.c_float(inv_temp), _ptr(lp), _ptr(lse), _ptr(am),
                                     _ptr(ent), _ptr(workspace), workspace.numel(),
                                     _stream(stream)), "rlk_logprob_entropy")
    return lp, lse, am, ent


def logprob_partials_shard(h, W_shard, targets, V: int, shard_begin: int, inv_temp: float = 1.0,
                           out=None, stream=None):
    """rlk_logprob_partials_shard: partials [T, ceil(rows/vocab_tile), 4] of one
    vocabulary shard W_shard = W[shard_begin : shard_begin + rows]."""
    import torch
    _need(h, torch.bfloat16, "h", 2)
    _need(W_shard, torch.bfloat16, "W_shard", 2)
    _need(targets, torch.int32, "targets", 1)
    T, H = h.shape
    rows = W_shard.shape[0]
    nvt_s = (rows + vocab_tile() - 1) // vocab_tile()
    if out is None:
        out = torch.empty((T, nvt_s, 4), dtype=torch.float32, device=h.device)
    _need(out, torch.float32, "out")
    _check(lib().rlk_logprob_partials_shard(_ptr(h), _ptr(W_shard), _ptr(targets), T, H, int(V),
                                            int(shard_begin), rows, ctypes.c_float(inv_temp),
                                            _ptr(out), out.numel() * 4, _stream(stream)),
           "rlk_logprob_partials_shard")
    return out


def lse_merge_sharded(partials, targets, V: int, out=None, stream=None):
    """rlk_lse_merge_sharded over gathered partials [R, T, tiles_per_shard, 4]."""
    import torch
    _need(partials, torch.float32, "partials", 4)
    _need(targets, torch.int32, "targets", 1)
    R, T, nvt_s, four = partials.shape
    if four != 4 or targets.shape[0] != T:
        raise ValueError("partials must be [R, T, tiles_per_shard, 4] and targets [T]")
    lp, lse, am = _outputs(T, partials.device, out)
    _check(lib().rlk_lse_merge_sharded(_ptr(partials), R, nvt_s, _ptr(targets), T, int(V),
                                       _ptr(lp), _ptr(lse), _ptr(am), _stream(stream)),
           "rlk_lse_merge_sharded")
    return lp, lse, am


def quantize_fp8_rows(x, stream=None):
    """rlk_quantize_fp8_rows: bf16 [rows, H] -> (e4m3 codes as uint8 [rows, H], f32 scales [rows])."""
    import torch
    _need(x, torch.bfloat16, "x", 2)
    rows, H = x.shape
    codes = torch.empty((rows, H), dtype=torch.uint8, device=x.device)
    scales = torch.empty(rows, dtype=torch.float32, device=x.device)
    _check(lib().rlk_quantize_fp8_rows(_ptr(x), rows, H, _ptr(codes), _ptr(scales),
                                       _stream(stream)), "rlk_quantize_fp8_rows")
    return codes, scales


def fp8_workspace_size(T: int, H: int, V: int) -> int:
    return lib().rlk_logprob_fp8_workspace_size(int(T), int(H), int(V))


def quantize_fp8_weight(W, out=None, stream=None):
    """rlk_quantize_fp8_weight: bf16 W [V, H] -> (tile-packed e4m3 codes as a flat uint8
    tensor, f32 scales [V]).  Pass out=(packed, scales) to reuse buffers."""
    import torch
    _need(W, torch.bfloat16, "W", 2)
    V, H = W.shape
    if out is None:
        packed = torch.empty(lib().rlk_fp8_weight_bytes(V, H), dtype=torch.uint8, device=W.device)
        scales = torch.empty(V, dtype=torch.float32, device=W.device)
    else:
        packed, scales = out
        _need(packed, torch.uint8, "packed", 1)
        _need(scales, torch.float32, "scales", 1)
        if packed.numel() < lib().rlk_fp8_weight_bytes(V, H) or scales.numel() < V:
            raise ValueError("out buffers too small for rlk_fp8_weight_bytes(V, H) / V")
    _check(lib().rlk_quantize_fp8_weight(_ptr(W), V, H, _ptr(packed), _ptr(scales),
                                         _stream(stream)), "rlk_quantize_fp8_weight")
    return packed, scales


def unpack_fp8_weight(packed, V: int, H: int):
    """Row-major [V, H] copy of a tile-packed fp8 weight (for inspection)."""
    bn = vocab_tile()
    nt = (V + bn - 1) // bn
    x = packed.view(nt, H // 128, bn, 128).permute(0, 2, 1, 3).reshape(nt * bn, H)
    return x[:V]


def logprob_fp8(h, W_packed, W_scales, targets, inv_temp: float = 1.0, workspace=None, out=None,
                stream=None):
    """rlk_logprob_fp8: (logp, lse, argmax) from bf16 h and a tile-packed e4m3 W
    (from quantize_fp8_weight); V = len(W_scales)."""
    import torch
    _need(h, torch.bfloat16, "h", 2)
    _need(W_packed, torch.uint8, "W_packed", 1)
    _need(W_scales, torch.float32, "W_scales", 1)
    _need(targets, torch.int32, "targets", 1)
    T, H = h.shape
    V = W_scales.shape[0]
    if W_packed.numel() < lib().rlk_fp8_weight_bytes(V, H) or targets.shape[0] != T:
        raise ValueError("W_packed must hold rlk_fp8_weight_bytes(V, H) bytes; targets [T]")
    lp, lse, am = _outputs(T, h.device, out)
    if workspace is None:
        workspace = torch.empty(max(1, fp8_workspace_size(T, H, V)), dtype=torch.uint8,
                                device=h.device)
    _need(workspace, torch.uint8, "workspace", 1)
    _check(lib().rlk_logprob_fp8(_ptr(h), _ptr(W_packed), _ptr(W_scales), _ptr(targets), T, H, V,
                                 ctypes.c_float(inv_temp), _ptr(lp), _ptr(lse), _ptr(am),
                                 _ptr(workspace), workspace.numel(), _stream(stream)),
           "rlk_logprob_fp8")
    return lp, lse, am


def quantize_fp8_row_blocks(x, stream=None):
    """rlk_quantize_fp8_row_blocks: bf16 [rows, H] -> (e4m3 codes uint8 [rows, H], f32
    scales [rows, H/128]) in 1 x 128 blocks."""
    import torch
    _need(x, torch.bfloat16, "x", 2)
    rows, H = x.shape
    codes = torch.empty((rows, H), dtype=torch.uint8, device=x.device)
    scales = torch.empty((rows, max(1, H // 128)), dtype=torch.float32, device=x.device)
    _check(lib().rlk_quantize_fp8_row_blocks(_ptr(x), rows, H, _ptr(codes), _ptr(scales),
                                             _stream(stream)), "rlk_quantize_fp8_row_blocks")
    return codes, scales


def quantize_fp8_weight_blocks(W, out=None, stream=None):
    """rlk_quantize_fp8_weight_blocks: bf16 W [V, H] -> (tile-packed e4m3 codes, flat
    uint8; f32 scales [ceil(V/128), H/128]) in 128 x 128 blocks."""
    import torch
    _need(W, torch.bfloat16, "W", 2)
    V, H = W.shape
    if out is None:
        packed = torch.empty(lib().rlk_fp8_weight_bytes(V, H), dtype=torch.uint8, device=W.device)
        scales = torch.empty(((V + 127) // 128, max(1, H // 128)), dtype=torch.float32,
                             device=W.device)
    else:
        packed, scales = out
        _need(packed, torch.uint8, "packed", 1)
        _need(scales, torch.float32, "scales")
        if (packed.numel() < lib().rlk_fp8_weight_bytes(V, H) or
                scales.numel() < lib().rlk_fp8_block_weight_scale_count(V, H)):
            raise ValueError("out buffers too small")
    _check(lib().rlk_quantize_fp8_weight_blocks(_ptr(W), V, H, _ptr(packed), _ptr(scales),
                                                _stream(stream)), "rlk_quantize_fp8_weight_blocks")
    return packed, scales


def fp8_block_workspace_size(T: int, H: int, V: int) -> int:
    return lib().rlk_logprob_fp8_block_workspace_size(int(T), int(H), int(V))


def logprob_fp8_block(h, W_packed, W_scales, targets, V: int, inv_temp: float = 1.0,
                      workspace=None, out=None, stream=None):
    """rlk_logprob_fp8_block: (logp, lse, argmax) from bf16 h and a block-quantised
    tile-packed e4m3 W with its [ceil(V/128), H/128] block scales."""
    import torch
    _need(h, torch.bfloat16, "h", 2)
    _need(W_packed, torch.uint8, "W_packed", 1)
    _need(W_scales, torch.float32, "W_scales")
    _need(targets, torch.int32, "targets", 1)
    T, H = h.shape
    if (W_packed.numel() < lib().rlk_fp8_weight_bytes(V, H) or targets.shape[0] != T or
            W_scales.numel() < lib().rlk_fp8_block_weight_scale_count(V, H)):
        raise ValueError("W_packed / W_scales too small for (V, H), or targets not [T]")
    lp, lse, am = _outputs(T, h.device, out)
    if workspace is None:
        workspace = torch.empty(max(1, fp8_block_workspace_size(T, H, V)), dtype=torch.uint8,
                                device=h.device)
    _need(workspace, torch.uint8, "workspace", 1)
    _check(lib().rlk_logprob_fp8_block(_ptr(h), _ptr(W_packed), _ptr(W_scales), _ptr(targets), T,
                                       H, int(V), ctypes.c_float(inv_temp), _ptr(lp), _ptr(lse),
                                       _ptr(am), _ptr(workspace), workspace.numel(),
                                       _stream(stream)), "rlk_logprob_fp8_block")
    return lp, lse, am
