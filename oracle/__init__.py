"""fp64 CPU oracle for the selected-token logprob -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline / reference
arm import this package.  The product library never does, and the two share no
code: this module only marshals numpy arrays into ``liboracle.so`` (built from
``oracle.c`` by :func:`build`).

Every function here is a thin ctypes wrapper; the arithmetic, and the passages
of the pages it follows, live in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(out_path: str = _LIB_PATH, mutant: int = 0, quiet: bool = True) -> str:
    """Compile oracle.c with gcc into a shared library and return its path.

    ``mutant`` > 0 plants one of the deliberate mistakes listed in oracle.c
    (used only by the test that shows the pins catch them).
    """
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", f"-DORACLE_MUTANT={int(mutant)}",
           "-o", out_path, _SRC, "-lm"]
    subprocess.run(cmd, check=True, capture_output=quiet)
    return out_path


def _bind(lib):
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_logprob.restype = ctypes.c_int
    lib.oracle_logprob.argtypes = [P, P, P, i64, i64, i64, ctypes.c_float, P, i64,
                                   P, P, P, P, P, P]
    lib.oracle_block_stats.restype = ctypes.c_int
    lib.oracle_block_stats.argtypes = [P, P, P, i64, i64, i64, ctypes.c_float, i64, P, i64,
                                       P, P, P, P]
    lib.oracle_merge_blocks.restype = ctypes.c_int
    lib.oracle_merge_blocks.argtypes = [P, P, P, P, P, i64, i64, i64, i64, P, P, P]
    lib.oracle_consistency_stats.restype = ctypes.c_int
    lib.oracle_consistency_stats.argtypes = [P, P, P, i64, P]
    lib.oracle_logprob_backward.restype = ctypes.c_int
    lib.oracle_logprob_backward.argtypes = [P, P, P, P, i64, i64, i64, ctypes.c_float, P, P, P]
    lib.oracle_entropy.restype = ctypes.c_int
    lib.oracle_entropy.argtypes = [P, P, i64, i64, i64, ctypes.c_float, P, i64, P]
    lib.oracle_quantize_fp8_rows.restype = ctypes.c_int
    lib.oracle_quantize_fp8_rows.argtypes = [P, i64, i64, P, P]
    lib.oracle_logprob_fp8.restype = ctypes.c_int
    lib.oracle_logprob_fp8.argtypes = [P, P, P, P, P, i64, i64, i64, ctypes.c_float, P, i64,
                                       P, P, P, P]
    lib.oracle_quantize_fp8_blocks.restype = ctypes.c_int
    lib.oracle_quantize_fp8_blocks.argtypes = [P, i64, i64, i64, P, P]
    lib.oracle_logprob_fp8_block.restype = ctypes.c_int
    lib.oracle_logprob_fp8_block.argtypes = [P, P, P, P, P, i64, i64, i64, ctypes.c_float, P, i64,
                                             P, P, P, P]
    lib.oracle_logprob_f64.restype = ctypes.c_int
    lib.oracle_logprob_f64.argtypes = [P, P, P, i64, i64, i64, ctypes.c_double, P, P]
    return lib


def load(path: Optional[str] = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if (not os.path.exists(_LIB_PATH)
                or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
            build()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _u16(x) -> np.ndarray:
    """bf16 bit patterns as a C-contiguous uint16 array (accepts torch bf16 tensors)."""
    if hasattr(x, "view") and hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch  # local: torch only used for the bit view
        x = x.detach().cpu().contiguous().view(torch.int16).numpy()
    a = np.ascontiguousarray(np.asarray(x))
    if a.dtype != np.uint16:
        a = a.view(np.uint16) if a.dtype == np.int16 else a.astype(np.uint16)
    return a


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def num_threads(lib=None) -> int:
    return (lib or load()).oracle_num_threads()


def logprob(h, W, targets, inv_temp: float = 1.0, rows=None, lib=None) -> dict:
    """Oracle selected-token logprob.

    h: [T,H] bf16 bits (uint16 / int16 numpy or torch bf16), W: [V,H] likewise,
    targets: [T] int32.  rows: optional list of row indices to evaluate.
    Returns dict of numpy arrays (one entry per evaluated row): logp, lse
    (float64), argmax (int64), top2gap, ztgt, zmax (float64).
    """
    lib = lib or load()
    h = _u16(h)
    W = _u16(W)
    tg = _i32(targets)
    T, H = h.shape
    V, H2 = W.shape
    assert H == H2 and tg.shape == (T,)
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = T if r is None else r.shape[0]
    out = {k: np.zeros(n, dtype=np.float64) for k in ("logp", "lse", "top2gap", "ztgt", "zmax")}
    out["argmax"] = np.zeros(n, dtype=np.int64)
    rc = lib.oracle_logprob(_ptr(h), _ptr(W), _ptr(tg), T, H, V, ctypes.c_float(inv_temp),
                            _ptr(r), n, _ptr(out["logp"]), _ptr(out["lse"]),
                            _ptr(out["argmax"]), _ptr(out["top2gap"]), _ptr(out["ztgt"]),
                            _ptr(out["zmax"]))
    if rc != 0:
        raise ValueError("oracle_logprob rejected its arguments")
    return out


def block_stats(h, W, targets, bn: int, inv_temp: float = 1.0, rows=None, lib=None) -> dict:
    """Per-vocabulary-block (m, s, a, zt) statistics, shape [n_rows, ceil(V/bn)]."""
    lib = lib or load()
    h = _u16(h)
    W = _u16(W)
    tg = _i32(targets)
    T, H = h.shape
    V = W.shape[0]
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = T if r is None else r.shape[0]
    nb = (V + bn - 1) // bn
    out = {"m": np.zeros((n, nb)), "s": np.zeros((n, nb)), "zt": np.zeros((n, nb)),
           "a": np.zeros((n, nb), dtype=np.int64)}
    rc = lib.oracle_block_stats(_ptr(h), _ptr(W), _ptr(tg), T, H, V, ctypes.c_float(inv_temp),
                                bn, _ptr(r), n, _ptr(out["m"]), _ptr(out["s"]),
                                _ptr(out["a"]), _ptr(out["zt"]))
    if rc != 0:
        raise ValueError("oracle_block_stats rejected its arguments")
    return out


def merge_blocks(m, s, a, zt, targets, V: int, bn: int, lib=None) -> dict:
    """fp64 merge of fp32 per-block statistics ([n_rows, n_blocks] each)."""
    lib = lib or load()
    m = np.ascontiguousarray(m, dtype=np.float32)
    s = np.ascontiguousarray(s, dtype=np.float32)
    a = np.ascontiguousarray(a, dtype=np.int32)
    zt = None if zt is None else np.ascontiguousarray(zt, dtype=np.float32)
    tg = None if targets is None else _i32(targets)
    n, nb = m.shape
    out = {"lse": np.zeros(n), "logp": np.zeros(n), "argmax": np.zeros(n, dtype=np.int64)}
    rc = lib.oracle_merge_blocks(_ptr(m), _ptr(s), _ptr(a), _ptr(zt), _ptr(tg), n, nb, V, bn,
                                 _ptr(out["lse"]), _ptr(out["logp"]), _ptr(out["argmax"]))
    if rc != 0:
        raise ValueError("oracle_merge_blocks rejected its arguments")
    return out


STAT_NAMES = ("max_abs", "mean_abs", "std_abs", "k3_mean", "sum_delta", "n_valid",
              "n_bit_mismatch", "first_mismatch")


def consistency_stats(a, b, mask=None, lib=None) -> np.ndarray:
    """Acceptance statistics (8 doubles, order as STAT_NAMES); a = train, b = rollout."""
    lib = lib or load()
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    if hasattr(b, "detach"):
        b = b.detach().cpu().numpy()
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    assert a.shape == b.shape and a.ndim == 1
    mk = None
    if mask is not None:
        if hasattr(mask, "detach"):
            mask = mask.detach().cpu().numpy()
        mk = np.ascontiguousarray(mask, dtype=np.int8)
        assert mk.shape == a.shape
    out = np.zeros(8, dtype=np.float64)
    rc = lib.oracle_consistency_stats(_ptr(a), _ptr(b), _ptr(mk), a.shape[0], _ptr(out))
    if rc != 0:
        raise ValueError("oracle_consistency_stats rejected its arguments")
    return out


def logprob_backward(h, W, targets, grad, inv_temp: float = 1.0, lib=None) -> dict:
    """fp64 gradients of logp w.r.t. the logits, h and W: dict(dz [T,V], dh [T,H],
    dW [V,H]) for upstream gradient `grad` [T] (small problems only)."""
    lib = lib or load()
    h = _u16(h)
    W = _u16(W)
    tg = _i32(targets)
    g = np.ascontiguousarray(np.asarray(grad.detach().cpu().numpy() if hasattr(grad, "detach")
                                        else grad, dtype=np.float64))
    T, H = h.shape
    V = W.shape[0]
    out = {"dz": np.zeros((T, V)), "dh": np.zeros((T, H)), "dW": np.zeros((V, H))}
    rc = lib.oracle_logprob_backward(_ptr(h), _ptr(W), _ptr(tg), _ptr(g), T, H, V,
                                     ctypes.c_float(inv_temp), _ptr(out["dz"]), _ptr(out["dh"]),
                                     _ptr(out["dW"]))
    if rc != 0:
        raise ValueError("oracle_logprob_backward rejected its arguments")
    return out


def logprob_f64(h, W, targets, inv_temp: float = 1.0, lib=None) -> dict:
    """Forward on fp64 inputs (h [T,H], W [V,H] float64): dict(logp, lse)."""
    lib = lib or load()
    h = np.ascontiguousarray(h, dtype=np.float64)
    W = np.ascontiguousarray(W, dtype=np.float64)
    tg = _i32(targets)
    T, H = h.shape
    V = W.shape[0]
    out = {"logp": np.zeros(T), "lse": np.zeros(T)}
    rc = lib.oracle_logprob_f64(_ptr(h), _ptr(W), _ptr(tg), T, H, V, float(inv_temp),
                                _ptr(out["logp"]), _ptr(out["lse"]))
    if rc != 0:
        raise ValueError("oracle_logprob_f64 rejected its arguments")
    return out


def entropy(h, W, inv_temp: float = 1.0, rows=None, lib=None) -> np.ndarray:
    """Per-token softmax entropy over the whole vocabulary (fp64), one per row."""
    lib = lib or load()
    h = _u16(h)
    W = _u16(W)
    T, H = h.shape
    V = W.shape[0]
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = T if r is None else r.shape[0]
    out = np.zeros(n)
    rc = lib.oracle_entropy(_ptr(h), _ptr(W), T, H, V, ctypes.c_float(inv_temp), _ptr(r), n,
                            _ptr(out))
    if rc != 0:
        raise ValueError("oracle_entropy rejected its arguments")
    return out


def quantize_fp8_rows(x, lib=None):
    """Per-row e4m3 quantisation of a bf16 matrix: (codes uint8 [rows,H], scales f32 [rows])."""
    lib = lib or load()
    x = _u16(x)
    rows, H = x.shape
    codes = np.zeros((rows, H), dtype=np.uint8)
    scales = np.zeros(rows, dtype=np.float32)
    rc = lib.oracle_quantize_fp8_rows(_ptr(x), rows, H, _ptr(codes), _ptr(scales))
    if rc != 0:
        raise ValueError("oracle_quantize_fp8_rows rejected its arguments")
    return codes, scales


def logprob_fp8(qh, sh, qw, sw, targets, inv_temp: float = 1.0, rows=None, lib=None) -> dict:
    """Selected-token logprob from e4m3 codes and per-row scales (fp64)."""
    lib = lib or load()
    qh = np.ascontiguousarray(qh, dtype=np.uint8)
    qw = np.ascontiguousarray(qw, dtype=np.uint8)
    sh = np.ascontiguousarray(sh, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    tg = _i32(targets)
    T, H = qh.shape
    V = qw.shape[0]
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = T if r is None else r.shape[0]
    out = {k: np.zeros(n) for k in ("logp", "lse", "top2gap")}
    out["argmax"] = np.zeros(n, dtype=np.int64)
    rc = lib.oracle_logprob_fp8(_ptr(qh), _ptr(sh), _ptr(qw), _ptr(sw), _ptr(tg), T, H, V,
                                ctypes.c_float(inv_temp), _ptr(r), n, _ptr(out["logp"]),
                                _ptr(out["lse"]), _ptr(out["argmax"]), _ptr(out["top2gap"]))
    if rc != 0:
        raise ValueError("oracle_logprob_fp8 rejected its arguments")
    return out


def quantize_fp8_blocks(x, block_rows: int, lib=None):
    """Block e4m3 quantisation of bf16 bits [rows, H] in block_rows x 128 blocks:
    returns (codes uint8 [rows, H], scales float32 [ceil(rows/block_rows), ceil(H/128)])."""
    lib = lib or load()
    x = _u16(x)
    rows, H = x.shape
    nkb = (H + 127) // 128
    nrb = (rows + block_rows - 1) // block_rows
    codes = np.zeros((rows, H), dtype=np.uint8)
    scales = np.zeros((nrb, nkb), dtype=np.float32)
    if lib.oracle_quantize_fp8_blocks(_ptr(x), rows, H, int(block_rows), _ptr(codes),
                                      _ptr(scales)) != 0:
        raise ValueError("oracle_quantize_fp8_blocks rejected its arguments")
    return codes, scales


def logprob_fp8_block(qh, sh, qw, sw, targets, inv_temp: float = 1.0, rows=None, lib=None) -> dict:
    """Oracle logprob from block-quantised operands: qh [T,H] / sh [T, ceil(H/128)]
    (1 x 128 blocks), qw [V,H] / sw [ceil(V/128), ceil(H/128)] (128 x 128 blocks)."""
    lib = lib or load()
    qh = np.ascontiguousarray(qh, dtype=np.uint8)
    qw = np.ascontiguousarray(qw, dtype=np.uint8)
    sh = np.ascontiguousarray(sh, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    tg = _i32(targets)
    T, H = qh.shape
    V = qw.shape[0]
    nkb = (H + 127) // 128
    assert qw.shape[1] == H and sh.shape == (T, nkb) and sw.shape == ((V + 127) // 128, nkb)
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = T if r is None else r.shape[0]
    out = {k: np.zeros(n, dtype=np.float64) for k in ("logp", "lse", "top2gap")}
    out["argmax"] = np.zeros(n, dtype=np.int64)
    if lib.oracle_logprob_fp8_block(_ptr(qh), _ptr(sh), _ptr(qw), _ptr(sw), _ptr(tg), T, H, V,
                                    ctypes.c_float(inv_temp), _ptr(r), n, _ptr(out["logp"]),
                                    _ptr(out["lse"]), _ptr(out["argmax"]),
                                    _ptr(out["top2gap"])) != 0:
        raise ValueError("oracle_logprob_fp8_block rejected its arguments")
    return out
