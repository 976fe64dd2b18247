"""Shared helpers of the GPU tests: run the CUDA path through the binding and
compare it with the oracle under the tolerances of the numerical contract.

Tolerances (written here once, used by every parity test):
  |logp_gpu - logp_oracle| <= 5e-4                     (absolute)
  |lse_gpu  - lse_oracle|  <= 1e-5 * max(1, |lse|)     (relative; absolute near 0)
  argmax exact wherever the oracle's top-2 logit gap exceeds 1e-3
Invariance checks are bitwise (uint32 views of logp / lse, int32 argmax).
"""
import numpy as np
import torch

LOGP_ATOL = 5e-4
LSE_RTOL = 1e-5
GAP_SURE = 1e-3


def to_dev(d, dev="cuda"):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def gpu_logprob(h, W, tg, inv_temp=1.0):
    import invariant_token_logprob_gb300 as rlk
    lp, lse, am = rlk.logprob(h, W, tg, inv_temp)
    rlk.check_device_error()
    return lp.cpu().numpy(), lse.cpu().numpy(), am.cpu().numpy()


def assert_parity(gpu, ref, rows=None, what=""):
    lp, lse, am = gpu
    if rows is not None:
        lp, lse, am = lp[rows], lse[rows], am[rows]
    dlp = np.abs(lp.astype(np.float64) - ref["logp"])
    dlse = np.abs(lse.astype(np.float64) - ref["lse"])
    assert np.all(np.isfinite(lp)) and np.all(np.isfinite(lse)), f"{what}: non-finite output"
    assert dlp.max() <= LOGP_ATOL, f"{what}: max |dlogp| {dlp.max():.3g} at {dlp.argmax()}"
    lim = LSE_RTOL * np.maximum(1.0, np.abs(ref["lse"]))
    assert np.all(dlse <= lim), f"{what}: lse rel err {np.max(dlse / lim) * LSE_RTOL:.3g}"
    sure = ref["top2gap"] > GAP_SURE
    bad = np.nonzero(sure & (am != ref["argmax"]))[0]
    assert bad.size == 0, f"{what}: argmax mismatch at rows {bad[:10]}"
    return dict(max_dlogp=float(dlp.max()), max_dlse=float(dlse.max()))


def bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x).view(np.uint32 if x.dtype == np.float32 else x.dtype)


def assert_bitwise(a, b, what=""):
    for name, x, y in zip(("logp", "lse", "argmax"), a, b):
        bx, by = bits(x), bits(y)
        n = int(np.count_nonzero(bx != by))
        assert n == 0, f"{what}: {n} bitwise mismatches in {name}"
