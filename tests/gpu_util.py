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


def assert_block_records(P, bs, h, W, bn, inv_temp=1.0, j0=0, what=""):
    """Per-(row, vocabulary tile) records {m, s, a, zt} of the CUDA path, P
    [T, ntiles, 4] float32 for global tiles j0 .. j0 + ntiles - 1, against the
    oracle's per-block statistics bs (oracle.block_stats over the whole V).
    m, s, zt within 1e-5 relative; a exact wherever the tile's largest logit is
    clear of its runner-up by more than 1e-3 (h, W: bf16 CPU tensors, used only
    to find those tiles)."""
    m, s = P[..., 0].astype(np.float64), P[..., 1].astype(np.float64)
    a, zt = P[..., 2].view(np.int32), P[..., 3].astype(np.float64)
    nt = m.shape[1]
    sl = slice(j0, j0 + nt)
    bm, bsum, bzt, ba = bs["m"][:, sl], bs["s"][:, sl], bs["zt"][:, sl], bs["a"][:, sl]
    assert m.shape == bm.shape, (what, m.shape, bm.shape)
    assert np.all(np.abs(m - bm) <= 1e-5 * np.maximum(1, np.abs(bm))), f"{what}: m"
    assert np.all(np.abs(s - bsum) <= 1e-5 * bsum), f"{what}: s"
    assert np.all(np.abs(zt - bzt) <= 1e-5 * np.maximum(1, np.abs(bzt))), f"{what}: zt"
    V = W.shape[0]
    z = (h.double() @ W.double().T).numpy() * float(np.float32(inv_temp))
    for j in range(nt):
        g = j0 + j
        zz = np.sort(z[:, g * bn:min(V, (g + 1) * bn)], axis=1)
        clear = (zz[:, -1] - zz[:, -2] > 1e-3) if zz.shape[1] > 1 else np.ones(z.shape[0], bool)
        assert np.array_equal(a[clear, j], ba[clear, j]), f"{what}: a of tile {g}"
