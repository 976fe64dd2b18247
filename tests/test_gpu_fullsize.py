"""GPU tests at the full workload sizes (H=4096/5120, V=151936), in the launch
configuration the benchmark times.  Oracle parity: every row of the T=4096
training batch, every row of the 256-row decode pool, 2048 seeded rows of the
T=16384 prefill batch, and every outlier row plus 2048 seeded other rows of
the T=32768 / H=5120 batch.  The fp64 oracle costs about 0.4 core-seconds per
row at H=4096, so it runs on the host cores in a background thread (ctypes
releases the interpreter lock) while the GPU checks of the same test run.  The
numerical contract -- a row's bits independent of T, batch position,
chunking, phase and repetition -- is checked bitwise on every row.

Workloads (seeded, synthetic; stand-ins for a Qwen3-8B LM head):
  training recompute   T=4096 (8 packed x 512), H=4096, RMS-normalised hidden
  decode sweep         a pool of 256 rows evaluated at every batch size 1..256
                       in shuffled compositions (2 sweeps, different shuffles)
  prefill vs decode    4 x 4096 = 16384 rows, inv_temp = fp32(1/0.7): one call,
                       chunks of 512, chunks of 64, token by token
  large packed batch   T=32768, H=5120, 1% outlier rows x8, 10% of tokens
                       masked out of the statistics
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bitwise, assert_parity, gpu_logprob
from invariant_token_logprob_gb300.inputs import lm_head_inputs

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
V = 151936


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import invariant_token_logprob_gb300 as rlk
    rlk.lib()
    yield
    torch.cuda.empty_cache()


def _sample_rows(T, n, seed, must=()):
    g = np.random.default_rng(seed)
    rows = set(int(x) for x in g.choice(T, size=min(n, T), replace=False))
    rows.update(int(x) for x in must)
    return np.array(sorted(rows), dtype=np.int64)


_POOL = ThreadPoolExecutor(max_workers=1)


def _oracle(d, rows, inv_temp, olib):
    """Start the oracle on `rows` (None: every row) of the inputs; returns a
    future.  The inputs are copied to the host here, before any GPU work of the
    caller changes them."""
    h, W, tg = d["h"].cpu(), d["W"].cpu(), d["targets"].cpu()
    return _POOL.submit(oracle.logprob, h, W, tg, inv_temp, rows=rows, lib=olib)


def _concat(parts):
    return tuple(np.concatenate([p[k] for p in parts]) for k in range(3))


def test_training_recompute_T4096(olib):
    T, H = 4096, 4096
    d = lm_head_inputs(T, H, V, seed=0, device="cuda")
    h, W, tg = d["h"], d["W"], d["targets"]
    ref = _oracle(d, None, 1.0, olib)  # every row
    full = gpu_logprob(h, W, tg)
    # per-sequence calls (8 x 512) -- the packed batch split into its sequences
    seq = _concat([gpu_logprob(h[i:i + 512].contiguous(), W, tg[i:i + 512].contiguous())
                   for i in range(0, T, 512)])
    assert_bitwise(full, seq, "8 x 512 vs packed 4096")
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(3)).cuda()
    pg = gpu_logprob(h[perm].contiguous(), W, tg[perm].contiguous())
    inv = torch.argsort(perm).cpu().numpy()
    assert_bitwise(full, tuple(x[inv] for x in pg), "permuted rows")
    assert_bitwise(full, gpu_logprob(h, W, tg), "repeat")
    assert_parity(full, ref.result(), what="T=4096, every row")


def test_decode_batch_sweep(olib):
    """Every row of a 256-row pool, at every batch size 1..256 in shuffled
    compositions (32,896 row evaluations per sweep, two sweeps), is bit-identical
    to its value in the B=256 call."""
    P, H = 256, 4096
    d = lm_head_inputs(P, H, V, seed=2, device="cuda")
    h, W, tg = d["h"], d["W"], d["targets"]
    oref = _oracle(d, None, 1.0, olib)  # every pool row
    ref = gpu_logprob(h, W, tg)
    evaluations = 0
    for sweep in range(2):
        for B in range(1, P + 1):
            g = torch.Generator().manual_seed(10_000 * (sweep + 1) + B)
            sel = torch.randperm(P, generator=g)[:B]
            got = gpu_logprob(h[sel.cuda()].contiguous(), W, tg[sel.cuda()].contiguous())
            s = sel.numpy()
            assert_bitwise(tuple(x[s] for x in ref), got, f"sweep {sweep} B={B}")
            evaluations += B
    assert evaluations == 2 * P * (P + 1) // 2
    assert_parity(ref, oref.result(), what="pool, every row")


def test_prefill_vs_decode_phase_consistency(olib):
    import invariant_token_logprob_gb300 as rlk
    T, H = 4 * 4096, 4096
    it = float(np.float32(1.0 / 0.7))
    d = lm_head_inputs(T, H, V, seed=4, device="cuda")
    h, W, tg = d["h"], d["W"], d["targets"]
    rows = _sample_rows(T, 2048, 6, must=(0, 4095, 4096, T - 1))
    ref = _oracle(d, rows, it, olib)
    one = gpu_logprob(h, W, tg, it)
    for c in (512, 64):
        got = _concat([gpu_logprob(h[i:i + c].contiguous(), W, tg[i:i + c].contiguous(), it)
                       for i in range(0, T, c)])
        assert_bitwise(one, got, f"chunks of {c}")
    # token by token (decode): one row per call
    lp = torch.empty(T, device="cuda")
    lse = torch.empty(T, device="cuda")
    am = torch.empty(T, device="cuda", dtype=torch.int32)
    for i in range(T):
        rlk.logprob(h[i:i + 1], W, tg[i:i + 1], it, out=(lp[i:i + 1], lse[i:i + 1], am[i:i + 1]))
    rlk.check_device_error()
    tok = (lp.cpu().numpy(), lse.cpu().numpy(), am.cpu().numpy())
    assert_bitwise(one, tok, "token by token")
    # the pages' acceptance statistics between the prefill and decode paths: all 0
    st = rlk.consistency_stats(torch.from_numpy(one[0]).cuda(), lp)
    for k in ("max_abs", "mean_abs", "std_abs", "k3_mean", "sum_delta", "n_bit_mismatch"):
        assert st[k] == 0.0, (k, st[k])
    assert st["n_valid"] == T and st["first_mismatch"] == -1
    assert_parity(one, ref.result(), rows=rows, what="T=16384 one call, 2048+ rows")


def test_large_packed_batch_outliers_and_mask(olib):
    import invariant_token_logprob_gb300 as rlk
    T, H = 32768, 5120
    d = lm_head_inputs(T, H, V, seed=5, device="cuda", outlier_frac=0.01, mask_zero_frac=0.1)
    h, W, tg, mask = d["h"], d["W"], d["targets"], d["mask"]
    out_rows = d["outlier_rows"].cpu().numpy()
    others = np.setdiff1d(np.arange(T), out_rows)
    g = np.random.default_rng(9)
    sample = g.choice(others, 2048, replace=False)
    rows = np.unique(np.concatenate([out_rows, sample, [0, T - 1]]))
    assert rows.size >= out_rows.size + 2048
    ref = _oracle(d, rows, 1.0, olib)  # every outlier row plus 2048 others
    one = gpu_logprob(h, W, tg)
    got = _concat([gpu_logprob(h[i:i + 512].contiguous(), W, tg[i:i + 512].contiguous())
                   for i in range(0, T, 512)])
    assert_bitwise(one, got, "chunks of 512")
    st = rlk.consistency_stats(torch.from_numpy(one[0]).cuda(), torch.from_numpy(got[0]).cuda(), mask)
    assert st["n_valid"] == int(mask.sum().item()) == T - round(0.1 * T)
    assert st["max_abs"] == 0.0 and st["k3_mean"] == 0.0 and st["n_bit_mismatch"] == 0
    assert_parity(one, ref.result(), rows=rows, what="T=32768 H=5120, outliers + 2048 rows")
