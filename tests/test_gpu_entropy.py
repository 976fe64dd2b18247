"""GPU tests of rlk_logprob_entropy (per-token softmax entropy from the same
vocabulary-tile partials).

Tolerance: |entropy_gpu - entropy_oracle| <= 5e-4, the logp tolerance; the
entropy log S - U/S is built from the same fp32 tile statistics as the LSE.
Its logp / lse / argmax must be bit-identical to rlk_logprob's, and its own bits
must not depend on the batch composition (same contract as the forward)."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bitwise, assert_parity, to_dev
from invariant_token_logprob_gb300.inputs import lm_head_inputs, tiny_inputs

pytestmark = pytest.mark.gpu
ENT_ATOL = 5e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import invariant_token_logprob_gb300 as rlk
    rlk.lib()


def _np(xs):
    return tuple(x.cpu().numpy() for x in xs)


def _ent(d, it=1.0):
    import invariant_token_logprob_gb300 as rlk
    out = rlk.logprob_entropy(d["h"], d["W"], d["targets"], it)
    rlk.check_device_error()
    return _np(out)


@pytest.mark.parametrize("case", ["tiny", (1, 64, 1, 1), (7, 72, 1000, 2), (130, 256, 2049, 3),
                                  (300, 128, 33, 4),
                                  (6, 64, 250000, 5)])  # 977 tiles a row: two slot groups per lane
def test_entropy_matches_oracle_and_forward_bits(case, olib):
    import invariant_token_logprob_gb300 as rlk
    if case == "tiny":
        d = tiny_inputs(seed=0, device="cuda")
        it = 1.0
    else:
        T, H, V, seed = case
        d = to_dev(lm_head_inputs(T, H, V, seed=seed, hidden="normal", w_std=0.05))
        it = float(np.float32(1 / 0.7)) if seed % 2 else 1.0
    lp, lse, am, ent = _ent(d, it)
    fwd = _np(rlk.logprob(d["h"], d["W"], d["targets"], it))
    assert_bitwise(fwd, (lp, lse, am), f"{case}: entropy path vs rlk_logprob")
    ref_e = oracle.entropy(d["h"].cpu(), d["W"].cpu(), it, lib=olib)
    assert np.all(np.abs(ent.astype(np.float64) - ref_e) <= ENT_ATOL), \
        f"{case}: max |dH| {np.max(np.abs(ent - ref_e)):.3g}"
    ref = oracle.logprob(d["h"].cpu(), d["W"].cpu(), d["targets"].cpu(), it, lib=olib)
    assert_parity((lp, lse, am), ref, what=str(case))


def test_entropy_uniform_is_log_v():
    for V in (1, 1000, 151936):
        h = torch.randn(5, 64, device="cuda").to(torch.bfloat16)
        W = torch.zeros(V, 64, device="cuda", dtype=torch.bfloat16)
        tg = torch.zeros(5, device="cuda", dtype=torch.int32)
        _, _, _, ent = _ent(dict(h=h, W=W, targets=tg))
        assert np.all(np.abs(ent - math.log(V)) <= ENT_ATOL * max(1, math.log(V))), ent


@pytest.mark.slow
def test_entropy_full_size_parity_and_invariance(olib):
    T, H, V = 4096, 4096, 151936
    d = lm_head_inputs(T, H, V, seed=12, device="cuda")
    lp, lse, am, ent = _ent(d)
    rows = np.array([0, 5, 2048, T - 1])
    ref_e = oracle.entropy(d["h"].cpu(), d["W"].cpu(), 1.0, rows=rows, lib=olib)
    assert np.all(np.abs(ent[rows].astype(np.float64) - ref_e) <= ENT_ATOL)
    parts = [_ent(dict(h=d["h"][i:i + 512].contiguous(), W=d["W"],
                       targets=d["targets"][i:i + 512].contiguous())) for i in range(0, T, 512)]
    got = np.concatenate([p[3] for p in parts])
    assert np.array_equal(got.view(np.uint32), ent.view(np.uint32)), "entropy chunk invariance"
    one = _ent(dict(h=d["h"][7:8].contiguous(), W=d["W"], targets=d["targets"][7:8].contiguous()))
    assert one[3].view(np.uint32)[0] == ent.view(np.uint32)[7], "entropy T=1 vs T=4096"
