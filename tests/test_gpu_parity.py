"""GPU parity at small sizes: every output of the CUDA path against the fp64
oracle, element by element, on seeded inputs spanning several tiles and ragged
tails in T, H and V; plus the degenerate cases (V = 1, W = 0, exact integer
logits with ties, ignored targets) and the two phases on their own (partials
vs the oracle's per-block statistics; merge vs the oracle's fp64 merge)."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bitwise, assert_block_records, assert_parity, gpu_logprob, to_dev
from invariant_token_logprob_gb300.inputs import lm_head_inputs, tiny_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import invariant_token_logprob_gb300 as rlk
    rlk.lib()


def test_tiny_full_parity_and_forced_ties(olib):
    d = tiny_inputs(seed=0, device="cuda")
    gpu = gpu_logprob(d["h"], d["W"], d["targets"], 1.0)
    ref = oracle.logprob(d["h"], d["W"], d["targets"], 1.0, lib=olib)
    assert_parity(gpu, ref, what="tiny")
    # forced exact ties: the lower vocabulary index wins, on both copies of each row
    exp = d["expected_tie_argmax"].numpy()
    src, dst = d["dup_src"].cpu().numpy(), d["dup_dst"].cpu().numpy()
    assert np.array_equal(gpu[2][src], exp)
    assert np.array_equal(gpu[2][dst], exp)
    # the same hidden row at two batch positions: identical lse / argmax bits
    assert np.array_equal(gpu[1][src].view(np.uint32), gpu[1][dst].view(np.uint32))


@pytest.mark.parametrize("T,H,V,seed", [
    (1, 64, 1, 1), (3, 8, 257, 2), (130, 72, 1000, 3), (257, 136, 2049, 4),
    (5, 4096, 3000, 5), (129, 512, 512, 6), (300, 64, 33, 7), (2, 1024, 151936, 8),
    (6, 64, 250000, 9),  # 977 tiles a row: the merge folds two groups of 24 slots per lane
])
def test_ragged_shapes(T, H, V, seed, olib):
    d = to_dev(lm_head_inputs(T, H, V, seed=seed))
    it = 1.0 / 0.7 if seed % 2 else 1.0
    gpu = gpu_logprob(d["h"], d["W"], d["targets"], it)
    ref = oracle.logprob(d["h"].cpu(), d["W"].cpu(), d["targets"].cpu(), it, lib=olib)
    assert_parity(gpu, ref, what=f"T={T} H={H} V={V}")


def test_zero_weights_closed_form():
    for V in (1, 1024, 151936):
        T, H = 7, 64
        h = torch.randn(T, H, device="cuda").to(torch.bfloat16)
        W = torch.zeros(V, H, device="cuda", dtype=torch.bfloat16)
        tg = torch.arange(T, device="cuda", dtype=torch.int32) % V
        lp, lse, am = gpu_logprob(h, W, tg)
        lnV = math.log(V)
        assert np.all(np.abs(lse - lnV) <= 1e-5 * max(1.0, lnV)), lse
        assert np.all(np.abs(lp + lnV) <= 5e-4)
        assert np.all(am == 0)


def test_exact_integer_logits_and_ties(olib):
    """Small-integer bf16 inputs make every fp32 logit an exact integer, so the
    GPU argmax must equal the oracle's lowest-index argmax exactly, ties included."""
    g = torch.Generator().manual_seed(17)
    T, H, V = 200, 32, 700
    h = torch.randint(-3, 4, (T, H), generator=g).to(torch.bfloat16)
    W = torch.randint(-2, 3, (V, H), generator=g).to(torch.bfloat16)
    W[650] = W[3]      # duplicated rows: exact ties across vocabulary tiles
    W[300] = W[299]
    tg = torch.randint(-1, V, (T,), generator=g, dtype=torch.int32)
    gpu = gpu_logprob(h.cuda(), W.cuda(), tg.cuda(), 0.5)
    ref = oracle.logprob(h, W, tg, 0.5, lib=olib)
    assert np.array_equal(gpu[2], ref["argmax"])
    assert_parity(gpu, ref, what="integer logits")
    assert np.all(gpu[0][tg.numpy() < 0] == 0.0)


def test_ignored_targets_write_zero(olib):
    d = lm_head_inputs(16, 64, 600, seed=9)
    d["targets"][:2] = torch.tensor([-1, -100], dtype=torch.int32)
    dd = to_dev(d)
    gpu = gpu_logprob(dd["h"], dd["W"], dd["targets"])  # negative: ignored, nothing flagged
    assert np.all(gpu[0][:2] == 0.0)
    ref = oracle.logprob(d["h"], d["W"], d["targets"], lib=olib)
    assert_parity(gpu, ref, what="ignored targets")


@pytest.mark.parametrize("T", [5, 300])  # single CTA and CTA pair shapes
def test_targets_beyond_V_are_flagged(olib, T):
    """A target >= V cannot be checked on the host: the row gets logp = 0 like an
    ignored row, and the merge counts it in the device's error records, which
    rlk_check_device_error reports as RLK_ERR_TARGET_RANGE (then cleared)."""
    import invariant_token_logprob_gb300 as rlk
    V = 600
    d = lm_head_inputs(T, 64, V, seed=9)
    d["targets"][:4] = torch.tensor([-1, V, V + 7, 2**31 - 1], dtype=torch.int32)
    dd = to_dev(d)
    rlk.check_device_error()
    lp, lse, am = rlk.logprob(dd["h"], dd["W"], dd["targets"])
    bits, rows = rlk.take_device_errors()
    assert (bits, rows) == (0, 3)
    gpu = (lp.cpu().numpy(), lse.cpu().numpy(), am.cpu().numpy())
    assert np.all(gpu[0][:4] == 0.0)
    assert_parity(gpu, oracle.logprob(d["h"], d["W"], d["targets"], lib=olib), what="targets >= V")
    rlk.logprob(dd["h"], dd["W"], dd["targets"])
    with pytest.raises(rlk.RlkError) as e:
        rlk.check_device_error()
    assert e.value.status == 7  # RLK_ERR_TARGET_RANGE
    rlk.check_device_error()  # cleared by the read
    # in-range targets raise nothing
    dd["targets"][:4] = torch.tensor([0, V - 1, 1, 2], dtype=torch.int32, device="cuda")
    rlk.logprob(dd["h"], dd["W"], dd["targets"])
    assert rlk.take_device_errors() == (0, 0)


def test_temperature_is_one_exact_multiply():
    """inv_temp = 2 equals doubling W bit for bit (both exact in fp32/bf16)."""
    d = to_dev(lm_head_inputs(40, 256, 1500, seed=12))
    a = gpu_logprob(d["h"], d["W"], d["targets"], 2.0)
    b = gpu_logprob(d["h"], (d["W"].float() * 2).to(torch.bfloat16), d["targets"], 1.0)
    assert_bitwise(a, b, "inv_temp=2 vs 2W")


def test_partials_match_oracle_block_stats(olib):
    """Phase 1 alone: each (row, 256-column tile) record {m, s, a, zt} against the
    oracle's per-block statistics."""
    import invariant_token_logprob_gb300 as rlk
    T, H, V = 150, 192, 1300
    d = lm_head_inputs(T, H, V, seed=21)
    dd = to_dev(d)
    P = rlk.logprob_partials(dd["h"], dd["W"], dd["targets"], 1.0)
    rlk.check_device_error()
    P = P.cpu().numpy()
    bs = oracle.block_stats(d["h"], d["W"], d["targets"], rlk.vocab_tile(), 1.0, lib=olib)
    assert_block_records(P, bs, d["h"], d["W"], rlk.vocab_tile(), what="partials")


@pytest.mark.parametrize("V", [151936, 250000, 1000003])
def test_merge_alone_matches_oracle_fp64_merge(olib, V):
    """Phase 2 alone on synthetic partials (including -inf blocks and equal
    maxima).  V = 250000 and 1000003 give rows of 977 and 3907 tiles: the merge
    folds more than one group of 24 slots per lane."""
    import invariant_token_logprob_gb300 as rlk
    g = np.random.default_rng(4)
    nvt = (V + 255) // 256
    T = 333
    m = g.normal(0, 3, (T, nvt)).astype(np.float32)
    m[:, 5] = m[:, 100]                       # equal maxima in different tiles
    m[7, :] = 0.0                             # a row where every tile ties
    m[8, 1:] = -np.inf                        # a row with only one populated tile
    s = g.uniform(1.0, 256.0, (T, nvt)).astype(np.float32)
    s[8, 1:] = 0.0
    a = (np.arange(nvt, dtype=np.int32)[None, :] * 256 + g.integers(0, 128, (T, nvt))).astype(np.int32)
    zt = g.normal(0, 3, (T, nvt)).astype(np.float32)
    tg = g.integers(0, V, T).astype(np.int32)
    tg[:3] = -1
    P = np.stack([m, s, a.view(np.float32), zt], axis=-1)
    Pd = torch.from_numpy(P).cuda()
    lp, lse, am = rlk.lse_merge(Pd, torch.from_numpy(tg).cuda(), V)
    lp, lse, am = lp.cpu().numpy(), lse.cpu().numpy(), am.cpu().numpy()
    ref = oracle.merge_blocks(m, s, a, zt, tg, V, 256, lib=olib)
    assert np.all(np.abs(lse - ref["lse"]) <= 2e-6 * np.maximum(1, np.abs(ref["lse"])))
    assert np.all(np.abs(lp - ref["logp"]) <= 2e-5)
    assert np.array_equal(am, ref["argmax"])
    assert np.all(lp[:3] == 0.0)


def test_consistency_stats_match_oracle(olib):
    import invariant_token_logprob_gb300 as rlk
    g = np.random.default_rng(8)
    for n in (1, 1000, 16384, 16385, 100003):
        b = g.normal(-3, 1, n).astype(np.float32)
        a = b + (g.normal(0, 1e-3, n) * (g.uniform(size=n) < 0.3)).astype(np.float32)
        mask = (g.uniform(size=n) > 0.1).astype(np.int8)
        for mk in (None, mask):
            st = rlk.consistency_stats(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(),
                                       None if mk is None else torch.from_numpy(mk).cuda())
            ref = oracle.consistency_stats(a, b, mk, lib=olib)
            got = np.array([st[k] for k in rlk.STAT_NAMES])
            assert got[0] == ref[0]
            assert np.allclose(got[1:5], ref[1:5], rtol=1e-9, atol=1e-15)
            assert np.array_equal(got[5:], ref[5:])
    # diff = 0: identical inputs give all-zero statistics
    x = torch.randn(5000, device="cuda")
    st = rlk.consistency_stats(x, x.clone())
    assert all(st[k] == 0.0 for k in ("max_abs", "mean_abs", "std_abs", "k3_mean", "sum_delta",
                                      "n_bit_mismatch"))
    assert st["first_mismatch"] == -1.0 and st["n_valid"] == 5000


@pytest.mark.parametrize("H", [136, 320])
def test_pair_and_single_cta_calls_agree_bitwise(H, olib):
    """T = 300 runs as CTA pairs: units of two row tiles, the odd tile of the
    last unit past the end of h (not copied), H = 136 / 320 an odd number of
    64-element k-blocks (3 / 5: a half-filled last stage), V = 3001 a ragged
    last vocabulary tile whose odd half is not copied.  Chunks of at most 128
    rows run as single CTAs; chunks of 129+ rows as pairs again.  Every row's
    bits must agree across all of them, and a sample matches the oracle."""
    d = lm_head_inputs(300, H, 3001, seed=22 + H, hidden="normal", w_std=0.05)
    dd = to_dev(d)
    full = gpu_logprob(dd["h"], dd["W"], dd["targets"])
    for c in (1, 64, 128, 129, 150, 299):
        parts = [gpu_logprob(dd["h"][i:i + c].contiguous(), dd["W"],
                             dd["targets"][i:i + c].contiguous()) for i in range(0, 300, c)]
        got = tuple(np.concatenate([p[k] for p in parts]) for k in range(3))
        assert_bitwise(full, got, f"H={H} chunk={c}")
    rows = np.array([0, 127, 128, 255, 256, 299])
    ref = oracle.logprob(d["h"][rows], d["W"], d["targets"][rows], lib=olib)
    assert_parity(tuple(x[rows] for x in full), ref, what=f"H={H} sampled rows")


def test_consistency_stats_async_matches_sync_bitwise(olib):
    """rlk_consistency_stats_async: the stream-ordered variant writes the same
    bits as the synchronous call (same kernels, same fixed order), into device
    memory, with a caller workspace reused across calls; n = 0 writes the empty
    result."""
    import invariant_token_logprob_gb300 as rlk
    g = np.random.default_rng(9)
    out = torch.full((8,), float("nan"), dtype=torch.float64, device="cuda")
    ws = torch.empty(max(16, rlk.stats_workspace_size(100003)), dtype=torch.uint8, device="cuda")
    for n in (1, 16384, 16385, 100003):
        b = g.normal(-3, 1, n).astype(np.float32)
        a = b + (g.normal(0, 1e-3, n) * (g.uniform(size=n) < 0.3)).astype(np.float32)
        mask = (g.uniform(size=n) > 0.1).astype(np.int8)
        for mk in (None, mask):
            ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
            tm = None if mk is None else torch.from_numpy(mk).cuda()
            rlk.consistency_stats_async(ta, tb, tm, out=out, workspace=ws)
            got = out.cpu().numpy()
            ref = np.array([rlk.consistency_stats(ta, tb, tm)[k] for k in rlk.STAT_NAMES])
            assert np.array_equal(got.view(np.uint64), ref.view(np.uint64)), (n, got, ref)
            oref = oracle.consistency_stats(a, b, mk, lib=olib)
            assert got[0] == oref[0] and np.array_equal(got[5:], oref[5:])
    e = torch.empty(0, device="cuda")
    rlk.consistency_stats_async(e, e, out=out, workspace=ws)
    assert out.cpu().tolist() == [0.0] * 7 + [-1.0]


def test_chunking_permutation_and_repeat_invariance_small():
    """Bitwise: the tiny workload as one call, in every chunk size 1..64, in a
    permuted order, and repeated, gives identical bits for every row."""
    d = tiny_inputs(seed=0, device="cuda")
    h, W, tg = d["h"], d["W"], d["targets"]
    T = h.shape[0]
    full = gpu_logprob(h, W, tg)
    for c in range(1, T + 1):
        parts = [gpu_logprob(h[i:i + c].contiguous(), W, tg[i:i + c].contiguous())
                 for i in range(0, T, c)]
        got = tuple(np.concatenate([p[k] for p in parts]) for k in range(3))
        assert_bitwise(full, got, f"chunk={c}")
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(5)).cuda()
    pg = gpu_logprob(h[perm].contiguous(), W, tg[perm].contiguous())
    inv = torch.argsort(perm).cpu().numpy()
    assert_bitwise(full, tuple(x[inv] for x in pg), "permuted rows")
    for _ in range(3):
        assert_bitwise(full, gpu_logprob(h, W, tg), "repeat")


def test_padding_rows_do_not_leak():
    """A row's bits do not depend on what else shares its 128-row tile."""
    d = lm_head_inputs(128, 256, 3000, seed=31)
    dd = to_dev(d)
    base = gpu_logprob(dd["h"], dd["W"], dd["targets"])
    h2 = dd["h"].clone()
    h2[1:] = (h2[1:].float() * -7.0).to(torch.bfloat16)  # change every other row
    other = gpu_logprob(h2, dd["W"], dd["targets"])
    assert_bitwise(tuple(x[:1] for x in base), tuple(x[:1] for x in other), "row 0 neighbours")


@pytest.mark.parametrize("T", [1, 5, 15, 16, 17, 40])
def test_caller_workspace_matches_cached_workspace(T):
    """rlk_logprob_ws with an exactly-sized caller workspace gives rlk_logprob's
    bits; one byte less is refused before anything runs."""
    import invariant_token_logprob_gb300 as rlk
    d = to_dev(lm_head_inputs(T, 256, 3000, seed=50 + T))
    need = rlk.workspace_size(T, 256, 3000)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    a = rlk.logprob_ws(d["h"], d["W"], d["targets"], ws)
    b = rlk.logprob(d["h"], d["W"], d["targets"])
    rlk.check_device_error()
    assert_bitwise(tuple(x.cpu().numpy() for x in a), tuple(x.cpu().numpy() for x in b), f"T={T}")
    with pytest.raises(rlk.RlkError) as ei:
        rlk.logprob_ws(d["h"], d["W"], d["targets"], ws[:need - 1])
    assert ei.value.status == 5


def test_zero_rows_everywhere():
    """T = 0 is a valid call for every entry point: empty outputs, nothing
    launched, no error.  The backward's grad_W is then an empty sum: when it is
    overwritten it becomes zero, when it is accumulated into it stays as it was."""
    import ctypes
    import invariant_token_logprob_gb300 as rlk
    H, V = 256, 1000
    d = to_dev(lm_head_inputs(4, H, V, seed=3))
    h0, tg0, W = d["h"][:0].contiguous(), d["targets"][:0].contiguous(), d["W"]
    outs = [rlk.logprob(h0, W, tg0),
            rlk.logprob_fp8(h0, *rlk.quantize_fp8_weight(W), tg0),
            rlk.logprob_fp8_block(h0, *rlk.quantize_fp8_weight_blocks(W), tg0, V),
            rlk.logprob_entropy(h0, W, tg0)]
    parts = rlk.logprob_partials(h0, W, tg0)
    outs.append(rlk.lse_merge(parts, tg0, V))
    assert parts.shape[0] == 0
    for out in outs:
        assert all(x.numel() == 0 for x in out)
    L = rlk.lib()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    gW = torch.full((V, H), float("nan"), device="cuda")
    assert L.rlk_logprob_backward(None, None, None, None, None, 0, H, V, ctypes.c_float(1.0), None,
                                  ctypes.c_void_p(gW.data_ptr()), 0, None, 0, st) == 0
    torch.cuda.synchronize()
    assert torch.all(gW == 0)
    base = torch.randn(V, H, device="cuda")
    gW = base.clone()
    assert L.rlk_logprob_backward(None, None, None, None, None, 0, H, V, ctypes.c_float(1.0), None,
                                  ctypes.c_void_p(gW.data_ptr()), 1, None, 0, st) == 0
    torch.cuda.synchronize()
    assert torch.equal(gW, base)
    rlk.check_device_error()
