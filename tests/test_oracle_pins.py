"""Pins for the fp64 CPU oracle: each check ties it to something other than
itself -- a closed form, an invariance of the mathematics, an exact brute force
in arbitrary precision, a library routine (scipy) on an independent code path,
or the pages' own worked example (tests/golden/).

Every pin is a function of the loaded oracle library so that
``test_pins_catch_planted_mistakes`` can run the same pins against oracle builds
with a deliberate mistake planted (ORACLE_MUTANT in oracle.c) and show that each
mistake fails at least one pin.
"""
import json
import math
import os

import mpmath
import numpy as np
import pytest
import scipy.special

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """float -> bf16 bits by round-to-nearest-even (inputs here are bf16-exact)."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    back = (r.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(back, f), "test input is not bf16-exact"
    return r


def _bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------- pins

def pin_zero_weights(lib):
    """W = 0: every logit is 0, so LSE = ln V, logp = -ln V, argmax = 0 (lowest
    index among V-way tie), top-2 gap 0."""
    for V in (1, 7, 1024, 151936):
        H, T = 16, 3
        rng = np.random.default_rng(V)
        h = _bf16_bits(rng.integers(-3, 4, size=(T, H)).astype(np.float32))
        W = np.zeros((V, H), dtype=np.uint16)
        tg = np.array([0, V - 1, V // 2], dtype=np.int32)
        r = oracle.logprob(h, W, tg, 1.0, lib=lib)
        lnV = float(mpmath.log(V))
        assert np.allclose(r["lse"], lnV, rtol=0, atol=1e-12 * max(1.0, lnV))
        assert np.allclose(r["logp"], -lnV, rtol=0, atol=1e-12 * max(1.0, lnV))
        assert np.all(r["argmax"] == 0)
        if V > 1:
            assert np.all(r["top2gap"] == 0.0)


def pin_one_hot_dominant(lib):
    """h = c e_k, W[v*,k] = b, all else 0: z_{v*} = b c inv_temp, other z = 0.
    logp(v*) = -log1p((V-1) exp(-z*)), logp(other) = -z* - log1p(...).
    Uses the last hidden column k = H-1 in one case, and inv_temp != 1."""
    cases = [(64, 1000, 5, 63, 2.0, 4.0, 1.0), (32, 4096, 4095, 31, 1.5, 3.0, 2.0),
             (16, 77, 0, 0, -2.0, 4.0, 0.5)]
    for H, V, vstar, k, c, b, it in cases:
        h = np.zeros((2, H), np.float32)
        h[:, k] = c
        W = np.zeros((V, H), np.float32)
        W[vstar, k] = b
        other = (vstar + 1) % V
        tg = np.array([vstar, other], np.int32)
        r = oracle.logprob(_bf16_bits(h), _bf16_bits(W), tg, it, lib=lib)
        zs = mpmath.mpf(b) * c * it
        tail = mpmath.log1p((V - 1) * mpmath.exp(-zs))
        exp_logp = [float(-tail), float(-zs - tail)]
        exp_lse = float(zs + tail)
        assert np.allclose(r["logp"], exp_logp, rtol=1e-13, atol=1e-13), (r["logp"], exp_logp)
        assert np.allclose(r["lse"], exp_lse, rtol=1e-13, atol=1e-13)
        if zs > 0:
            assert np.all(r["argmax"] == vstar)
        else:
            assert np.all(r["argmax"] == (0 if vstar != 0 else 1))


def pin_shift_invariance(lib):
    """Append a hidden column equal to 1 and a weight column equal to c (bf16-exact):
    every logit moves by c, so LSE moves by c and logp is unchanged."""
    rng = np.random.default_rng(7)
    T, H, V = 4, 48, 777
    h = rng.standard_normal((T, H)).astype(np.float32)
    W = (0.05 * rng.standard_normal((V, H))).astype(np.float32)
    hb = _bits_to_f64(_bf16_bits_round(h)).astype(np.float32)
    Wb = _bits_to_f64(_bf16_bits_round(W)).astype(np.float32)
    tg = rng.integers(0, V, T).astype(np.int32)
    base = oracle.logprob(_bf16_bits(hb), _bf16_bits(Wb), tg, 1.0, lib=lib)
    for c in (3.0, -2.5, 0.125):
        h2 = np.concatenate([hb, np.ones((T, 1), np.float32)], 1)
        W2 = np.concatenate([Wb, np.full((V, 1), c, np.float32)], 1)
        s = oracle.logprob(_bf16_bits(h2), _bf16_bits(W2), tg, 1.0, lib=lib)
        assert np.allclose(s["lse"] - base["lse"], c, rtol=0, atol=1e-12)
        assert np.allclose(s["logp"], base["logp"], rtol=0, atol=1e-12)
        assert np.array_equal(s["argmax"], base["argmax"])


def pin_temperature(lib):
    """inv_temp = 2 is the same as doubling W (both exact), bit for bit in fp64;
    inv_temp = 0.5 the same as halving W."""
    rng = np.random.default_rng(11)
    T, H, V = 3, 40, 500
    h = _bf16_bits_round(rng.standard_normal((T, H)).astype(np.float32))
    Wf = _bits_to_f64(_bf16_bits_round((0.05 * rng.standard_normal((V, H))).astype(np.float32)))
    tg = rng.integers(0, V, T).astype(np.int32)
    for it, scale in ((2.0, 2.0), (0.5, 0.5)):
        a = oracle.logprob(h, _bf16_bits(Wf.astype(np.float32)), tg, it, lib=lib)
        b = oracle.logprob(h, _bf16_bits((Wf * scale).astype(np.float32)), tg, 1.0, lib=lib)
        for k in ("logp", "lse", "argmax", "zmax"):
            assert np.array_equal(a[k], b[k]), k


def pin_brute_force_exact(lib):
    """Small-integer bf16 inputs: logits are exact integers (Python ints), LSE by
    mpmath at 40 digits, argmax the lowest index of the exact maximum."""
    mpmath.mp.dps = 40
    rng = np.random.default_rng(3)
    for trial in range(6):
        T, H, V = 4, int(rng.integers(1, 17)), int(rng.integers(1, 33))
        hi = rng.integers(-4, 5, size=(T, H))
        Wi = rng.integers(-3, 4, size=(V, H))
        if V > 3:
            Wi[V - 1] = Wi[1]  # exact duplicate row: forces ties in some rows
        it = (1.0, 0.5, 2.0)[trial % 3]
        tg = rng.integers(-1, V, size=T).astype(np.int32)
        r = oracle.logprob(_bf16_bits(hi.astype(np.float32)), _bf16_bits(Wi.astype(np.float32)),
                           tg, it, lib=lib)
        for t in range(T):
            z = [int(sum(int(hi[t, k]) * int(Wi[v, k]) for k in range(H))) for v in range(V)]
            zm = [mpmath.mpf(x) * mpmath.mpf(it) for x in z]
            lse = mpmath.log(mpmath.fsum(mpmath.exp(x) for x in zm))
            amax = z.index(max(z))
            assert abs(r["lse"][t] - float(lse)) <= 1e-13 * max(1.0, abs(float(lse)))
            assert r["argmax"][t] == amax
            lp = float(zm[tg[t]] - lse) if tg[t] >= 0 else 0.0
            assert abs(r["logp"][t] - lp) <= 1e-13 * max(1.0, abs(lp))
            srt = sorted(zm, reverse=True)
            gap = float(srt[0] - srt[1]) if V > 1 else math.inf
            assert r["top2gap"][t] == gap


def pin_scipy_logsumexp(lib):
    """Independent code path: fp64 logits by numpy/BLAS matmul, LSE and
    log-softmax by scipy.special; agreement to 1e-11."""
    rng = np.random.default_rng(5)
    T, H, V = 6, 96, 3001
    h = _bf16_bits_round(rng.standard_normal((T, H)).astype(np.float32))
    W = _bf16_bits_round((0.03 * rng.standard_normal((V, H))).astype(np.float32))
    it = 1.0 / 0.7
    tg = rng.integers(0, V, T).astype(np.int32)
    r = oracle.logprob(h, W, tg, it, lib=lib)
    z = (_bits_to_f64(h) @ _bits_to_f64(W).T) * float(np.float32(it))
    lse = scipy.special.logsumexp(z, axis=1)
    ls = scipy.special.log_softmax(z, axis=1)
    assert np.allclose(r["lse"], lse, rtol=0, atol=1e-11)
    assert np.allclose(r["logp"], ls[np.arange(T), tg], rtol=0, atol=1e-11)
    assert np.array_equal(r["argmax"], np.argmax(z, axis=1))


def pin_ignored_targets(lib):
    """A target outside [0, V) is an ignored row: logp = 0, LSE still computed."""
    rng = np.random.default_rng(9)
    T, H, V = 4, 8, 50
    h = _bf16_bits_round(rng.standard_normal((T, H)).astype(np.float32))
    W = _bf16_bits_round(rng.standard_normal((V, H)).astype(np.float32))
    tg = np.array([-1, V, -100, 3], np.int32)
    r = oracle.logprob(h, W, tg, 1.0, lib=lib)
    assert np.all(r["logp"][:3] == 0.0)
    assert r["logp"][3] < 0.0
    z = _bits_to_f64(h) @ _bits_to_f64(W).T
    assert np.allclose(r["lse"], scipy.special.logsumexp(z, axis=1), atol=1e-11)


def pin_block_stats_and_merge(lib):
    """Per-block (m, s, a, zt) of the vocabulary against numpy on independently
    computed logits; the fp64 merge of those blocks reproduces the whole-vocab
    LSE / argmax / logp (the blockwise merge of the RL-Kernel blog, §四)."""
    rng = np.random.default_rng(13)
    T, H, V, bn = 5, 64, 1000, 128
    h = _bf16_bits_round(rng.standard_normal((T, H)).astype(np.float32))
    W = _bf16_bits_round((0.05 * rng.standard_normal((V, H))).astype(np.float32))
    tg = rng.integers(0, V, T).astype(np.int32)
    bs = oracle.block_stats(h, W, tg, bn, 1.0, lib=lib)
    z = _bits_to_f64(h) @ _bits_to_f64(W).T
    nb = (V + bn - 1) // bn
    assert bs["m"].shape == (T, nb)
    for j in range(nb):
        zz = z[:, j * bn:min(V, (j + 1) * bn)]
        assert np.allclose(bs["m"][:, j], zz.max(1), atol=1e-12)
        assert np.array_equal(bs["a"][:, j], j * bn + zz.argmax(1))
        assert np.allclose(bs["s"][:, j], np.exp(zz - zz.max(1, keepdims=True)).sum(1), rtol=1e-12)
        inb = (tg >= j * bn) & (tg < (j + 1) * bn)
        assert np.allclose(bs["zt"][inb, j], z[inb, tg[inb]], atol=1e-12)
        assert np.all(bs["zt"][~inb, j] == 0.0)
    full = oracle.logprob(h, W, tg, 1.0, lib=lib)
    mg = oracle.merge_blocks(bs["m"].astype(np.float32), bs["s"].astype(np.float32),
                             bs["a"].astype(np.int32), bs["zt"].astype(np.float32), tg, V, bn,
                             lib=lib)
    # fp32 storage of the partials costs ~1e-7 relative
    assert np.allclose(mg["lse"], full["lse"], rtol=2e-7, atol=2e-7)
    assert np.allclose(mg["logp"], full["logp"], rtol=0, atol=1e-6)
    assert np.array_equal(mg["argmax"], full["argmax"])
    # exact case: four equal blocks with m = 0, s = 1 -> LSE = ln 4, argmax = lowest a
    m4 = np.zeros((1, 4), np.float32)
    s4 = np.ones((1, 4), np.float32)
    a4 = np.array([[30, 10, 20, 40]], np.int32)
    e = oracle.merge_blocks(m4, s4, a4, None, None, 64, 16, lib=lib)
    assert abs(e["lse"][0] - math.log(4.0)) < 1e-15 and e["argmax"][0] == 10
    # a block at -inf (e.g. fully masked) contributes nothing
    mi = np.array([[1.0, -np.inf]], np.float32)
    si = np.array([[2.0, 0.0]], np.float32)
    ai = np.array([[3, 0]], np.int32)
    e = oracle.merge_blocks(mi, si, ai, None, None, 64, 32, lib=lib)
    assert abs(e["lse"][0] - (1.0 + math.log(2.0))) < 1e-15 and e["argmax"][0] == 3


def pin_worked_example(lib):
    """The pages' worked example (tests/golden/worked_example.json): 200 tokens,
    rollout -2.300, train -2.308: per-token ratio ~0.992, cumulative log-ratio
    1.6, sequence ratio ~0.20; max = mean |gap| = 0.008, std 0."""
    g = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    n = g["n_tokens"]
    a = np.full(n, g["train_logp"], np.float32)
    b = np.full(n, g["rollout_logp"], np.float32)
    st = oracle.consistency_stats(a, b, lib=lib)
    gap32 = float(np.float64(np.float32(g["train_logp"])) - np.float64(np.float32(g["rollout_logp"])))
    assert abs(st[0] - g["per_token_gap"]) < 1e-6 and abs(st[1] - g["per_token_gap"]) < 1e-6
    assert st[0] == abs(gap32) and st[1] == pytest.approx(abs(gap32), rel=1e-15)
    assert st[2] == pytest.approx(0.0, abs=1e-15)
    assert st[4] == pytest.approx(-g["cumulative_log_gap_printed"], abs=1e-4)
    assert round(math.exp(gap32), g["per_token_ratio_printed_decimals"]) == g["per_token_ratio_printed"]
    assert round(math.exp(st[4]), g["sequence_ratio_printed_decimals"]) == g["sequence_ratio_printed"]
    lo, hi = g["clip_interval_printed"]
    assert not (lo <= math.exp(st[4]) <= hi)
    assert st[5] == n and st[6] == n and st[7] == 0
    # k3 = r - 1 - log r with log r = gap: closed form by mpmath
    k3 = float(mpmath.expm1(mpmath.mpf(gap32)) - mpmath.mpf(gap32))
    assert st[3] == pytest.approx(k3, rel=1e-12)


def pin_stats_closed_forms(lib):
    """Population std, masking, bit-mismatch counting, empty input, identity."""
    b = np.array([0.0, 1.0, -2.0, 5.0, 7.0], np.float32)
    a = b + np.array([1.0, -2.0, 3.0, 0.0, 100.0], np.float32)
    mask = np.array([1, 1, 1, 1, 0], np.int8)
    st = oracle.consistency_stats(a, b, mask, lib=lib)
    # valid |d| = 1, 2, 3, 0: mean 1.5, population var 1.25
    assert st[0] == 3.0 and st[1] == 1.5
    assert st[2] == pytest.approx(math.sqrt(1.25), rel=1e-15)
    assert st[4] == 2.0 and st[5] == 4 and st[6] == 3 and st[7] == 0
    k3 = sum(float(mpmath.expm1(d) - d) for d in (1.0, -2.0, 3.0, 0.0)) / 4
    assert st[3] == pytest.approx(k3, rel=1e-13)
    # +0.0 vs -0.0: equal values, different bits
    st = oracle.consistency_stats(np.array([1.0, 0.0], np.float32),
                                  np.array([1.0, -0.0], np.float32), lib=lib)
    assert st[0] == 0.0 and st[6] == 1 and st[7] == 1
    # identical inputs: every statistic is exactly 0 (the pages' diff = 0)
    x = np.random.default_rng(1).standard_normal(1000).astype(np.float32)
    st = oracle.consistency_stats(x, x.copy(), lib=lib)
    assert np.all(st[[0, 1, 2, 3, 4, 6]] == 0.0) and st[5] == 1000 and st[7] == -1
    # nothing valid
    st = oracle.consistency_stats(x, x + 1, np.zeros(1000, np.int8), lib=lib)
    assert np.all(st[:7] == 0.0) and st[7] == -1
    # small gaps: k3 ~ d^2 / 2 with no cancellation loss
    d = np.float32(1e-6)
    st = oracle.consistency_stats(np.array([d], np.float32), np.array([0.0], np.float32), lib=lib)
    assert st[3] == pytest.approx(float(mpmath.expm1(mpmath.mpf(float(d))) - float(d)), rel=1e-9)


def _bf16_bits_round(x: np.ndarray) -> np.ndarray:
    """Round arbitrary fp32 to bf16 bits (RNE)."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def pin_backward_finite_differences(lib):
    """dh and dW of the oracle backward equal central finite differences of the
    oracle's own fp64 forward (loss = sum_t g_t logp_t), with inv_temp != 1 and
    an ignored row."""
    rng = np.random.default_rng(21)
    T, H, V, it = 3, 5, 11, 1.5
    hb = _bf16_bits_round(rng.standard_normal((T, H)).astype(np.float32))
    Wb = _bf16_bits_round((0.7 * rng.standard_normal((V, H))).astype(np.float32))
    hf, Wf = _bits_to_f64(hb), _bits_to_f64(Wb)
    tg = np.array([4, -1, 10], np.int32)
    g = np.array([0.7, 1.3, -0.4])
    b = oracle.logprob_backward(hb, Wb, tg, g, it, lib=lib)

    def loss(hh, WW):
        return float(np.dot(g, oracle.logprob_f64(hh, WW, tg, it, lib=lib)["logp"]))

    eps = 1e-6
    for t in range(T):
        for k in range(H):
            hp, hm = hf.copy(), hf.copy()
            hp[t, k] += eps
            hm[t, k] -= eps
            fd = (loss(hp, Wf) - loss(hm, Wf)) / (2 * eps)
            assert abs(b["dh"][t, k] - fd) <= 1e-6 * max(1.0, abs(fd)), (t, k, b["dh"][t, k], fd)
    for v in range(V):
        for k in range(H):
            Wp, Wm = Wf.copy(), Wf.copy()
            Wp[v, k] += eps
            Wm[v, k] -= eps
            fd = (loss(hf, Wp) - loss(hf, Wm)) / (2 * eps)
            assert abs(b["dW"][v, k] - fd) <= 1e-6 * max(1.0, abs(fd)), (v, k, b["dW"][v, k], fd)
    # dz sums to zero over the vocabulary on valid rows and is 0 on ignored rows
    assert np.allclose(b["dz"].sum(1)[[0, 2]], 0.0, atol=1e-14)
    assert np.all(b["dz"][1] == 0.0) and np.all(b["dh"][1] == 0.0)


def pin_backward_closed_forms(lib):
    """W = 0: p is uniform, so dz = g (onehot - 1/V), dh = 0 and
    dW[v] = inv_temp sum_t g_t (onehot_v - 1/V) h_t.  Temperature: (inv_temp 2, W)
    and (1, 2W) give the same dh, and dW halves."""
    rng = np.random.default_rng(22)
    T, H, V = 4, 6, 9
    hb = _bf16_bits_round(rng.standard_normal((T, H)).astype(np.float32))
    hf = _bits_to_f64(hb)
    tg = rng.integers(0, V, T).astype(np.int32)
    g = rng.standard_normal(T)
    b = oracle.logprob_backward(hb, np.zeros((V, H), np.uint16), tg, g, 2.0, lib=lib)
    onehot = np.zeros((T, V))
    onehot[np.arange(T), tg] = 1.0
    dz = g[:, None] * (onehot - 1.0 / V)
    assert np.allclose(b["dz"], dz, atol=1e-15)
    assert np.all(b["dh"] == 0.0)
    assert np.allclose(b["dW"], 2.0 * dz.T @ hf, atol=1e-13)
    Wb = _bf16_bits_round((0.3 * rng.standard_normal((V, H))).astype(np.float32))
    W2 = _bf16_bits((2.0 * _bits_to_f64(Wb)).astype(np.float32))
    a = oracle.logprob_backward(hb, Wb, tg, g, 2.0, lib=lib)
    c = oracle.logprob_backward(hb, W2, tg, g, 1.0, lib=lib)
    assert np.allclose(a["dh"], c["dh"], rtol=1e-13, atol=1e-15)
    assert np.allclose(a["dW"], 2.0 * c["dW"], rtol=1e-13, atol=1e-15)


def pin_entropy(lib):
    """Entropy: W = 0 gives the uniform maximum ln V; a one-hot-dominant row has
    the two-level closed form; random rows agree with scipy.stats.entropy of the
    BLAS-computed softmax; an mpmath brute force on integer logits."""
    import scipy.stats
    for V in (1, 9, 151936):
        h = _bf16_bits(np.ones((2, 8), np.float32))
        e = oracle.entropy(h, np.zeros((V, 8), np.uint16), 1.0, lib=lib)
        assert np.allclose(e, float(mpmath.log(V)), atol=1e-12)
    H, V, k, c, b = 16, 500, 3, 2.0, 3.0
    h = np.zeros((1, H), np.float32)
    h[0, k] = c
    W = np.zeros((V, H), np.float32)
    W[7, k] = b
    e = oracle.entropy(_bf16_bits(h), _bf16_bits(W), 1.0, lib=lib)
    zs = mpmath.mpf(b * c)
    S = mpmath.exp(zs) + (V - 1)
    p1, q = mpmath.exp(zs) / S, 1 / S
    assert abs(e[0] - float(-(p1 * mpmath.log(p1)) - (V - 1) * q * mpmath.log(q))) < 1e-12
    rng = np.random.default_rng(31)
    hb = _bf16_bits_round(rng.standard_normal((5, 64)).astype(np.float32))
    Wb = _bf16_bits_round((0.1 * rng.standard_normal((2000, 64))).astype(np.float32))
    z = (_bits_to_f64(hb) @ _bits_to_f64(Wb).T) * float(np.float32(1 / 0.7))
    p = scipy.special.softmax(z, axis=1)
    e = oracle.entropy(hb, Wb, 1 / 0.7, lib=lib)
    assert np.allclose(e, scipy.stats.entropy(p, axis=1), atol=1e-10)
    mpmath.mp.dps = 40
    hi = rng.integers(-3, 4, (2, 6))
    Wi = rng.integers(-2, 3, (13, 6))
    e = oracle.entropy(_bf16_bits(hi.astype(np.float32)), _bf16_bits(Wi.astype(np.float32)), 1.0,
                       lib=lib)
    for t in range(2):
        zz = [mpmath.mpf(int(np.dot(hi[t], Wi[v]))) for v in range(13)]
        lse = mpmath.log(mpmath.fsum(mpmath.exp(x) for x in zz))
        ent = -mpmath.fsum(mpmath.exp(x - lse) * (x - lse) for x in zz)
        assert abs(e[t] - float(ent)) < 1e-13


def _e4m3_table():
    """All 256 e4m3 values decoded by PyTorch's float8_e4m3fn (a library routine)."""
    import torch
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def pin_fp8_quantiser(lib):
    """Per-row e4m3 quantisation: scale = amax/448 in fp32 (1 for a zero row);
    each code is the nearest e4m3 value to x/s (fp32 division), ties to the even
    code, by brute force over all codes; agrees with torch's RNE cast."""
    import torch
    tab = _e4m3_table()
    finite = np.isfinite(tab)
    rng = np.random.default_rng(41)
    x = rng.standard_normal((6, 96)).astype(np.float32) * np.array([1, 10, 1e-3, 300, 1, 0])[:, None]
    x[4, :8] = [0.5, -0.5, 1.0, 3.0, -448.0, 2.0, 0.0, 7.0]  # exact values and a tie pattern
    x[4, 8:12] = [-0.0, -1e-30, 1e-30, -3e-5]                # signed zeros and underflow to 0
    xb = _bf16_bits_round(x)
    codes, scales = oracle.quantize_fp8_rows(xb, lib=lib)
    xf = _bits_to_f64(xb).astype(np.float32)
    for r in range(6):
        amax = np.float32(np.max(np.abs(xf[r])))
        exp_s = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
        assert scales[r] == exp_s
        y = (xf[r] / scales[r]).astype(np.float32).astype(np.float64)
        for k in range(96):
            d = np.where(finite, np.abs(tab - y[k]), np.inf)
            best = np.flatnonzero(d == d.min())
            want = [c for c in best if c & 1 == 0] or list(best)
            got = codes[r, k] & 0x7F if y[k] <= 0 and tab[codes[r, k]] <= 0 else codes[r, k]
            want = [c & 0x7F for c in want] if y[k] <= 0 else want
            assert got in want or (y[k] == 0 and tab[codes[r, k]] == 0), (r, k, y[k])
        ref = torch.from_numpy((xf[r] / scales[r]).astype(np.float32)).to(torch.float8_e4m3fn)
        assert np.array_equal(codes[r], ref.view(torch.uint8).numpy())  # codes, sign of 0 included
    assert np.all(tab[codes[5]] == 0) and scales[5] == 1.0  # signed zeros keep their sign


def pin_fp8_logprob(lib):
    """FP8 logprob: with inputs that quantise exactly (row amax 448 * 2^-6, values
    e4m3 integers times 2^-6) it equals the bf16 oracle; on random inputs it equals
    scipy's log-softmax of the dequantised logits."""
    rng = np.random.default_rng(42)
    ints = np.array([0, 1, 2, 3, 4, 5, 6, 7, 8, 16, 32, 448], np.float32)
    T, H, V = 3, 24, 300
    hq = rng.choice(ints, (T, H)) * rng.choice([-1, 1], (T, H))
    wq = rng.choice(ints[:9], (V, H)) * rng.choice([-1, 1], (V, H))
    hq[:, 0] = 448.0
    wq[:, 0] = 448.0
    hb = _bf16_bits((hq * 2.0 ** -6).astype(np.float32))
    wb = _bf16_bits((wq * 2.0 ** -9).astype(np.float32))
    tg = rng.integers(0, V, T).astype(np.int32)
    qh, sh = oracle.quantize_fp8_rows(hb, lib=lib)
    qw, sw = oracle.quantize_fp8_rows(wb, lib=lib)
    assert np.all(sh == 2.0 ** -6) and np.all(sw == 2.0 ** -9)
    a = oracle.logprob_fp8(qh, sh, qw, sw, tg, 0.5, lib=lib)
    b = oracle.logprob(hb, wb, tg, 0.5, lib=lib)
    for k in ("logp", "lse", "argmax"):
        assert np.allclose(a[k], b[k], rtol=1e-14, atol=1e-14), k
    tab = _e4m3_table()
    hr = _bf16_bits_round(rng.standard_normal((4, 64)).astype(np.float32))
    wr = _bf16_bits_round((0.05 * rng.standard_normal((700, 64))).astype(np.float32))
    qh, sh = oracle.quantize_fp8_rows(hr, lib=lib)
    qw, sw = oracle.quantize_fp8_rows(wr, lib=lib)
    tg = rng.integers(0, 700, 4).astype(np.int32)
    z = (tab[qh] @ tab[qw].T) * sh.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :]
    r = oracle.logprob_fp8(qh, sh, qw, sw, tg, 1.0, lib=lib)
    assert np.allclose(r["lse"], scipy.special.logsumexp(z, axis=1), atol=1e-11)
    assert np.allclose(r["logp"], scipy.special.log_softmax(z, axis=1)[np.arange(4), tg], atol=1e-11)
    assert np.array_equal(r["argmax"], np.argmax(z, axis=1))


def _exact_block_operand(rng, rows, H, block_rows, ints):
    """bf16 matrix whose block_rows x 128 blocks quantise exactly: each block is
    2^e times e4m3-representable integers, with one element 448 * 2^e, so its
    scale amax/448 is exactly 2^e (e drawn per block) and every code is exact."""
    x = np.zeros((rows, H), np.float32)
    for r0 in range(0, rows, block_rows):
        for k0 in range(0, H, 128):
            r1, k1 = min(rows, r0 + block_rows), min(H, k0 + 128)
            e = int(rng.integers(-12, -2))
            blk = rng.choice(ints, (r1 - r0, k1 - k0)) * rng.choice([-1, 1], (r1 - r0, k1 - k0))
            blk[0, 0] = 448.0
            x[r0:r1, k0:k1] = blk * 2.0 ** e
    return x


def pin_fp8_block_quantiser(lib):
    """Block e4m3 quantisation (1 x 128 and 128 x 128 blocks, ragged edges): each
    block's scale is its amax/448 in fp32, each code torch's RNE cast of x/s."""
    import torch
    rng = np.random.default_rng(43)
    x = rng.standard_normal((130, 200)).astype(np.float32)
    x[:, 128:] *= 40.0          # a second k block with a different scale
    x[128:, :] *= 1e-3          # a second, short row block
    x[5, 130:140] = 0.0
    xb = _bf16_bits_round(x)
    xf = _bits_to_f64(xb).astype(np.float32)
    for br in (1, 128):
        codes, scales = oracle.quantize_fp8_blocks(xb, br, lib=lib)
        assert scales.shape == ((130 + br - 1) // br, 2)
        for rb in range(scales.shape[0]):
            for b in range(2):
                blk = xf[rb * br:(rb + 1) * br, b * 128:(b + 1) * 128]
                amax = np.float32(np.max(np.abs(blk)))
                s = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
                assert scales[rb, b] == s, (br, rb, b)
                ref = torch.from_numpy((blk / s).astype(np.float32)).to(torch.float8_e4m3fn)
                got = codes[rb * br:(rb + 1) * br, b * 128:(b + 1) * 128]
                assert np.array_equal(got, ref.view(torch.uint8).numpy()), (br, rb, b)


def pin_fp8_block_logprob(lib):
    """Block-FP8 logprob: on inputs whose blocks quantise exactly (every block a
    different power-of-two scale) it equals the bf16 oracle, which the per-row
    fp8 oracle on the same inputs does not (the pin sees block scales); on random
    inputs it equals scipy's log-softmax of the block-dequantised logits."""
    rng = np.random.default_rng(44)
    ints = np.array([0, 1, 2, 3, 4, 5, 6, 7, 8, 12, 16, 32], np.float32)
    T, H, V = 3, 320, 300           # 3 k blocks (the last ragged), 3 W block rows (ragged)
    hb = _bf16_bits(_exact_block_operand(rng, T, H, 1, ints))
    wb = _bf16_bits(_exact_block_operand(rng, V, H, 128, ints))
    tg = rng.integers(0, V, T).astype(np.int32)
    qh, sh = oracle.quantize_fp8_blocks(hb, 1, lib=lib)
    qw, sw = oracle.quantize_fp8_blocks(wb, 128, lib=lib)
    assert len(np.unique(sh)) > 3 and len(np.unique(sw)) > 3   # scales differ by block
    assert np.all(np.log2(sh) == np.round(np.log2(sh)))        # exact powers of two
    a = oracle.logprob_fp8_block(qh, sh, qw, sw, tg, 0.5, lib=lib)
    b = oracle.logprob(hb, wb, tg, 0.5, lib=lib)
    for k in ("logp", "lse", "argmax"):
        assert np.allclose(a[k], b[k], rtol=1e-12, atol=1e-12), k
    qr, sr = oracle.quantize_fp8_rows(hb, lib=lib)
    qv, sv = oracle.quantize_fp8_rows(wb, lib=lib)
    c = oracle.logprob_fp8(qr, sr, qv, sv, tg, 0.5, lib=lib)
    assert not np.allclose(c["logp"], b["logp"], rtol=1e-6, atol=1e-6)
    tab = _e4m3_table()
    hr = _bf16_bits_round(rng.standard_normal((4, 256)).astype(np.float32))
    wr = _bf16_bits_round((0.05 * rng.standard_normal((260, 256))).astype(np.float32))
    qh, sh = oracle.quantize_fp8_blocks(hr, 1, lib=lib)
    qw, sw = oracle.quantize_fp8_blocks(wr, 128, lib=lib)
    tg = rng.integers(0, 260, 4).astype(np.int32)
    z = np.zeros((4, 260))
    for bk in range(2):
        ks = slice(bk * 128, (bk + 1) * 128)
        z += (tab[qh[:, ks]] @ tab[qw[:, ks]].T) * sh[:, bk].astype(np.float64)[:, None] * \
            sw[np.arange(260) // 128, bk].astype(np.float64)[None, :]
    r = oracle.logprob_fp8_block(qh, sh, qw, sw, tg, 1.0, lib=lib)
    assert np.allclose(r["lse"], scipy.special.logsumexp(z, axis=1), atol=1e-11)
    assert np.allclose(r["logp"], scipy.special.log_softmax(z, axis=1)[np.arange(4), tg], atol=1e-11)
    assert np.array_equal(r["argmax"], np.argmax(z, axis=1))


PINS = [pin_zero_weights, pin_one_hot_dominant, pin_shift_invariance, pin_temperature,
        pin_brute_force_exact, pin_scipy_logsumexp, pin_ignored_targets,
        pin_block_stats_and_merge, pin_worked_example, pin_stats_closed_forms,
        pin_backward_finite_differences, pin_backward_closed_forms, pin_entropy,
        pin_fp8_quantiser, pin_fp8_logprob, pin_fp8_block_quantiser, pin_fp8_block_logprob]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin, olib):
    pin(olib)


def test_tie_rows_of_tiny_input(olib):
    """The tiny workload's forced ties resolve to the lower vocabulary index."""
    import torch
    from invariant_token_logprob_gb300.inputs import tiny_inputs
    d = tiny_inputs(seed=0)
    rows = torch.cat([d["dup_src"], d["dup_dst"]]).numpy()
    r = oracle.logprob(d["h"], d["W"], d["targets"], 1.0, rows=rows, lib=olib)
    exp = np.concatenate([d["expected_tie_argmax"].numpy()] * 2)
    assert np.array_equal(r["argmax"], exp)
    assert np.all(r["top2gap"] == 0.0)
    # duplicated hidden rows give identical results
    n = len(rows) // 2
    for k in ("logp", "lse", "argmax"):
        if k == "logp":
            continue  # targets differ between the copies
        assert np.array_equal(r[k][:n], r[k][n:])


def test_pins_catch_planted_mistakes(tmp_path):
    """Each deliberate mistake of oracle.c (ORACLE_MUTANT 1..9: dropped term,
    divided temperature, highest-index ties, LSE without the max, flipped logp
    sign, swapped gap direction, sample variance, backward without inv_temp,
    unnormalised softmax in the backward, entropy without the LSE shift, fp8
    rounding up instead of to nearest) fails at least one pin."""
    for mutant in range(1, 14):
        path = str(tmp_path / f"liboracle_m{mutant}.so")
        oracle.build(path, mutant=mutant)
        lib = oracle.load(path)
        failed = []
        for pin in PINS:
            try:
                pin(lib)
            except AssertionError:
                failed.append(pin.__name__)
        assert failed, f"mutant {mutant} passed every pin"
