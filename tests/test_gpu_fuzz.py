"""Seeded random shapes through the forward entry points (GPU).

Twenty shapes drawn from one fixed seed cover both launch shapes and every
ragged edge at once:
- T in 1..700: single CTA and CTA pair, ragged row tiles;
- H a multiple of 8 up to 1024: ragged 64-element k blocks;
- V in 1..40000: ragged 256-column vocabulary tiles;
- inv_temp in [0.5, 2] as an fp32 value.

For each shape:
- rlk_logprob matches the oracle, on every row of the small shapes and on a
  seeded sample plus the tile edges of the larger ones;
- splitting the rows at a random point into two calls gives the same bits;
- rlk_logprob_entropy gives the forward's logp / lse / argmax bits, and an
  entropy within the entropy tests' tolerance of the oracle's;
- the vocabulary cut into R shards of whole tiles (R random, every shard
  non-empty), merged, gives the forward's bits.
Ten smaller shapes (H a multiple of 128) take the backward and both FP8
formats through the same kind of check.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bitwise, assert_parity, to_dev
from invariant_token_logprob_gb300.inputs import lm_head_inputs

pytestmark = pytest.mark.gpu

ENT_ATOL = 5e-4          # the entropy tests' bound
FULL_ORACLE_MACS = 2e9   # up to this T*H*V the oracle runs on every row


def _shapes(n=20, seed=20261203):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        T = int(g.choice([1, 2, 5, 16, 17, 127, 128, 129, 200, 255, 256, 257, 384, 511, 700])
                if i % 2 else g.integers(1, 701))
        H = int(8 * g.integers(1, 129))
        V = int(g.choice([1, 2, 255, 256, 257, 511, 4096, 4097]) if i % 3 == 0
                else g.integers(1, 40001))
        it = float(np.float32(g.uniform(0.5, 2.0)))
        out.append((T, H, V, it, 1000 + i))
    return out


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import invariant_token_logprob_gb300 as rlk
    rlk.lib()


def _np(xs):
    return tuple(x.cpu().numpy() for x in xs)


def _rows(T, H, V, seed):
    if T * H * V <= FULL_ORACLE_MACS:
        return None
    g = np.random.default_rng(seed)
    edges = [r for r in (0, 127, 128, 255, 256, T - 1) if r < T]
    return np.unique(np.concatenate([g.choice(T, min(T, 48), replace=False), edges]))


@pytest.mark.parametrize("T,H,V,it,seed", _shapes())
def test_random_shape(olib, T, H, V, it, seed):
    import invariant_token_logprob_gb300 as rlk
    d = lm_head_inputs(T, H, V, seed=seed, hidden="normal" if seed % 2 else "rms")
    dd = to_dev(d)
    what = f"T={T} H={H} V={V} inv_temp={it}"
    full = _np(rlk.logprob(dd["h"], dd["W"], dd["targets"], it))
    rlk.check_device_error()

    rows = _rows(T, H, V, seed)
    ref = oracle.logprob(d["h"], d["W"], d["targets"], it, rows=rows, lib=olib)
    assert_parity(full, ref, rows=rows, what=what)

    if T > 1:  # two calls, split at a random row
        c = int(np.random.default_rng(seed).integers(1, T))
        a = _np(rlk.logprob(dd["h"][:c].contiguous(), dd["W"], dd["targets"][:c].contiguous(), it))
        b = _np(rlk.logprob(dd["h"][c:].contiguous(), dd["W"], dd["targets"][c:].contiguous(), it))
        assert_bitwise(full, tuple(np.concatenate([x, y]) for x, y in zip(a, b)),
                       f"{what}: split at {c}")

    lp, lse, am, ent = rlk.logprob_entropy(dd["h"], dd["W"], dd["targets"], it)
    rlk.check_device_error()
    assert_bitwise(full, _np((lp, lse, am)), f"{what}: entropy call")
    ent = ent.cpu().numpy()
    ref_e = oracle.entropy(d["h"], d["W"], it, rows=rows, lib=olib)
    got_e = ent if rows is None else ent[rows]
    assert np.all(np.abs(got_e.astype(np.float64) - ref_e) <= ENT_ATOL), \
        f"{what}: entropy error {np.max(np.abs(got_e - ref_e)):.3g}"

    bn = rlk.vocab_tile()
    nvt = (V + bn - 1) // bn
    R = int(np.random.default_rng(seed + 1).integers(1, min(nvt, 8) + 1))
    nvt_s = (nvt + R - 1) // R
    R = (nvt + nvt_s - 1) // nvt_s  # every shard holds at least one tile
    # slots past the last tile stay NaN: the merge must not read them
    buf = torch.full((R, T, nvt_s, 4), float("nan"), dtype=torch.float32, device="cuda")
    for r in range(R):
        lo, hi = r * nvt_s * bn, min((r + 1) * nvt_s * bn, V)
        out = torch.empty((T, (hi - lo + bn - 1) // bn, 4), dtype=torch.float32, device="cuda")
        rlk.logprob_partials_shard(dd["h"], dd["W"][lo:hi].contiguous(), dd["targets"], V, lo, it,
                                   out=out)
        buf[r, :, : out.shape[1]] = out
    got = _np(rlk.lse_merge_sharded(buf, dd["targets"], V))
    rlk.check_device_error()
    assert_bitwise(full, got, f"{what}: {R} shards")


def _small_shapes(n=10, seed=20261204):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        T = int(g.choice([1, 4, 5, 128, 129, 256]) if i % 2 else g.integers(1, 301))
        H = int(128 * g.integers(1, 7))
        V = int(g.choice([1, 255, 257, 4097]) if i % 3 == 0 else g.integers(1, 6001))
        it = float(np.float32(g.uniform(0.5, 2.0)))
        out.append((T, H, V, it, 2000 + i))
    return out


@pytest.mark.parametrize("T,H,V,it,seed", _small_shapes())
def test_random_shape_backward_and_fp8(olib, T, H, V, it, seed):
    """Ten smaller random shapes (H a multiple of 128, as the fp8 formats need):
    the backward's dz, grad_h and grad_W within the backward tests' bf16 error
    model of the oracle; per-row and block FP8 logprobs against their oracle
    modes on the codes and scales the GPU quantisers wrote (which must equal
    the oracle's bit for bit)."""
    import invariant_token_logprob_gb300 as rlk
    d = lm_head_inputs(T, H, V, seed=seed, hidden="normal", w_std=0.05)
    dd = to_dev(d)
    what = f"T={T} H={H} V={V} inv_temp={it}"

    # backward, with the same bounds as the backward tests
    grad = torch.randn(T, generator=torch.Generator().manual_seed(seed)).float()
    _, lse, _ = rlk.logprob(dd["h"], dd["W"], dd["targets"], it)
    gh, gW, ws = rlk.logprob_backward(dd["h"], dd["W"], dd["targets"], lse, grad.cuda(), it)
    rlk.check_device_error()
    dz = rlk.backward_dz(ws, T, V).float().cpu().numpy().astype(np.float64)
    ref = oracle.logprob_backward(d["h"], d["W"], d["targets"], grad.double().numpy(), it,
                                  lib=olib)
    hf = d["h"].float().numpy().astype(np.float64)
    Wf = d["W"].float().numpy().astype(np.float64)
    g = grad.double().numpy()
    assert np.all(np.abs(dz - ref["dz"]) <= 2.0 ** -8 * np.abs(ref["dz"]) + 2e-5 * np.abs(g)[:, None]), \
        f"{what}: dz"
    bh = it * 2.0 ** -7 * (np.abs(ref["dz"]) @ np.abs(Wf)) + 1e-6
    assert np.all(np.abs(gh.cpu().numpy() - ref["dh"]) <= bh), f"{what}: grad_h"
    bw = it * 2.0 ** -7 * (np.abs(ref["dz"]).T @ np.abs(hf)) + 1e-6
    assert np.all(np.abs(gW.cpu().numpy() - ref["dW"]) <= bw), f"{what}: grad_W"

    # per-row FP8
    wq, wsc = rlk.quantize_fp8_weight(dd["W"])
    got = _np(rlk.logprob_fp8(dd["h"], wq, wsc, dd["targets"], it))
    rlk.check_device_error()
    qh, sh = oracle.quantize_fp8_rows(d["h"], lib=olib)
    qw, sw = oracle.quantize_fp8_rows(d["W"], lib=olib)
    assert np.array_equal(qw, rlk.unpack_fp8_weight(wq, V, H).cpu().numpy()), f"{what}: W codes"
    assert np.array_equal(sw.view(np.uint32), wsc.cpu().numpy().view(np.uint32)), f"{what}: W scales"
    assert_parity(got, oracle.logprob_fp8(qh, sh, qw, sw, d["targets"], it, lib=olib),
                  what=f"fp8 {what}")

    # block FP8
    bq, bs = rlk.quantize_fp8_weight_blocks(dd["W"])
    got = _np(rlk.logprob_fp8_block(dd["h"], bq, bs, dd["targets"], V, it))
    rlk.check_device_error()
    hc, hs = rlk.quantize_fp8_row_blocks(dd["h"])
    rhc, rhs = oracle.quantize_fp8_blocks(d["h"], 1, lib=olib)
    rwc, rws = oracle.quantize_fp8_blocks(d["W"], 128, lib=olib)
    assert np.array_equal(hc.cpu().numpy()[:T], rhc) and \
        np.array_equal(hs.cpu().numpy().view(np.uint32), rhs.view(np.uint32)), f"{what}: h blocks"
    assert np.array_equal(rlk.unpack_fp8_weight(bq, V, H).cpu().numpy(), rwc) and \
        np.array_equal(bs.cpu().numpy().view(np.uint32), rws.view(np.uint32)), f"{what}: W blocks"
    assert_parity(got, oracle.logprob_fp8_block(rhc, rhs, rwc, rws, d["targets"], it, lib=olib),
                  what=f"block fp8 {what}")
