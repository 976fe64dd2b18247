"""GPU tests of the block-scaled FP8 (W8A8) LM-head variant (1 x 128 activation
blocks, 128 x 128 weight blocks).

* Quantisation is integer work: the e4m3 codes and fp32 block scales of h and
  of the tile-packed W must equal the oracle's bit for bit.
* The logprob is compared with the oracle's fp64 block-FP8 logprob on the same
  codes and scales under the parity tolerances of the bf16 path; what remains
  is the fp32 summation on the tensor core within each 128-element block and
  the fp32 promotion (scale and add) across blocks.
* The batch-invariance contract holds for this variant too: bitwise across
  chunkings, batch positions and repetition.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bitwise, assert_parity, to_dev
from invariant_token_logprob_gb300.inputs import lm_head_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import invariant_token_logprob_gb300 as rlk
    rlk.lib()


def _np(xs):
    return tuple(x.cpu().numpy() for x in xs)


def _bits(x):
    return np.ascontiguousarray(x).view(np.uint32)


def test_block_quantisers_are_bit_exact(olib):
    import invariant_token_logprob_gb300 as rlk
    g = torch.Generator().manual_seed(7)
    x = torch.randn(37, 512, generator=g) * torch.logspace(-4, 3, 37)[:, None]
    x[:, 128:256] *= 50.0                        # blocks of one row with different scales
    x[3] = 0.0                                   # all-zero blocks: scale 1, codes 0
    x[4, :5] = torch.tensor([448.0, -448.0, 1e-30, 3.0, -0.0])
    x[5, 256:384] = 0.0
    xb = x.to(torch.bfloat16)
    codes, scales = rlk.quantize_fp8_row_blocks(xb.cuda())
    torch.cuda.synchronize()
    rc, rs = oracle.quantize_fp8_blocks(xb, 1, lib=olib)
    assert np.array_equal(_bits(scales.cpu().numpy()), _bits(rs))
    assert np.array_equal(codes.cpu().numpy(), rc)
    for V, H in ((1000, 384), (300, 256), (256, 128)):   # ragged and whole last tiles
        W = (torch.randn(V, H, generator=g) * torch.logspace(-3, 1, V)[:, None]).to(torch.bfloat16)
        W[:, :128] *= 16
        packed, ws = rlk.quantize_fp8_weight_blocks(W.cuda())
        torch.cuda.synchronize()
        wc, wsr = oracle.quantize_fp8_blocks(W, 128, lib=olib)
        assert np.array_equal(_bits(ws.cpu().numpy()), _bits(wsr)), (V, H)
        unp = rlk.unpack_fp8_weight(packed, V, H).cpu().numpy()
        assert np.array_equal(unp, wc), (V, H)
        nt = (V + 255) // 256
        full = packed.view(nt, H // 128, 256, 128).permute(0, 2, 1, 3).reshape(nt * 256, H)
        assert torch.all(full[V:] == 0)          # padding rows of the last tile: zero codes
    rlk.check_device_error()


def test_block_weight_quantiser_division_is_ieee_on_its_whole_input_domain():
    """Exhaustive, like the per-row quantiser's test: for every positive finite
    bf16 amax, one 128-row band of W holds every finite bf16 value with
    |x| <= amax (the others 0) spread over four 128 x 128 blocks, so the blocks
    see about 2.1e9 (x, block scale) pairs in all.  The reference takes each
    block's own max, its scale max / 448 by IEEE division (1 for a zero block)
    and the codes as torch's float8 e4m3 cast of the IEEE quotient x / scale,
    all on the same device; scales and codes must match bit for bit, signed
    zeros included."""
    import invariant_token_logprob_gb300 as rlk
    pat = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    base = torch.where(torch.isfinite(pat.float()), pat, torch.zeros_like(pat)).cuda()
    mags = pat[1:0x7F80].float().cuda()  # every positive finite bf16 value, ascending
    absb = base.float().abs()
    A = 512
    for c0 in range(0, mags.numel(), A):
        amax = mags[c0:c0 + A]
        n = amax.numel()
        vals = torch.where(absb[None, :] <= amax[:, None], base[None, :],
                           torch.zeros_like(base)[None, :])
        # band a: block kb holds values kb * 16384 + (row * 128 + col)
        W = vals.view(n, 4, 128, 128).permute(0, 2, 1, 3).reshape(n * 128, 512).contiguous()
        packed, scales = rlk.quantize_fp8_weight_blocks(W)
        codes = rlk.unpack_fp8_weight(packed, n * 128, 512)
        bmax = W.float().abs().view(n, 128, 4, 128).amax(dim=(1, 3))  # [band, k block]
        ref_s = torch.where(bmax > 0, bmax / torch.full_like(bmax, 448.0), torch.ones_like(bmax))
        assert torch.equal(scales.view(torch.int32), ref_s.view(torch.int32)), c0
        sfull = ref_s[:, None, :, None].expand(n, 128, 4, 128).reshape(n * 128, 512)
        ref = (W.float() / sfull).to(torch.float8_e4m3fn).view(torch.uint8)
        bad = (codes != ref).nonzero()
        assert bad.numel() == 0, (c0, bad[:5].tolist())
    rlk.check_device_error()


def _quantised(rlk, d):
    """GPU block codes/scales of h and W (the ones the kernel reads), on the host."""
    hc, hs = rlk.quantize_fp8_row_blocks(d["h"])
    wp, ws = rlk.quantize_fp8_weight_blocks(d["W"])
    V, H = d["W"].shape
    wc = rlk.unpack_fp8_weight(wp, V, H)
    torch.cuda.synchronize()
    return (hc.cpu().numpy(), hs.cpu().numpy(), wc.cpu().numpy(), ws.cpu().numpy()), wp, ws


@pytest.mark.parametrize("T,H,V,it", [(64, 256, 1000, 1.0),
                                      (300, 512, 3000, float(np.float32(1 / 0.7))),
                                      (5, 128, 257, 2.0),
                                      (130, 384, 700, 1.0),
                                      # CTA pair: the last vocabulary tile's odd half lies
                                      # past V (not copied), one k block
                                      (200, 128, 2100, 1.0)])
def test_block_fp8_logprob_matches_oracle(olib, T, H, V, it):
    import invariant_token_logprob_gb300 as rlk
    d = to_dev(lm_head_inputs(T, H, V, seed=T + H, hidden="normal", w_std=0.05))
    (hc, hs, wc, ws_), wp, ws = _quantised(rlk, d)
    got = _np(rlk.logprob_fp8_block(d["h"], wp, ws, d["targets"], V, it))
    rlk.check_device_error()
    ref = oracle.logprob_fp8_block(hc, hs, wc, ws_, d["targets"].cpu(), it, lib=olib)
    assert_parity(got, ref, what=f"block fp8 T={T} H={H} V={V}")


@pytest.mark.parametrize("H", [128, 384, 4096])
def test_block_fp8_decode_quantises_h_in_the_kernel(olib, H):
    """Calls of at most 16 rows quantise h in the block-FP8 kernel (1 x 128
    blocks, two work items per row).  Their rows must carry the bits of a
    32-row call, which runs the block quantiser kernel, and match the oracle
    on the GPU quantiser's codes.  H = 128 is one k block (the second half of
    each row empty), H = 384 an odd number of blocks.  A zero row and a tiny
    row check the scale-1 and subnormal paths."""
    import invariant_token_logprob_gb300 as rlk
    T, V = 32, 1000
    d = to_dev(lm_head_inputs(T, H, V, seed=H + 5, hidden="normal", w_std=0.05))
    d["h"][2] = 0.0
    d["h"][3] = (d["h"][3].float() * 1e-30).to(torch.bfloat16)
    (hc, hs, wc, ws_), wp, ws = _quantised(rlk, d)
    full = _np(rlk.logprob_fp8_block(d["h"], wp, ws, d["targets"], V))
    rlk.check_device_error()
    ref = oracle.logprob_fp8_block(hc, hs, wc, ws_, d["targets"].cpu(), 1.0, lib=olib)
    assert_parity(full, ref, what=f"block fp8 H={H}")
    for c in (1, 2, 3, 4, 5, 8, 15, 16):
        parts = [_np(rlk.logprob_fp8_block(d["h"][i:i + c].contiguous(), wp, ws,
                                           d["targets"][i:i + c].contiguous(), V))
                 for i in range(0, T, c)]
        got = tuple(np.concatenate([p[k] for p in parts]) for k in range(3))
        assert_bitwise(full, got, f"H={H}, chunks of {c}")
    rlk.check_device_error()


def test_block_fp8_batch_invariance():
    import invariant_token_logprob_gb300 as rlk
    T, H, V = 300, 512, 5000
    d = to_dev(lm_head_inputs(T, H, V, seed=77))
    wp, ws = rlk.quantize_fp8_weight_blocks(d["W"])
    full = _np(rlk.logprob_fp8_block(d["h"], wp, ws, d["targets"], V))
    for c in (1, 7, 128, 129):
        parts = [_np(rlk.logprob_fp8_block(d["h"][i:i + c].contiguous(), wp, ws,
                                           d["targets"][i:i + c].contiguous(), V))
                 for i in range(0, T, c)]
        got = tuple(np.concatenate([p[k] for p in parts]) for k in range(3))
        assert_bitwise(full, got, f"chunks of {c}")
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(1)).cuda()
    pg = _np(rlk.logprob_fp8_block(d["h"][perm].contiguous(), wp, ws, d["targets"][perm].contiguous(), V))
    inv = torch.argsort(perm).cpu().numpy()
    assert_bitwise(full, tuple(x[inv] for x in pg), "permuted rows")
    assert_bitwise(full, _np(rlk.logprob_fp8_block(d["h"], wp, ws, d["targets"], V)), "repeat")
    rlk.check_device_error()


@pytest.mark.slow
def test_block_fp8_full_size_sampled_rows_and_decode(olib):
    """T=4096, H=4096, V=151936: oracle parity on 64 seeded rows (plus the tile
    edges) on the kernel's own codes and scales; one-row decode calls give the
    bits of the T=4096 call."""
    import invariant_token_logprob_gb300 as rlk
    T, H, V = 4096, 4096, 151936
    d = lm_head_inputs(T, H, V, seed=21, device="cuda")
    (hc, hs, wc, ws_), wp, ws = _quantised(rlk, d)
    full = _np(rlk.logprob_fp8_block(d["h"], wp, ws, d["targets"], V))
    rlk.check_device_error()
    rows = np.unique(np.concatenate([np.random.default_rng(3).choice(T, 64, replace=False),
                                     [0, 127, 128, T - 1]]))
    ref = oracle.logprob_fp8_block(hc, hs, wc, ws_, d["targets"].cpu(), 1.0, rows=rows, lib=olib)
    assert_parity(full, ref, rows=rows, what="block fp8 T=4096 sampled rows")
    for t in (0, 1, 2047, T - 1):
        one = _np(rlk.logprob_fp8_block(d["h"][t:t + 1].contiguous(), wp, ws,
                                        d["targets"][t:t + 1].contiguous(), V))
        assert_bitwise(tuple(x[t:t + 1] for x in full), one, f"decode row {t}")
    rlk.check_device_error()
