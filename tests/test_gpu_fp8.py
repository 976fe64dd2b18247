"""GPU tests of the FP8 (W8A8) LM-head variant.

* Quantisation is integer work: e4m3 codes and fp32 scales must equal the
  oracle's bit for bit (both take the rounding decision on the same fp32
  quotient x / s).
* The logprob is compared with the oracle's fp64 logprob on the same codes and
  scales, under the parity tolerances of the bf16 path (|dlogp| <= 5e-4,
  |dlse| <= 1e-5 max(1, |lse|), argmax exact where the top-2 gap > 1e-3): the
  only difference left is the fp32 accumulation of exact code products.
* The batch-invariance contract holds for this variant too (bitwise).
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


def test_quantiser_codes_and_scales_are_bit_exact(olib):
    import invariant_token_logprob_gb300 as rlk
    g = torch.Generator().manual_seed(5)
    x = torch.randn(37, 4096, generator=g) * torch.logspace(-4, 3, 37)[:, None]
    x[3] = 0.0                                    # all-zero row: scale 1, codes 0
    x[4, :5] = torch.tensor([448.0, -448.0, 1e-30, 3.0, -0.0])
    xb = x.to(torch.bfloat16)
    codes, scales = rlk.quantize_fp8_rows(xb.cuda())
    torch.cuda.synchronize()
    rc, rs = oracle.quantize_fp8_rows(xb, lib=olib)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_quantiser_division_is_ieee_on_its_whole_input_domain():
    """Exhaustive: a row's scale is s = amax / 448 for a bf16 amax, and its codes
    are the e4m3 RNE of the fp32 IEEE quotient x / s for bf16 x with |x| <= amax.
    Every positive finite bf16 amax is taken, each row holding every finite bf16
    value with |x| <= amax (the others replaced by 0, so the row's amax is
    exactly that value): about 2.1e9 (x, s) pairs.  The reference is torch's
    division by a device tensor (true IEEE division) and its float8 e4m3 cast,
    computed on the same device; scales and codes must match bit for bit, signed
    zeros included."""
    import invariant_token_logprob_gb300 as rlk
    pat = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    base = torch.where(torch.isfinite(pat.float()), pat, torch.zeros_like(pat)).cuda()
    mags = pat[1:0x7F80].float().cuda()  # every positive finite bf16 value, ascending
    absb = base.float().abs()
    for c0 in range(0, mags.numel(), 512):
        amax = mags[c0:c0 + 512]
        rows = torch.where(absb[None, :] <= amax[:, None], base[None, :],
                           torch.zeros_like(base)[None, :]).contiguous()
        codes, scales = rlk.quantize_fp8_rows(rows)
        ref_s = amax / torch.full_like(amax, 448.0)
        assert torch.equal(scales.view(torch.int32), ref_s.view(torch.int32)), c0
        ref = (rows.float() / scales[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
        bad = (codes != ref).nonzero()
        assert bad.numel() == 0, (c0, bad[:5].tolist())
    rlk.check_device_error()


def test_weight_quantiser_division_is_ieee_on_its_whole_input_domain():
    """Exhaustive for the weight quantiser (rows in registers, H = 4096): for
    every positive finite bf16 amax, 16 rows of W hold every finite bf16 value
    with |x| <= amax (the others 0), so the rows see about 2.1e9 (x, row
    scale) pairs in all.  The reference takes each row's own max, its scale
    max / 448 by IEEE division (1 for a zero row) and the codes as torch's
    float8 e4m3 cast of the IEEE quotient x / scale, all on the same device;
    scales and unpacked codes must match bit for bit, signed zeros included."""
    import invariant_token_logprob_gb300 as rlk
    pat = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    base = torch.where(torch.isfinite(pat.float()), pat, torch.zeros_like(pat)).cuda()
    mags = pat[1:0x7F80].float().cuda()  # every positive finite bf16 value, ascending
    absb = base.float().abs()
    A, H = 128, 4096
    for c0 in range(0, mags.numel(), A):
        amax = mags[c0:c0 + A]
        n = amax.numel()
        W = torch.where(absb[None, :] <= amax[:, None], base[None, :],
                        torch.zeros_like(base)[None, :]).reshape(n * 16, H).contiguous()
        packed, scales = rlk.quantize_fp8_weight(W)
        codes = rlk.unpack_fp8_weight(packed, n * 16, H)
        rmax = W.float().abs().amax(dim=1)
        ref_s = torch.where(rmax > 0, rmax / torch.full_like(rmax, 448.0), torch.ones_like(rmax))
        assert torch.equal(scales.view(torch.int32), ref_s.view(torch.int32)), c0
        ref = (W.float() / ref_s[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
        bad = (codes != ref).nonzero()
        assert bad.numel() == 0, (c0, bad[:5].tolist())
    rlk.check_device_error()


@pytest.mark.parametrize("H", [384, 5120])  # rows in registers / the two-pass kernel (H > 4096)
def test_weight_quantiser_both_kernels_bit_exact(olib, H):
    """The weight quantiser keeps a row in one warp's registers up to H = 4096
    and takes the two-pass kernel above; both must give the oracle's codes and
    scales, with ragged last tiles (V = 777) and rows of very different
    magnitude."""
    import invariant_token_logprob_gb300 as rlk
    V = 777
    g = torch.Generator().manual_seed(H)
    W = (torch.randn(V, H, generator=g) * torch.logspace(-6, 2, V)[:, None]).to(torch.bfloat16)
    W[5] = 0.0
    packed, scales = rlk.quantize_fp8_weight(W.cuda())
    torch.cuda.synchronize()
    rc, rs = oracle.quantize_fp8_rows(W, lib=olib)
    assert np.array_equal(rlk.unpack_fp8_weight(packed, V, H).cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert torch.all(rlk.unpack_fp8_weight(packed, 1024, H)[V:] == 0)
    rlk.check_device_error()


def test_packed_weight_codes_are_bit_exact_and_padded_with_zeros(olib):
    """The tile-packed fp8 weight holds the oracle's row codes (after unpacking)
    and zero codes in the padding rows of the last vocabulary tile."""
    import invariant_token_logprob_gb300 as rlk
    V, H = 1000, 384
    W = (torch.randn(V, H, generator=torch.Generator().manual_seed(6)) * 0.02).to(torch.bfloat16)
    packed, scales = rlk.quantize_fp8_weight(W.cuda())
    torch.cuda.synchronize()
    assert packed.numel() == 1024 * H
    rc, rs = oracle.quantize_fp8_rows(W, lib=olib)
    assert np.array_equal(rlk.unpack_fp8_weight(packed, V, H).cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    full = rlk.unpack_fp8_weight(packed, 1024, H)  # including the padding rows
    assert torch.all(full[V:] == 0)


@pytest.mark.parametrize("T,H,V,seed", [(64, 256, 1024, 1), (3, 128, 777, 2), (130, 512, 3001, 3),
                                        (2, 4096, 151936, 4), (300, 384, 2049, 5)])
def test_fp8_logprob_matches_oracle(T, H, V, seed, olib):
    import invariant_token_logprob_gb300 as rlk
    d = to_dev(lm_head_inputs(T, H, V, seed=seed))
    it = float(np.float32(1 / 0.7)) if seed % 2 else 1.0
    wq, ws = rlk.quantize_fp8_weight(d["W"])
    gpu = _np(rlk.logprob_fp8(d["h"], wq, ws, d["targets"], it))
    rlk.check_device_error()
    qh, sh = oracle.quantize_fp8_rows(d["h"].cpu(), lib=olib)
    qw, sw = oracle.quantize_fp8_rows(d["W"].cpu(), lib=olib)
    assert np.array_equal(qw, rlk.unpack_fp8_weight(wq, V, H).cpu().numpy())
    ref = oracle.logprob_fp8(qh, sh, qw, sw, d["targets"].cpu(), it, lib=olib)
    assert_parity(gpu, ref, what=f"fp8 T={T} H={H} V={V}")


def test_fp8_batch_invariance_small():
    import invariant_token_logprob_gb300 as rlk
    d = to_dev(lm_head_inputs(64, 256, 3000, seed=9))
    wq, ws = rlk.quantize_fp8_weight(d["W"])
    full = _np(rlk.logprob_fp8(d["h"], wq, ws, d["targets"]))
    for c in (1, 5, 16, 17, 63):
        parts = [_np(rlk.logprob_fp8(d["h"][i:i + c].contiguous(), wq, ws,
                                     d["targets"][i:i + c].contiguous())) for i in range(0, 64, c)]
        got = tuple(np.concatenate([p[k] for p in parts]) for k in range(3))
        assert_bitwise(full, got, f"fp8 chunk={c}")


def test_fp8_pair_and_single_cta_calls_agree_bitwise():
    """T = 300 runs as CTA pairs (two row tiles per unit; the odd tile of the
    last unit lies past the padded h and is not copied), H = 384 gives an odd
    number of 128-element k-blocks (a half-filled last stage), V = 2049 a
    one-column last vocabulary tile whose odd half is not copied.  Chunks of
    at most 128 rows run as single CTAs: every row's bits must agree."""
    import invariant_token_logprob_gb300 as rlk
    d = to_dev(lm_head_inputs(300, 384, 2049, seed=21))
    wq, ws = rlk.quantize_fp8_weight(d["W"])
    full = _np(rlk.logprob_fp8(d["h"], wq, ws, d["targets"]))
    for c in (1, 100, 128, 129, 150):
        parts = [_np(rlk.logprob_fp8(d["h"][i:i + c].contiguous(), wq, ws,
                                     d["targets"][i:i + c].contiguous())) for i in range(0, 300, c)]
        got = tuple(np.concatenate([p[k] for p in parts]) for k in range(3))
        assert_bitwise(full, got, f"fp8 T=300 chunk={c}")


@pytest.mark.parametrize("H", [128, 384, 4096, 5120])
def test_fp8_decode_calls_quantise_h_in_the_kernel(olib, H):
    """Calls of at most 4 rows with H <= 4096 quantise h inside the LM-head
    kernel (H = 5120 takes the quantiser kernel).  Same codes and scales as the
    quantiser, so every row's bits must equal those of a 40-row call (quantiser
    kernel, single CTA), including an all-zero row and a row whose scale takes
    the IEEE-division path, and the rows must match the oracle on the
    quantiser's codes."""
    import invariant_token_logprob_gb300 as rlk
    T, V = 40, 700
    d = to_dev(lm_head_inputs(T, H, V, seed=H))
    d["h"][5] = 0.0                                  # all-zero row: scale 1, codes 0
    d["h"][6] *= 1e-30                               # tiny row: the IEEE-division path
    d["h"][7, ::3] = -d["h"][7, ::3]
    wq, ws = rlk.quantize_fp8_weight(d["W"])
    full = _np(rlk.logprob_fp8(d["h"], wq, ws, d["targets"]))
    for c in (1, 2, 3, 4, 16):
        parts = [_np(rlk.logprob_fp8(d["h"][i:i + c].contiguous(), wq, ws,
                                     d["targets"][i:i + c].contiguous())) for i in range(0, T, c)]
        got = tuple(np.concatenate([p[k] for p in parts]) for k in range(3))
        assert_bitwise(full, got, f"fp8 H={H} chunk={c}")
    rlk.check_device_error()
    qh, sh = oracle.quantize_fp8_rows(d["h"].cpu(), lib=olib)
    qw, sw = oracle.quantize_fp8_rows(d["W"].cpu(), lib=olib)
    ref = oracle.logprob_fp8(qh, sh, qw, sw, d["targets"].cpu(), 1.0, lib=olib)
    assert_parity(full, ref, what=f"fp8 H={H}")


@pytest.mark.slow
def test_fp8_full_size_parity_and_invariance(olib):
    import invariant_token_logprob_gb300 as rlk
    T, H, V = 4096, 4096, 151936
    d = lm_head_inputs(T, H, V, seed=13, device="cuda")
    wq, ws = rlk.quantize_fp8_weight(d["W"])
    full = _np(rlk.logprob_fp8(d["h"], wq, ws, d["targets"]))
    rows = np.array([0, 1, 1000, 2048, T - 1])
    hs = d["h"][torch.from_numpy(rows).cuda()].cpu()
    qh, sh = oracle.quantize_fp8_rows(hs, lib=olib)
    ref = oracle.logprob_fp8(qh, sh, rlk.unpack_fp8_weight(wq, V, H).cpu().numpy(), ws.cpu().numpy(),
                             d["targets"][torch.from_numpy(rows).cuda()].cpu(), 1.0, lib=olib)
    assert_parity(tuple(x[rows] for x in full), ref, what="fp8 T=4096")
    seq = [_np(rlk.logprob_fp8(d["h"][i:i + 512].contiguous(), wq, ws,
                               d["targets"][i:i + 512].contiguous())) for i in range(0, T, 512)]
    assert_bitwise(full, tuple(np.concatenate([p[k] for p in seq]) for k in range(3)), "fp8 8x512")
    one = _np(rlk.logprob_fp8(d["h"][7:8].contiguous(), wq, ws, d["targets"][7:8].contiguous()))
    assert_bitwise(tuple(x[7:8] for x in full), one, "fp8 T=1 vs T=4096")
    # 4 rows: the largest call whose h the LM-head kernel quantises itself
    four = _np(rlk.logprob_fp8(d["h"][100:104].contiguous(), wq, ws,
                               d["targets"][100:104].contiguous()))
    assert_bitwise(tuple(x[100:104] for x in full), four, "fp8 T=4 vs T=4096")
    rlk.check_device_error()
