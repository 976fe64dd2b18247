"""GPU tests of the logprob backward against the fp64 oracle.

Error model, from the arithmetic of the CUDA path: the logits are the
forward's fp32 logits, p = exp(z - lse) in fp32 (relative error ~1e-6), dz is
rounded once to bf16 (relative error <= 2^-9), and the two products are bf16 x
bf16 -> fp32 tensor-core GEMMs of the library.  So, elementwise,
  |dz_gpu - dz|  <= 2^-8 |dz| + 2e-5 |g|
  |dh_gpu - dh|  <= inv_temp 2^-7 sum_v |dz[t,v]| |W[v,k]| + 1e-6
  |dW_gpu - dW|  <= inv_temp 2^-7 sum_t |dz[t,v]| |h[t,k]| + 1e-6
(a factor 2 of margin over the bf16 rounding bound).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import to_dev
from invariant_token_logprob_gb300.inputs import lm_head_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import invariant_token_logprob_gb300 as rlk
    rlk.lib()


def _bf16_to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _run(d, grad, it, need_h=True, need_W=True, grad_W=None):
    import invariant_token_logprob_gb300 as rlk
    lp, lse, am = rlk.logprob(d["h"], d["W"], d["targets"], it)
    gh, gW, ws = rlk.logprob_backward(d["h"], d["W"], d["targets"], lse, grad, it,
                                      need_h=need_h, need_W=need_W, grad_W=grad_W)
    rlk.check_device_error()
    T, V = d["h"].shape[0], d["W"].shape[0]
    return gh, gW, rlk.backward_dz(ws, T, V)


def _check(d, grad, it, gh, gW, dz, what):
    hf, Wf = _bf16_to_f64(d["h"]), _bf16_to_f64(d["W"])
    ref = oracle.logprob_backward(d["h"].cpu(), d["W"].cpu(), d["targets"].cpu(),
                                  grad.cpu().double().numpy(), it)
    g = grad.cpu().double().numpy()
    dzg = dz.float().cpu().numpy().astype(np.float64)
    bz = 2.0 ** -8 * np.abs(ref["dz"]) + 2e-5 * np.abs(g)[:, None]
    assert np.all(np.abs(dzg - ref["dz"]) <= bz), f"{what}: dz"
    if gh is not None:
        bh = it * 2.0 ** -7 * (np.abs(ref["dz"]) @ np.abs(Wf)) + 1e-6
        err = np.abs(gh.cpu().numpy() - ref["dh"])
        assert np.all(err <= bh), f"{what}: dh worst ratio {np.max(err / bh):.3g}"
    if gW is not None:
        bw = it * 2.0 ** -7 * (np.abs(ref["dz"]).T @ np.abs(hf)) + 1e-6
        err = np.abs(gW.cpu().numpy() - ref["dW"])
        assert np.all(err <= bw), f"{what}: dW worst ratio {np.max(err / bw):.3g}"
    return ref


@pytest.mark.parametrize("T,H,V,seed", [(40, 192, 1000, 1), (3, 64, 777, 2), (130, 128, 1001, 3),
                                        (16, 256, 2048, 4)])
def test_backward_matches_oracle(T, H, V, seed):
    d = to_dev(lm_head_inputs(T, H, V, seed=seed, hidden="normal", w_std=0.05))
    d["targets"][0] = -1  # an ignored row
    it = float(np.float32(1 / 0.7)) if seed % 2 else 1.0
    grad = torch.randn(T, device="cuda", generator=torch.Generator("cuda").manual_seed(seed))
    gh, gW, dz = _run(d, grad, it)
    _check(d, grad, it, gh, gW, dz, f"T={T} H={H} V={V}")
    assert torch.all(dz[0] == 0) and torch.all(gh[0] == 0)


@pytest.mark.parametrize("T,H,V,it", [
    (40, 192, 20000, 1.0),                     # grad_h in 8 K ranges; H one ragged unit
    (300, 320, 3001, float(np.float32(1 / 0.7))),  # ragged T (2 pair units), H, V, k-blocks
    (257, 256, 70000, 1.0),                    # odd row tile of the last pair unit alone
    (7, 64, 129, 2.0),                         # smaller than one tile everywhere
])
def test_gemms_match_fp64_products_of_the_kernels_dz(T, H, V, it):
    """The two tensor-core products alone, against fp64 products of the dz the
    dz kernel wrote (so the bf16 rounding of dz is not part of the error): each
    element is an fp32 sum of exact bf16 products, so |error| stays within
    2^-13 of sum |terms| (the sum order is fixed but not the fp64 one); a wrong
    operand, index or k step would be off by O(1) of it."""
    import invariant_token_logprob_gb300 as rlk
    d = to_dev(lm_head_inputs(T, H, V, seed=T + V, hidden="normal", w_std=0.05))
    grad = torch.randn(T, device="cuda", generator=torch.Generator("cuda").manual_seed(T))
    base = torch.randn(V, H, device="cuda", generator=torch.Generator("cuda").manual_seed(V))
    gh, gW, dz = _run(d, grad, it, grad_W=base.clone())
    dz64 = dz.double().cpu()
    W64, h64 = d["W"].double().cpu(), d["h"].double().cpu()
    t = float(np.float32(it))
    ref_h = t * (dz64 @ W64)
    bound_h = 2.0 ** -13 * t * (dz64.abs() @ W64.abs()) + 1e-30
    assert torch.all((gh.double().cpu() - ref_h).abs() <= bound_h), "grad_h"
    ref_W = base.double().cpu() + t * (dz64.T @ h64)
    bound_W = 2.0 ** -13 * (base.double().cpu().abs() + t * (dz64.abs().T @ h64.abs())) + 1e-30
    assert torch.all((gW.double().cpu() - ref_W).abs() <= bound_W), "grad_W (accumulated)"
    # overwritten (the tiled-store path of the epilogue), and grad_h unchanged by it
    gh2, gW2, dz2 = _run(d, grad, it)
    assert torch.equal(dz2.view(torch.int16), dz.view(torch.int16)) and torch.equal(gh2, gh)
    ref_W2 = t * (dz64.T @ h64)
    bound_W2 = 2.0 ** -13 * t * (dz64.abs().T @ h64.abs()) + 1e-30
    assert torch.all((gW2.double().cpu() - ref_W2).abs() <= bound_W2), "grad_W (overwritten)"


def test_backward_accumulates_and_skips():
    d = to_dev(lm_head_inputs(20, 64, 500, seed=7))
    grad = torch.randn(20, device="cuda")
    gh, gW, dz = _run(d, grad, 1.0)
    base = torch.randn(500, 64, device="cuda")
    _, gW2, _ = _run(d, grad, 1.0, need_h=False, grad_W=base.clone())
    assert torch.allclose(gW2, base + gW, rtol=1e-6, atol=1e-6)
    gh3, gW3, _ = _run(d, grad, 1.0, need_W=False)
    assert gW3 is None and torch.equal(gh3, gh)


def test_backward_is_deterministic():
    d = to_dev(lm_head_inputs(300, 256, 3000, seed=8))
    grad = torch.randn(300, device="cuda")
    a = _run(d, grad, 1.0)
    b = _run(d, grad, 1.0)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y)


def test_autograd_function_matches_oracle():
    import invariant_token_logprob_gb300 as rlk
    d = to_dev(lm_head_inputs(24, 128, 900, seed=9, hidden="normal", w_std=0.05))
    h = d["h"].clone().requires_grad_(True)
    W = d["W"].clone().requires_grad_(True)
    lp = rlk.selected_token_logprob(h, W, d["targets"], 1.0)
    ref_lp, _, _ = rlk.logprob(d["h"], d["W"], d["targets"], 1.0)
    assert torch.equal(lp.detach(), ref_lp)  # forward values are the kernel's
    w = torch.linspace(-1, 1, 24, device="cuda")
    (lp * w).sum().backward()
    ref = oracle.logprob_backward(d["h"].cpu(), d["W"].cpu(), d["targets"].cpu(),
                                  w.cpu().double().numpy(), 1.0)
    Wf, hf = _bf16_to_f64(d["W"]), _bf16_to_f64(d["h"])
    # one more bf16 rounding: the gradients are returned in the parameters' dtype
    bh = 2.0 ** -7 * (np.abs(ref["dz"]) @ np.abs(Wf)) + 2.0 ** -8 * np.abs(ref["dh"]) + 1e-6
    bw = 2.0 ** -7 * (np.abs(ref["dz"]).T @ np.abs(hf)) + 2.0 ** -8 * np.abs(ref["dW"]) + 1e-6
    assert h.grad.dtype == torch.bfloat16 and W.grad.dtype == torch.bfloat16
    assert np.all(np.abs(_bf16_to_f64(h.grad) - ref["dh"]) <= bh)
    assert np.all(np.abs(_bf16_to_f64(W.grad) - ref["dW"]) <= bw)


@pytest.mark.slow
def test_backward_full_size_sampled_rows_and_invariant():
    """T=4096, H=4096, V=151936: dh on sampled rows against the oracle (dh[t]
    depends on row t only), and sum_v dW[v,:] = 0 (every dz row sums to 0)."""
    import invariant_token_logprob_gb300 as rlk
    T, H, V = 4096, 4096, 151936
    d = lm_head_inputs(T, H, V, seed=11, device="cuda")
    grad = torch.randn(T, device="cuda", generator=torch.Generator("cuda").manual_seed(1))
    lp, lse, am = rlk.logprob(d["h"], d["W"], d["targets"], 1.0)
    gh, gW, ws = rlk.logprob_backward(d["h"], d["W"], d["targets"], lse, grad, 1.0)
    rlk.check_device_error()
    rows = np.array([0, 1, 2047, T - 1])
    sub = oracle.logprob_backward(d["h"][rows].cpu(), d["W"].cpu(), d["targets"][rows].cpu(),
                                  grad[rows].cpu().double().numpy(), 1.0)
    Wf = d["W"].float().cpu().numpy().astype(np.float64)
    bh = 2.0 ** -7 * (np.abs(sub["dz"]) @ np.abs(Wf)) + 1e-6
    assert np.all(np.abs(gh[rows].cpu().numpy() - sub["dh"]) <= bh)
    dz = rlk.backward_dz(ws, T, V)
    dzf = dz[rows].float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(dzf - sub["dz"]) <= 2.0 ** -8 * np.abs(sub["dz"]) +
                  2e-5 * np.abs(grad[rows].cpu().numpy())[:, None])
    # sum over the vocabulary of dW: zero up to the bf16 rounding of dz
    # (|sum_v dz_gpu[t,v]| <= 2^-9 sum_v |dz[t,v]|; a factor 2 of margin)
    col = gW.double().sum(0).cpu().numpy()
    scale = (dz.float().abs().sum(1).double() @ d["h"].double().abs()).cpu().numpy()
    assert np.all(np.abs(col) <= 2.0 ** -8 * scale + 1e-3)
