"""Seeded synthetic inputs shaped like an LLM LM head (e.g. Qwen3-8B: H=4096,
V=151936).  No model weights or datasets exist here, so these stand in for them.

This module holds data construction only -- no part of the logprob method's
arithmetic -- so both the CUDA path and the CPU oracle can be fed the same bytes
from it.  Every draw comes from one ``torch.Generator`` seeded explicitly, in a
fixed order (W, h, targets, then the optional extras), on the device asked for.

Recipe (all bf16 rounding is torch's round-to-nearest-even):
  W       ~ N(0, w_std) in fp32, rounded to bf16 ([V,H], row-major)
  h       ~ N(0, 1) in fp32; with hidden="rms" each row is divided by its RMS
            (an RMS-normalised final hidden state), then rounded to bf16 ([T,H])
  targets ~ uniform int32 in [0, V)
  outliers: a seeded choice of round(outlier_frac*T) rows is multiplied by
            outlier_scale after rounding (x8 is exact in bf16)
  mask    : int8, 1 = valid; a seeded choice of round(mask_zero_frac*T) zeros
"""
from __future__ import annotations

import torch

# Vocabulary index pairs (v_star, v_copy) used to force exact argmax ties:
# v_copy receives a bit-exact copy of W[v_star].  Five copies land above their
# source and three below; several cross 32-, 128- and 256-column boundaries.
TIE_PAIRS = ((100, 37), (300, 301), (511, 512), (700, 640),
             (905, 1000), (5, 1023), (767, 768), (400, 129))


def lm_head_inputs(T: int, H: int, V: int, seed: int = 0, device="cpu",
                   hidden: str = "rms", w_std: float = 0.02,
                   outlier_frac: float = 0.0, outlier_scale: float = 8.0,
                   mask_zero_frac: float = 0.0) -> dict:
    """Return dict(h=[T,H] bf16, W=[V,H] bf16, targets=[T] int32, mask=[T] int8,
    outlier_rows=int64 tensor) on `device`."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    W = (torch.randn(V, H, generator=g, device=device, dtype=torch.float32) * w_std).to(torch.bfloat16)
    h = torch.randn(T, H, generator=g, device=device, dtype=torch.float32)
    if hidden == "rms":
        h = h * torch.rsqrt(h.pow(2).mean(dim=-1, keepdim=True))
    elif hidden != "normal":
        raise ValueError("hidden must be 'rms' or 'normal'")
    h = h.to(torch.bfloat16)
    targets = torch.randint(0, V, (T,), generator=g, device=device, dtype=torch.int32)
    n_out = int(round(outlier_frac * T))
    outlier_rows = torch.empty(0, dtype=torch.int64, device=device)
    if n_out > 0:
        outlier_rows = torch.randperm(T, generator=g, device=device)[:n_out].sort().values
        h[outlier_rows] = h[outlier_rows] * outlier_scale
    mask = torch.ones(T, dtype=torch.int8, device=device)
    n_zero = int(round(mask_zero_frac * T))
    if n_zero > 0:
        zero_rows = torch.randperm(T, generator=g, device=device)[:n_zero]
        mask[zero_rows] = 0
    return dict(h=h, W=W, targets=targets, mask=mask, outlier_rows=outlier_rows)


def tiny_inputs(seed: int = 0, device="cpu", T: int = 64, H: int = 256, V: int = 1024) -> dict:
    """The small case: h ~ N(0,1) (not normalised), W ~ N(0, 0.02), inv_temp 1.

    Eight hidden rows are copied to eight other positions (the same row at two
    batch positions).  For those eight source rows, vocabulary row v_star is set
    to bf16(0.05 * h[t]) -- which makes it that row's clear maximum -- and copied
    bit-exactly to v_copy, so the row's maximum is an exact two-way tie whose
    expected argmax is min(v_star, v_copy).  Returns the lm_head_inputs dict plus
    tie_rows, dup_src, dup_dst and expected_tie_argmax.
    """
    if V < 1024 or T < 16:
        raise ValueError("tiny_inputs needs V >= 1024 and T >= 16")
    d = lm_head_inputs(T, H, V, seed=seed, device=device, hidden="normal")
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) + 1)
    perm = torch.randperm(T, generator=g, device=device)
    src, dst = perm[:8], perm[8:16]
    h, W = d["h"], d["W"]
    h[dst] = h[src]
    expected = []
    for i, (vs, vc) in enumerate(TIE_PAIRS):
        t = int(src[i])
        W[vs] = (h[t].float() * 0.05).to(torch.bfloat16)
        W[vc] = W[vs]
        expected.append(min(vs, vc))
    d.update(tie_rows=src.clone(), dup_src=src.clone(), dup_dst=dst.clone(),
             expected_tie_argmax=torch.tensor(expected, dtype=torch.int64))
    return d
