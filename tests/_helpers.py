"""Shared test helpers: tolerances and comparisons against the fp64 oracle.

Tolerances (the target's stated bar): bf16 outputs within max-abs 2e-2 and mean-abs 2e-3 of
the oracle; LSE within 1e-3 relative (|d| <= 1e-3 * max(1, |ref|)); gradients within
5e-2 * max|ref grad| per tensor; tile-visit sets bit-exact. A gradient that is exactly zero
in exact arithmetic (one visible key: dS = P (dP - D) = 0) is held to an absolute floor of
5e-2 * 1e-4, far below any non-degenerate gradient of unit-variance inputs.
"""
import numpy as np
import torch

import attention_attn_fwd_bwd_gb300 as af
from attention_attn_fwd_bwd_gb300 import inputs

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_REL = 1e-3
GRAD_REL_MAX = 5e-2
GRAD_ABS_FLOOR = 1e-4


def f64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, np.float64)


def check_out(got, ref, what="O"):
    got, ref = f64(got), f64(ref)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    assert err.max() <= O_MAX_ABS, f"{what}: max-abs err {err.max():.3e} > {O_MAX_ABS}"
    assert err.mean() <= O_MEAN_ABS, f"{what}: mean-abs err {err.mean():.3e} > {O_MEAN_ABS}"
    return err.max(), err.mean()


def check_lse(got, ref, what="LSE"):
    got, ref = f64(got), f64(ref)
    assert got.shape == ref.shape
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: -inf pattern differs"
    assert np.all(got[~fin] == ref[~fin]), f"{what}: masked rows must be -inf"
    if fin.any():
        err = np.abs(got[fin] - ref[fin]) / np.maximum(1.0, np.abs(ref[fin]))
        assert err.max() <= LSE_REL, f"{what}: rel err {err.max():.3e} > {LSE_REL}"
        return err.max()
    return 0.0


def check_grad(got, ref, what):
    got, ref = f64(got), f64(ref)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    scale = max(np.abs(ref).max(), GRAD_ABS_FLOOR)
    err = np.abs(got - ref).max()
    assert err <= GRAD_REL_MAX * scale, f"{what}: max err {err:.3e} > {GRAD_REL_MAX} * {scale:.3e}"
    return err / scale


def variant_pair(name, N, Hq, dev, seed=0, B=2):
    """(gpu Variant, oracle Variant) for a named combinator set."""
    import oracle

    if name == "full":
        return af.Variant(mask=af.MASK_FULL), oracle.Variant(mask=0)
    if name == "causal":
        return af.Variant(mask=af.MASK_CAUSAL), oracle.Variant(mask=1)
    if name.startswith("window"):
        W = int(name.split("_")[1])
        causal = name.endswith("_c")
        return (af.Variant(mask=af.MASK_WINDOW, window=W, causal=causal),
                oracle.Variant(mask=2, window=W, causal=causal))
    if name.startswith("alibi"):
        sl = inputs.alibi_slopes(Hq)
        mk = 0 if name == "alibi_full" else 1
        return (af.Variant(mask=mk, bias=af.BIAS_ALIBI,
                           alibi_slopes=torch.tensor(sl, dtype=torch.float32, device=dev)),
                oracle.Variant(mask=mk, bias=1, slopes=sl.astype(np.float32).astype(np.float64)))
    if name == "bigbird":
        rp, ci = inputs.bigbird_csr(-(-N // 64), seed=3003)
        return (af.Variant(mask=af.MASK_BLOCK_SPARSE, bs_block=64,
                           bs_row_ptr=torch.tensor(rp, device=dev),
                           bs_col_idx=torch.tensor(ci, device=dev)),
                oracle.Variant(mask=3, bs_block=64, bs_row_ptr=rp, bs_col_idx=ci))
    if name.startswith("addbias"):
        g = torch.Generator("cpu").manual_seed(seed + 77)
        dt = torch.bfloat16 if "bf16" in name else torch.float32
        shape = (1, Hq, N, N) if "bcast" in name else (B, Hq, N, N)
        ab = (torch.randn(*shape, generator=g) * 2).to(dt)
        mk = 1 if name.endswith("_c") else 0
        return (af.Variant(mask=mk, bias=af.BIAS_ADDITIVE, add_bias=ab.to(dev)),
                oracle.Variant(mask=mk, bias=2, add_bias=f64(ab)))
    if name.startswith("bs"):
        blk = int(name.split("_")[1])
        causal = name.endswith("_c")
        nb = -(-N // blk)
        rp, ci = inputs.bigbird_csr(nb, seed=seed + 11, n_random=2)
        return (af.Variant(mask=af.MASK_BLOCK_SPARSE, bs_block=blk, causal=causal,
                           bs_row_ptr=torch.tensor(rp, device=dev),
                           bs_col_idx=torch.tensor(ci, device=dev)),
                oracle.Variant(mask=3, bs_block=blk, causal=causal, bs_row_ptr=rp, bs_col_idx=ci))
    raise ValueError(name)
