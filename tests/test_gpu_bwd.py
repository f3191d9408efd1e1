"""GPU parity: the three-kernel backward (AttnFuse paper §4.4) through the C ABI vs the oracle.

Gradients are with respect to the un-rotated q and k, summed over GQA groups for dk and dv,
and must lie within 5e-2 * max|reference gradient| of the fp64 oracle's direct
differentiation. Covers rope fused / none, causal / full, GQA ratios, d 64 and 128, ragged N,
the training-step workload (B=8, Hq=32, Hkv=8, d=128, N=2048 and 4096; dq on sampled rows,
dk/dv on whole GQA groups) and run-to-run determinism (no atomics).
"""
import numpy as np
import pytest
import torch

import attention_attn_fwd_bwd_gb300 as af
from attention_attn_fwd_bwd_gb300 import inputs
from tests._helpers import check_grad, f64

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from attention_attn_fwd_bwd_gb300 import _build

    _build.build()
    af.load()
    assert af.device_status() == 0


def _gpu_fwd_bwd(x, theta, rope_mode, causal):
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    var = af.Variant(mask=af.MASK_CAUSAL if causal else af.MASK_FULL)
    out, lse = af.fwd(q, k, v, rope_theta=theta, rope_mode=rope_mode, variant=var)
    dq, dk, dv = af.bwd(q, k, v, out, lse, do, rope_theta=theta, rope_mode=rope_mode, variant=var)
    torch.cuda.synchronize()
    assert af.device_status() == 0
    return dq, dk, dv


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 63, 127, 129, 300])
@pytest.mark.parametrize("gqa", [(2, 2), (4, 2), (4, 1)])
@pytest.mark.parametrize("rope_mode", [af.ROPE_NONE, af.ROPE_FUSED])
def test_bwd_shapes_causal(d, N, gqa, rope_mode):
    import oracle

    Hq, Hkv = gqa
    x = inputs.prefill(2, Hq, Hkv, N, d, seed=N + d + Hq, with_dout=True)
    dq, dk, dv = _gpu_fwd_bwd(x, 1e4, rope_mode, True)
    _, _, rq, rk, rv = oracle.backward(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["dout"]),
                                       d ** -0.5, 1e4, rope_mode != af.ROPE_NONE,
                                       oracle.Variant(mask=1))
    check_grad(dq, rq, "dq")
    check_grad(dk, rk, "dk")
    check_grad(dv, rv, "dv")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [100, 384])
def test_bwd_full_mask(d, N):
    import oracle

    x = inputs.prefill(1, 4, 2, N, d, seed=7 + N, with_dout=True)
    dq, dk, dv = _gpu_fwd_bwd(x, 5e5, af.ROPE_FUSED, False)
    _, _, rq, rk, rv = oracle.backward(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["dout"]),
                                       d ** -0.5, 5e5, True, oracle.Variant(mask=0))
    check_grad(dq, rq, "dq")
    check_grad(dk, rk, "dk")
    check_grad(dv, rv, "dv")


def test_bwd_prerotate_mode_matches_fused():
    x = inputs.prefill(1, 4, 2, 300, 128, seed=3, with_dout=True)
    a = _gpu_fwd_bwd(x, 5e5, af.ROPE_FUSED, True)
    b = _gpu_fwd_bwd(x, 5e5, af.ROPE_PREROTATE, True)
    for u, w in zip(a, b):
        assert torch.equal(u, w)


def test_bwd_deterministic():
    x = inputs.prefill(2, 8, 2, 1000, 128, seed=4, with_dout=True)
    a = _gpu_fwd_bwd(x, 5e5, af.ROPE_FUSED, True)
    b = _gpu_fwd_bwd(x, 5e5, af.ROPE_FUSED, True)
    for u, w in zip(a, b):
        assert torch.equal(u, w)


@pytest.mark.parametrize("N", [2048, 4096])
def test_bwd_training_workload(N):
    """B=8, Hq=32, Hkv=8, d=128, theta=5e5, causal, fused RoPE; dq on sampled rows, dk/dv on
    two whole GQA groups (every row of those groups' key/value heads)."""
    import oracle

    B, Hq, Hkv, d = 8, 32, 8, 128
    x = inputs.prefill(B, Hq, Hkv, N, d, seed=4000 + N, with_dout=True)
    dq, dk, dv = _gpu_fwd_bwd(x, 5e5, af.ROPE_FUSED, True)
    q64, k64, v64, do64 = (f64(x[n]) for n in ("q", "k", "v", "dout"))
    var = oracle.Variant(mask=1)
    rows = inputs.sample_rows(B, Hq, N, 48, seed=N, always=[(0, 0, 0), (7, 31, N - 1), (3, 9, 128)])
    rdq = oracle.backward_dq_rows(q64, k64, v64, do64, d ** -0.5, 5e5, True, var, rows)
    dqc = dq.cpu()
    check_grad(torch.stack([dqc[b, h, m] for b, h, m in rows]), rdq, "dq rows")
    groups = [(0, 0), (7, 5)] if N == 2048 else [(5, 3)]
    _, _, _, rk, rv = oracle.backward(q64, k64, v64, do64, d ** -0.5, 5e5, True, var, groups=groups)
    dkc, dvc = dk.cpu(), dv.cpu()
    for b, h in groups:
        check_grad(dkc[b, h], rk[b, h], f"dk[{b},{h}]")
        check_grad(dvc[b, h], rv[b, h], f"dv[{b},{h}]")
