"""GPU: the forward on host buffers (copy-in, forward and copy-out pipelined over batch chunks)
gives exactly the device forward's results, and matches the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import attention_attn_fwd_bwd_gb300 as af
from attention_attn_fwd_bwd_gb300 import inputs
from tests._helpers import check_lse, check_out, f64, variant_pair

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from attention_attn_fwd_bwd_gb300 import _build

    _build.build()
    af.load()
    assert af.device_status() == 0


def _pinned(x):
    return x.contiguous().pin_memory()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("vname", ["causal", "window_100_c", "addbias_f32", "addbias_bcast", "alibi", "bs_64"])
@pytest.mark.parametrize("chunk_b", [1, 2])
def test_host_forward_equals_device_forward(d, vname, chunk_b):
    dev = torch.device("cuda")
    B, Hq, Hkv, N = 3, 4, 2, 300
    x = inputs.prefill(B, Hq, Hkv, N, d, seed=70 + d + chunk_b)
    gvar, _ = variant_pair(vname, N, Hq, dev, seed=5, B=B)
    TQ = -(-N // 128)
    if not vname.startswith("addbias"):
        gvar.tile_visits = torch.zeros((B, Hq, TQ, TQ), dtype=torch.uint8, device=dev)
    q, k, v = (_pinned(x[n]) for n in ("q", "k", "v"))
    out_h, lse_h = af.fwd_host(q, k, v, rope_theta=1e4, rope_mode=af.ROPE_FUSED, variant=gvar,
                               chunk_b=chunk_b)
    vis_h = gvar.tile_visits.clone() if gvar.tile_visits is not None else None
    if vis_h is not None:
        gvar.tile_visits.zero_()
    out_d, lse_d = af.fwd(x["q"].to(dev), x["k"].to(dev), x["v"].to(dev), rope_theta=1e4,
                          rope_mode=af.ROPE_FUSED, variant=gvar)
    torch.cuda.synchronize()
    assert af.device_status() == 0
    assert torch.equal(out_h, out_d.cpu())
    assert torch.equal(lse_h, lse_d.cpu())
    if vis_h is not None:
        assert torch.equal(vis_h, gvar.tile_visits)


@pytest.mark.parametrize("rope_mode", [af.ROPE_NONE, af.ROPE_FUSED, af.ROPE_PREROTATE])
def test_host_forward_vs_oracle(rope_mode):
    import oracle

    B, Hq, Hkv, N, d = 2, 8, 2, 517, 128
    x = inputs.prefill(B, Hq, Hkv, N, d, seed=91)
    q, k, v = (_pinned(x[n]) for n in ("q", "k", "v"))
    out, lse = af.fwd_host(q, k, v, rope_theta=5e5, rope_mode=rope_mode, chunk_b=1)
    assert af.device_status() == 0
    o_ref, l_ref = oracle.forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), d ** -0.5, 5e5,
                                  rope_mode != af.ROPE_NONE, oracle.Variant(mask=1))
    check_out(out, o_ref)
    check_lse(lse, l_ref)


def test_host_forward_pageable_and_relu():
    """Pageable (not pinned) buffers work too, and relu_attention has no LSE."""
    import oracle

    dev = torch.device("cuda")
    B, Hq, Hkv, N, d = 2, 4, 1, 200, 128
    x = inputs.prefill(B, Hq, Hkv, N, d, seed=92)
    gvar, ovar = variant_pair("causal", N, Hq, dev)
    gvar.norm, ovar.norm = af.NORM_RELU, oracle.NORM_RELU
    out, lse = af.fwd_host(x["q"], x["k"], x["v"], rope_theta=1e4, variant=gvar, chunk_b=1)
    assert lse is None
    o_ref, _ = oracle.forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), d ** -0.5, 1e4, True, ovar)
    check_out(out, o_ref)


def test_host_forward_argument_errors():
    x = inputs.prefill(2, 2, 2, 64, 64, seed=1)
    with pytest.raises(af.AttnfuseError, match="chunk_b"):
        af.fwd_host(x["q"], x["k"], x["v"], chunk_b=3)
    with pytest.raises(ValueError, match="CPU"):
        af.fwd_host(x["q"].cuda(), x["k"], x["v"])
    with pytest.raises(af.AttnfuseError, match="REUSE_TABLE"):
        af.fwd_host(x["q"], x["k"], x["v"], rope_mode=af.ROPE_FUSED | af.ROPE_REUSE_TABLE)
