"""relu_attention (the paper's §3.1 normaliser, read as O_m = (1/N) sum_n max(s_mn, 0) v_n over
the visible keys) on the GPU against the fp64 oracle: every mask and bias kind, each rope mode,
GQA ratios that map to each unit shape of the persistent forward, head dims 64 and 128, ragged N."""
import math

import numpy as np
import pytest
import torch

import attention_attn_fwd_bwd_gb300 as af
from attention_attn_fwd_bwd_gb300 import inputs
from tests._helpers import check_out, f64, variant_pair

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from attention_attn_fwd_bwd_gb300 import _build

    _build.build()
    af.load()


def _relu_run(B, Hq, Hkv, N, rope_mode, vname, seed, theta=1e4, d=128):
    import oracle

    dev = torch.device("cuda")
    x = inputs.prefill(B, Hq, Hkv, N, d, seed)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    gvar, ovar = variant_pair(vname, N, Hq, dev, seed, B=B)
    gvar.norm, ovar.norm = af.NORM_RELU, oracle.NORM_RELU
    scale = 1.0 / math.sqrt(d)
    out, lse = af.fwd(q, k, v, scale=scale, rope_theta=theta, rope_mode=rope_mode, variant=gvar)
    torch.cuda.synchronize()
    assert lse is None
    assert af.device_status() == 0
    o_ref, _ = oracle.forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale, theta,
                              rope_mode != af.ROPE_NONE, ovar)
    check_out(out, o_ref)
    if N >= 64:
        assert np.abs(o_ref).max() > 1e-3  # the case is not trivially zero


@pytest.mark.parametrize("vname", ["causal", "full", "window_100_c", "alibi", "addbias_f32",
                                   "bs_64_c", "bs_128"])
def test_relu_variants(vname):
    _relu_run(2, 4, 1, 517, af.ROPE_FUSED, vname, seed=400 + len(vname))


@pytest.mark.parametrize("rope_mode", [af.ROPE_NONE, af.ROPE_FUSED, af.ROPE_PREROTATE])
@pytest.mark.parametrize("gqa", [(4, 1), (2, 2), (3, 1)])
@pytest.mark.parametrize("N", [1, 129, 700])
def test_relu_shapes(rope_mode, gqa, N):
    _relu_run(1, gqa[0], gqa[1], N, rope_mode, "causal", seed=N + gqa[0])


def test_relu_rejects_lse_and_backward():
    dev = torch.device("cuda")
    x = inputs.prefill(1, 2, 2, 64, 128, 5)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    var = af.Variant(mask=af.MASK_CAUSAL, norm=af.NORM_RELU)
    with pytest.raises(ValueError, match="no LSE"):
        af.fwd(q, k, v, variant=var, lse=torch.empty(1, 2, 64, device=dev))
    out, _ = af.fwd(q, k, v, variant=var)
    with pytest.raises(af.AttnfuseError, match="softmax normaliser only"):
        af.bwd(q, k, v, out, torch.zeros(1, 2, 64, device=dev), out, variant=var)


@pytest.mark.parametrize("gqa", [(4, 1), (2, 2)])
@pytest.mark.parametrize("rope_mode", [af.ROPE_NONE, af.ROPE_FUSED])
def test_relu_head_dim_64(gqa, rope_mode):
    """Head dim 64 runs relu_attention on the persistent pair kernel for every group size."""
    _relu_run(2, gqa[0], gqa[1], 300, rope_mode, "causal", seed=64 + gqa[0], d=64)
