"""GPU parity: split-KV decode (AttnFuse paper §4.2) through the C ABI against the fp64 oracle.

Covers head dims 64/128, GQA ratios up to 16, ragged cache lengths (1, 100, 128, 129, 1000),
automatic and explicit split counts (one chunk, many chunks, more splits than tiles), rope on
q (fused) or off, and the Llama-3-70B head shape (Hq=64, Hkv=8, d=128) with a 32768-token cache
at B=1 and B=8, q at position 32767, split counts 1, 8, 32 and 128.
"""
import numpy as np
import pytest
import torch

import attention_attn_fwd_bwd_gb300 as af
from attention_attn_fwd_bwd_gb300 import inputs
from tests._helpers import check_lse, check_out, f64

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from attention_attn_fwd_bwd_gb300 import _build

    _build.build()
    af.load()
    assert af.device_status() == 0


def _run(B, Hq, Hkv, L, d, q_pos, theta, rope_mode, splits, seed, b_sel=None):
    import oracle

    x = inputs.decode(B, Hq, Hkv, L, d, seed)
    dev = torch.device("cuda")
    q, kc, vc = x["q"].to(dev), x["k_cache"].to(dev), x["v_cache"].to(dev)
    scale = d ** -0.5
    out, lse = af.decode(q, kc, vc, q_pos, scale=scale, rope_theta=theta, rope_mode=rope_mode,
                         num_splits=splits)
    torch.cuda.synchronize()
    assert af.device_status() == 0
    bs = list(range(B)) if b_sel is None else b_sel
    o_ref, l_ref = oracle.decode(f64(x["q"][bs]), f64(x["k_cache"][bs]), f64(x["v_cache"][bs]),
                                 q_pos, scale, theta, rope_q=(rope_mode == af.ROPE_FUSED))
    check_out(out[bs], o_ref)
    check_lse(lse[bs], l_ref)
    return out, lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("L", [1, 100, 128, 129, 1000])
@pytest.mark.parametrize("splits", [0, 1, 3, 8])
def test_decode_shapes(d, L, splits):
    _run(2, 8, 2, L, d, q_pos=L - 1, theta=1e4, rope_mode=af.ROPE_FUSED, splits=splits,
         seed=L * 3 + d + splits)


@pytest.mark.parametrize("gqa", [(4, 4), (16, 1), (32, 2)])
@pytest.mark.parametrize("rope_mode", [af.ROPE_NONE, af.ROPE_FUSED])
def test_decode_gqa_and_rope(gqa, rope_mode):
    Hq, Hkv = gqa
    _run(1, Hq, Hkv, 700, 128, q_pos=5000, theta=5e5, rope_mode=rope_mode, splits=0, seed=Hq)


def test_decode_split_invariance():
    """Every split count gives the same result up to fp32 reassociation."""
    x = inputs.decode(1, 8, 1, 4096, 128, 9)
    dev = torch.device("cuda")
    q, kc, vc = x["q"].to(dev), x["k_cache"].to(dev), x["v_cache"].to(dev)
    outs = [af.decode(q, kc, vc, 4095, rope_theta=5e5, num_splits=s) for s in (1, 4, 32)]
    torch.cuda.synchronize()
    for o, l in outs[1:]:
        assert (o.float() - outs[0][0].float()).abs().max().item() <= 2e-2
        assert (l - outs[0][1]).abs().max().item() <= 1e-4


@pytest.mark.parametrize("B,b_sel", [(1, None), (8, [0, 5, 7])])
@pytest.mark.parametrize("splits", [1, 8, 32, 128])
def test_decode_llama70b_shape(B, b_sel, splits):
    """Hq=64, Hkv=8, d=128, L=32768 cache, q at 32767, theta=5e5 (Llama-3-70B head shape)."""
    _run(B, 64, 8, 32768, 128, q_pos=32767, theta=5e5, rope_mode=af.ROPE_FUSED, splits=splits,
         seed=5000 + B, b_sel=b_sel)


def test_decode_equals_prefill_last_row():
    """Decode against a cache of rotated keys equals the last row of the fused prefill."""
    dev = torch.device("cuda")
    B, Hq, Hkv, N, d, theta = 1, 8, 2, 640, 128, 5e5
    x = inputs.prefill(B, Hq, Hkv, N, d, 11)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o_pre, l_pre = af.fwd(q, k, v, rope_theta=theta, rope_mode=af.ROPE_FUSED)
    k_rot = af.rope_prerotate(k, theta)  # bf16 rotated cache
    o_dec, l_dec = af.decode(q[:, :, -1].contiguous(), k_rot, v, N - 1, rope_theta=theta)
    torch.cuda.synchronize()
    assert (o_dec.float() - o_pre[:, :, -1].float()).abs().max().item() <= 2e-2
    assert (l_dec - l_pre[:, :, -1]).abs().max().item() <= 2e-2
