"""GPU: the combinator front end and ROPE_AUTO call the same kernels as the direct C-ABI calls
(bit-identical outputs and gradients), and autograd through a composed variant matches the
fp64 oracle, including the additive bias's gradient (AttnFuse paper §3.1, §4.4)."""
import numpy as np
import pytest
import torch

import attention_attn_fwd_bwd_gb300 as af
from attention_attn_fwd_bwd_gb300 import combinators as C
from attention_attn_fwd_bwd_gb300 import inputs
from tests._helpers import check_grad, check_out, f64

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from attention_attn_fwd_bwd_gb300 import _build

    _build.build()
    af.load()
    assert af.device_status() == 0


def _data(B, Hq, Hkv, N, d, seed):
    dev = torch.device("cuda")
    x = inputs.prefill(B, Hq, Hkv, N, d, seed, with_dout=True)
    return [x[n].to(dev) for n in ("q", "k", "v", "dout")]


def test_composed_forward_and_autograd_match_direct_calls():
    q, k, v, do = _data(2, 8, 2, 700, 128, 61)
    attn = C.attention(C.rope(5e5, "fused"), C.scaled_dot_product(), C.causal(), C.alibi(), C.softmax())
    qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = attn(qq, kk, vv)
    out.backward(do)
    var = attn.variant(8, q.device)
    o2, l2 = af.fwd(q, k, v, rope_theta=5e5, rope_mode=af.ROPE_FUSED, variant=var)
    g2 = af.bwd(q, k, v, o2, l2, do, rope_theta=5e5, rope_mode=af.ROPE_FUSED, variant=var)
    torch.cuda.synchronize()
    assert af.device_status() == 0
    assert torch.equal(out.detach(), o2)
    for a, b in zip((qq.grad, kk.grad, vv.grad), g2):
        assert torch.equal(a, b)


def test_composed_additive_bias_gradient_vs_oracle():
    import oracle

    B, H, N, d = 1, 4, 300, 64
    q, k, v, do = _data(B, H, H, N, d, 62)
    g = torch.Generator("cpu").manual_seed(63)
    bias = torch.randn(B, H, N, N, generator=g).cuda().requires_grad_(True)
    attn = C.attention(C.rope(1e4, "prerotate"), C.sliding_window(90), C.causal(), C.additive_bias(bias))
    qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = attn(qq, kk, vv)
    out.backward(do)
    torch.cuda.synchronize()
    assert af.device_status() == 0
    ovar = oracle.Variant(mask=2, window=90, causal=True, bias=2, add_bias=f64(bias.detach()))
    o, _, dq, dk, dv, db = oracle.backward(f64(q), f64(k), f64(v), f64(do), d ** -0.5, 1e4, True,
                                           ovar, with_dbias=True)
    check_out(out.detach(), o)
    check_grad(qq.grad, dq, "dq")
    check_grad(kk.grad, dk, "dk")
    check_grad(vv.grad, dv, "dv")
    check_grad(bias.grad, db, "dbias")


@pytest.mark.parametrize("N,d", [(512, 64), (2048, 64), (512, 128)])
def test_rope_auto_is_the_resolved_mode(N, d):
    q, k, v, do = _data(2, 4, 2, N, d, 64 + N)
    var = af.Variant(mask=af.MASK_CAUSAL)
    res = []
    for mode in (af.ROPE_AUTO, af.rope_auto_mode(N, d)):
        o, l = af.fwd(q, k, v, rope_theta=1e4, rope_mode=mode, variant=var)
        res.append((o, l))
    for mode in (af.ROPE_AUTO, af.rope_auto_mode(N, d, backward=True)):
        res.append(af.bwd(q, k, v, res[0][0], res[0][1], do, rope_theta=1e4, rope_mode=mode, variant=var))
    torch.cuda.synchronize()
    assert af.device_status() == 0
    for a, b in zip(res[0], res[1]):
        assert torch.equal(a, b)
    for a, b in zip(res[2], res[3]):
        assert torch.equal(a, b)
