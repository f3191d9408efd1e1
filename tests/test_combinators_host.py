"""The combinator front end (AttnFuse paper §3.1) and the ROPE_AUTO rule, without a GPU: how
compositions map onto one attnfuse_variant, which compositions are rejected, and which mode
the measured crossover picks."""
import math

import pytest
import torch

import attention_attn_fwd_bwd_gb300 as af
from attention_attn_fwd_bwd_gb300 import combinators as C


def test_mask_and_bias_mapping():
    cpu = torch.device("cpu")
    v = C.attention(C.causal(), C.softmax()).variant(4, cpu)
    assert (v.mask, v.bias) == (af.MASK_CAUSAL, af.BIAS_NONE)
    v = C.attention(C.sliding_window(100), C.causal()).variant(4, cpu)
    assert (v.mask, v.window, bool(v.causal)) == (af.MASK_WINDOW, 100, True)
    v = C.attention(C.sliding_window(7)).variant(4, cpu)
    assert (v.mask, v.window, bool(v.causal)) == (af.MASK_WINDOW, 7, False)
    rp, ci = torch.tensor([0, 1], dtype=torch.int32), torch.tensor([0], dtype=torch.int32)
    v = C.attention(C.block_sparse(rp, ci, 128), C.causal()).variant(4, cpu)
    assert (v.mask, v.bs_block, bool(v.causal)) == (af.MASK_BLOCK_SPARSE, 128, True)
    v = C.attention(C.full(), C.alibi()).variant(8, cpu)
    assert (v.mask, v.bias) == (af.MASK_FULL, af.BIAS_ALIBI)
    # default slopes: 2^(-8 (h + 1) / H), h 0-based (Press et al.)
    assert torch.allclose(v.alibi_slopes, torch.tensor([2.0 ** (-(h + 1)) for h in range(8)]))
    ab = torch.zeros(1, 4, 16, 16)
    a = C.attention(C.causal(), C.additive_bias(ab))
    v = a.variant(4, cpu)
    assert (v.mask, v.bias) == (af.MASK_CAUSAL, af.BIAS_ADDITIVE) and v.add_bias is ab
    cs = v.c_struct()
    assert cs.bias == af.BIAS_ADDITIVE and list(cs.add_bias_strides) == [0, 256, 16, 1]


def test_scale_and_rope_arguments():
    a = C.attention(C.rope(5e5, "fused"), C.scaled_dot_product(0.25), C.causal())
    assert (a.rope_mode, a.rope_theta, a.scale) == (af.ROPE_FUSED, 5e5, 0.25)
    a = C.attention(C.rope(), C.causal())
    assert a.rope_mode == af.ROPE_AUTO and a.scale is None
    a = C.attention(C.causal())
    assert a.rope_mode == af.ROPE_NONE
    with pytest.raises(ValueError):
        C.rope(1e4, "sideways")


@pytest.mark.parametrize("combo", [
    (C.full, C.causal),
    (lambda: C.sliding_window(4), lambda: C.block_sparse(None, None)),
    (C.alibi, lambda: C.additive_bias(torch.zeros(1))),
    (C.causal, C.causal),
])
def test_rejected_compositions(combo):
    with pytest.raises(ValueError):
        C.attention(*(f() for f in combo))


def test_relu_attention_maps_to_the_relu_normaliser():
    att = C.attention(C.rope(5e5), C.causal(), C.relu_attention())
    v = att.variant(4, torch.device("cpu"))
    assert v.norm == af.NORM_RELU and v.mask == af.MASK_CAUSAL
    assert C.attention(C.causal()).variant(4, torch.device("cpu")).norm == af.NORM_SOFTMAX
    with pytest.raises(ValueError, match="one normaliser"):
        C.attention(C.softmax(), C.relu_attention())


def test_rope_auto_rule():
    """The measured crossover (GB300, B*N = 16384): fusion wins for head dim 64 below
    N ~ 1.85k (forward) and ~ 260 (backward), for the head-dim-128 forward below N ~ 15k;
    pre-rotation everywhere else."""
    from attention_attn_fwd_bwd_gb300 import _build

    _build.build()
    af.load()
    for N in (1, 128, 1024, 1849):
        assert af.rope_auto_mode(N, 64) == af.ROPE_FUSED
    for N in (1850, 4096, 65536):
        assert af.rope_auto_mode(N, 64) == af.ROPE_PREROTATE
    for N in (1, 128, 257):
        assert af.rope_auto_mode(N, 64, backward=True) == af.ROPE_FUSED
    for N in (258, 1024, 4096):
        assert af.rope_auto_mode(N, 64, backward=True) == af.ROPE_PREROTATE
    for N in (1, 256, 4096, 14899):
        assert af.rope_auto_mode(N, 128) == af.ROPE_FUSED
    for N in (14900, 16384, 65536):
        assert af.rope_auto_mode(N, 128) == af.ROPE_PREROTATE
    for N in (1, 256, 4096):
        assert af.rope_auto_mode(N, 128, backward=True) == af.ROPE_PREROTATE
    # workspace sizes follow the resolved mode
    for N, d in ((512, 64), (4096, 64), (512, 128)):
        m = af.rope_auto_mode(N, d)
        assert af.fwd_workspace_size(2, 4, 2, N, d, af.ROPE_AUTO) == af.fwd_workspace_size(2, 4, 2, N, d, m)
        mb = af.rope_auto_mode(N, d, backward=True)
        assert af.bwd_workspace_size(2, 4, 2, N, d, af.ROPE_AUTO) == af.bwd_workspace_size(2, 4, 2, N, d, mb)
    with pytest.raises(af.AttnfuseError):
        af.rope_auto_mode(100, 96)
