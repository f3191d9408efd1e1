"""GPU parity at the size limits: a 32k-token causal forward with fused RoPE (sampled rows),
block-sparse layouts at the 65,536-token limit of the CSR tile tables, 16-way GQA, and a
long-sequence backward (dq on sampled rows, dk/dv on one whole head). AttnFuse paper §4.1-§4.4."""
import math

import numpy as np
import pytest
import torch

import attention_attn_fwd_bwd_gb300 as af
from attention_attn_fwd_bwd_gb300 import inputs
from tests._helpers import check_grad, check_lse, check_out, f64

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from attention_attn_fwd_bwd_gb300 import _build

    _build.build()
    af.load()
    assert af.device_status() == 0


def _fwd_sampled(B, Hq, Hkv, N, d, seed, gvar, ovar, rope_mode=af.ROPE_FUSED, theta=5e5, count=32):
    import oracle

    dev = torch.device("cuda")
    x = inputs.prefill(B, Hq, Hkv, N, d, seed)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    out, lse = af.fwd(q, k, v, rope_theta=theta, rope_mode=rope_mode, variant=gvar)
    torch.cuda.synchronize()
    assert af.device_status() == 0
    rows = inputs.sample_rows(B, Hq, N, count, seed=seed,
                              always=[(0, 0, 0), (B - 1, Hq - 1, N - 1), (0, Hq // 2, N // 2)])
    o, l = oracle.forward_rows(f64(x["q"]), f64(x["k"]), f64(x["v"]), d ** -0.5, theta,
                               rope_mode != af.ROPE_NONE, ovar, rows)
    oc, lc = out.cpu(), lse.cpu()
    check_out(torch.stack([oc[b, h, m] for b, h, m in rows]), o)
    check_lse(torch.stack([lc[b, h, m] for b, h, m in rows]), l)


@pytest.mark.parametrize("d", [64, 128])
def test_fwd_32k_tokens_causal(d):
    """B=1, N=32768: positions up to 32767 through the in-kernel (cos, sin) recurrences."""
    import oracle

    _fwd_sampled(1, 4, 2, 32768, d, 9001 + d, af.Variant(mask=af.MASK_CAUSAL), oracle.Variant(mask=1))


def test_fwd_gqa16():
    import oracle

    _fwd_sampled(2, 32, 2, 2048, 128, 9003, af.Variant(mask=af.MASK_CAUSAL), oracle.Variant(mask=1))


@pytest.mark.parametrize("blk", [64, 128])
def test_block_sparse_at_layout_limit(blk):
    """N = 65536 (the CSR tile tables' limit): a BigBird layout over 1024 / 512 block rows."""
    import oracle

    N = 65536
    rp, ci = inputs.bigbird_csr(N // blk, seed=9004 + blk, n_random=2)
    dev = torch.device("cuda")
    gvar = af.Variant(mask=af.MASK_BLOCK_SPARSE, bs_block=blk,
                      bs_row_ptr=torch.tensor(rp, device=dev), bs_col_idx=torch.tensor(ci, device=dev))
    ovar = oracle.Variant(mask=3, bs_block=blk, bs_row_ptr=rp, bs_col_idx=ci)
    _fwd_sampled(1, 2, 2, N, 64, 9005 + blk, gvar, ovar, theta=1e4, count=24)


def test_bwd_long_sequence():
    """B=1, Hq=4, Hkv=1, N=8192, d=128, causal, fused RoPE: dq on sampled rows, dk/dv of the
    single key/value head in full."""
    import oracle

    B, Hq, Hkv, N, d = 1, 4, 1, 8192, 128
    dev = torch.device("cuda")
    x = inputs.prefill(B, Hq, Hkv, N, d, 9006, with_dout=True)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    var = af.Variant(mask=af.MASK_CAUSAL)
    out, lse = af.fwd(q, k, v, rope_theta=5e5, variant=var)
    dq, dk, dv = af.bwd(q, k, v, out, lse, do, rope_theta=5e5, variant=var)
    torch.cuda.synchronize()
    assert af.device_status() == 0
    q64, k64, v64, do64 = (f64(x[n]) for n in ("q", "k", "v", "dout"))
    ovar = oracle.Variant(mask=1)
    rows = inputs.sample_rows(B, Hq, N, 24, seed=9007, always=[(0, 0, 0), (0, 3, N - 1), (0, 1, 4096)])
    rdq = oracle.backward_dq_rows(q64, k64, v64, do64, d ** -0.5, 5e5, True, ovar, rows)
    dqc = dq.cpu()
    check_grad(torch.stack([dqc[b, h, m] for b, h, m in rows]), rdq, "dq rows")
    _, _, _, rk, rv = oracle.backward(q64, k64, v64, do64, d ** -0.5, 5e5, True, ovar, groups=[(0, 0)])
    check_grad(dk.cpu()[0, 0], rk[0, 0], "dk")
    check_grad(dv.cpu()[0, 0], rv[0, 0], "dv")
