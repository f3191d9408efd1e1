"""GPU parity: the forward kernel (through the C ABI) against the fp64 oracle.

Covers the pages' forward (AttnFuse paper §4.1 fused RoPE, §2 softmax, §3.1 combinators,
§4.3 block skipping): rope modes NONE / FUSED / PREROTATE, masks FULL / CAUSAL / WINDOW /
BLOCK_SPARSE, ALiBi and additive bias, GQA ratios, head dims 64 and 128, ragged N (1, 63, 127,
129, ...), the tiny and full-size workloads (full size on sampled rows), bit-exact tile-visit
sets, and bitwise equality of FUSED and PREROTATE (same rotation code, same tables).
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import attention_attn_fwd_bwd_gb300 as af
from attention_attn_fwd_bwd_gb300 import inputs
from tests._helpers import variant_pair as _variants, check_lse, check_out, f64

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from attention_attn_fwd_bwd_gb300 import _build

    _build.build()
    af.load()
    assert af.device_status() == 0


def _run(B, Hq, Hkv, N, d, rope_mode, vname, seed, theta=10000.0, rows=None, visits=False):
    import oracle

    dev = torch.device("cuda")
    x = inputs.prefill(B, Hq, Hkv, N, d, seed)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    gvar, ovar = _variants(vname, N, Hq, dev, seed)
    TQ = -(-N // 128)
    if visits:
        gvar.tile_visits = torch.zeros((B, Hq, TQ, TQ), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(d)
    out, lse = af.fwd(q, k, v, scale=scale, rope_theta=theta, rope_mode=rope_mode, variant=gvar)
    torch.cuda.synchronize()
    assert af.device_status() == 0
    rope_on = rope_mode != af.ROPE_NONE
    q64, k64, v64 = f64(x["q"]), f64(x["k"]), f64(x["v"])
    if rows is None:
        o_ref, l_ref = oracle.forward(q64, k64, v64, scale, theta, rope_on, ovar)
        check_out(out, o_ref)
        check_lse(lse, l_ref)
    else:
        o_ref, l_ref = oracle.forward_rows(q64, k64, v64, scale, theta, rope_on, ovar, rows)
        oc, lc = out.cpu(), lse.cpu()
        got_o = torch.stack([oc[b, h, m] for b, h, m in rows])
        got_l = torch.stack([lc[b, h, m] for b, h, m in rows])
        check_out(got_o, o_ref)
        check_lse(got_l, l_ref)
    if visits:
        ref_vis = oracle.tile_visits(N, 128, 128, ovar)
        got = gvar.tile_visits.cpu().numpy()
        for b in range(B):
            for h in range(Hq):
                assert np.array_equal(got[b, h], ref_vis), f"tile visits differ at b={b} h={h}"
    return out, lse


def test_tiny_config():
    """Tiny RoPE+causal forward: B=1, H=2, N=128, d=64, theta=1e4, fused, O and LSE."""
    _run(1, 2, 2, 128, 64, af.ROPE_FUSED, "causal", seed=1000, visits=True)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 63, 127, 129, 300])
@pytest.mark.parametrize("gqa", [(2, 2), (4, 1), (4, 2), (3, 1)])
@pytest.mark.parametrize("rope_mode", [af.ROPE_NONE, af.ROPE_FUSED, af.ROPE_PREROTATE])
def test_shapes_causal(d, N, gqa, rope_mode):
    Hq, Hkv = gqa
    _run(2, Hq, Hkv, N, d, rope_mode, "causal", seed=N * 7 + d + Hq)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 200, 384])
def test_full_mask(d, N):
    _run(1, 4, 2, N, d, af.ROPE_FUSED, "full", seed=5 + N)


@pytest.mark.parametrize("vname", ["window_100_c", "window_128_c", "window_70",
                                   "alibi", "addbias_f32", "addbias_bf16_bcast",
                                   "bs_64", "bs_64_c", "bs_128", "bs_128_c"])
@pytest.mark.parametrize("d", [64, 128])
def test_variants(vname, d):
    _run(2, 4, 2, 517, d, af.ROPE_FUSED, vname, seed=31 + d, visits=True)


@pytest.mark.parametrize("vname", ["window_300_c", "alibi", "bs_64"])
def test_variants_mha_tile_pairs(vname):
    """Hq == Hkv: the kernel pairs consecutive q tiles of one head."""
    _run(1, 3, 3, 700, 64, af.ROPE_FUSED, vname, seed=9, visits=True)


@pytest.mark.parametrize("d", [64, 128])
def test_window_one_is_identity(d):
    """W = 1: every row sees only its own key, so P = 1, O_m = v_m exactly and LSE_m = s_mm.

    A single score carries the rounding of the rotated operands undamped, so LSE is checked
    against the rigorous bound for rounding q' and k' to fp16 (unit roundoff u = 2^-11):
    |s_hat - s| <= scale * sum_c |q'_c k'_c| * (2u + u^2), plus fp32 accumulation slack.
    """
    import oracle

    dev = torch.device("cuda")
    B, Hq, Hkv, N = 2, 4, 2, 517
    x = inputs.prefill(B, Hq, Hkv, N, d, 41)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    scale = d ** -0.5
    out, lse = af.fwd(q, k, v, scale=scale, rope_theta=1e4,
                      variant=af.Variant(mask=af.MASK_WINDOW, window=1, causal=True))
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), x["v"].repeat_interleave(Hq // Hkv, dim=1))
    pos = np.arange(N, dtype=np.float64)
    qr = np.stack([oracle.rope(f64(x["q"][b, h]), pos, 1e4) for b in range(B) for h in range(Hq)])
    kr = np.stack([oracle.rope(f64(x["k"][b, h // 2]), pos, 1e4) for b in range(B) for h in range(Hq)])
    s_exact = scale * np.einsum("rnc,rnc->rn", qr, kr)
    u = 2.0 ** -11
    bound = scale * np.einsum("rnc,rnc->rn", np.abs(qr), np.abs(kr)) * (2 * u + u * u) * 1.01 + 1e-6
    err = np.abs(f64(lse).reshape(B * Hq, N) - s_exact)
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound):.3f}"


def test_window_ge_n_equals_causal():
    dev = torch.device("cuda")
    x = inputs.prefill(1, 4, 2, 333, 128, 4)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o1, l1 = af.fwd(q, k, v, rope_theta=1e4, variant=af.Variant(mask=af.MASK_CAUSAL))
    o2, l2 = af.fwd(q, k, v, rope_theta=1e4,
                    variant=af.Variant(mask=af.MASK_WINDOW, window=333, causal=True))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d", [64, 128])
def test_fused_equals_prerotate_bitwise(d):
    """Same (cos, sin) table and rotation code: the two modes feed identical bf16 Q', K'."""
    dev = torch.device("cuda")
    x = inputs.prefill(2, 8, 2, 640, d, 5)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o1, l1 = af.fwd(q, k, v, rope_theta=5e5, rope_mode=af.ROPE_FUSED)
    o2, l2 = af.fwd(q, k, v, rope_theta=5e5, rope_mode=af.ROPE_PREROTATE)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_deterministic():
    dev = torch.device("cuda")
    x = inputs.prefill(2, 8, 2, 1000, 128, 6)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o1, l1 = af.fwd(q, k, v, rope_theta=5e5)
    o2, l2 = af.fwd(q, k, v, rope_theta=5e5)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_prerotate_kernel_vs_oracle_rope():
    import oracle

    dev = torch.device("cuda")
    x = inputs.prefill(2, 3, 3, 4100, 128, 7)["q"]
    xr = af.rope_prerotate(x.to(dev), 5e5)
    torch.cuda.synchronize()
    pos = np.tile(np.arange(4100, dtype=np.float64), 6)
    ref = oracle.rope(f64(x).reshape(-1, 128), pos, 5e5).reshape(x.shape)
    err = np.abs(f64(xr) - ref)
    # one bf16 rounding of the rotated value (|x| <~ 5 => ulp/2 <~ 2^-7) plus fp32 math
    assert err.max() <= 2.0 ** -6 and err.mean() < 2e-3


def test_strided_inputs():
    """Non-contiguous (B, N, H, d) layouts via strides."""
    import oracle

    dev = torch.device("cuda")
    B, Hq, Hkv, N, d = 2, 4, 2, 250, 64
    x = inputs.prefill(B, Hq, Hkv, N, d, 8)
    q = x["q"].transpose(1, 2).contiguous().to(dev).transpose(1, 2)
    k = x["k"].transpose(1, 2).contiguous().to(dev).transpose(1, 2)
    v = x["v"].transpose(1, 2).contiguous().to(dev).transpose(1, 2)
    out = torch.empty((B, N, Hq, d), dtype=torch.bfloat16, device=dev).transpose(1, 2)
    af.fwd(q, k, v, rope_theta=1e4, out=out)
    torch.cuda.synchronize()
    o_ref, _ = oracle.forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), d ** -0.5, 1e4, True,
                              oracle.Variant(mask=1))
    check_out(out, o_ref)


@pytest.mark.parametrize("rope_mode", [af.ROPE_FUSED, af.ROPE_PREROTATE])
def test_full_size_llama8b_sampled(rope_mode):
    """B=4, Hq=32, Hkv=8, N=4096, d=128, theta=5e5, causal: every row of one whole (b, h)
    slice, plus sampled rows of the others, vs the oracle."""
    rows = inputs.sample_rows(4, 32, 4096, 40, seed=2,
                              always=[(0, 0, 0), (3, 31, 4095), (1, 5, 4095), (2, 17, 128),
                                      (3, 30, 127), (0, 1, 2047)])
    rows = np.concatenate([rows, _slice_rows(1, 22, 4096)])
    _run(4, 32, 8, 4096, 128, rope_mode, "causal", seed=2000, theta=5e5, rows=rows)


def _slice_rows(b, h, N):
    """(b, h, m) for every query row m of one (b, h) slice."""
    m = np.arange(N, dtype=np.int64)
    return np.stack([np.full_like(m, b), np.full_like(m, h), m], axis=1)


@pytest.mark.parametrize("vname", ["window_1024_c", "alibi", "bigbird"])
def test_full_size_mask_variants_sampled(vname):
    """B=2, H=16, N=4096, d=64, theta=1e4, fused: window 1024 + causal, ALiBi, BigBird; one
    whole (b, h) slice plus sampled rows vs the oracle, tile-visit sets bit-exact."""
    import oracle

    dev = torch.device("cuda")
    B, H, N, d = 2, 16, 4096, 64
    seed = 3000 + {"window_1024_c": 1, "alibi": 2, "bigbird": 3}[vname]
    if vname == "bigbird":
        rp, ci = inputs.bigbird_csr(N // 64, seed=3003)
        gvar = af.Variant(mask=af.MASK_BLOCK_SPARSE, bs_block=64,
                          bs_row_ptr=torch.tensor(rp, device=dev),
                          bs_col_idx=torch.tensor(ci, device=dev))
        ovar = oracle.Variant(mask=3, bs_block=64, bs_row_ptr=rp, bs_col_idx=ci)
    else:
        gvar, ovar = _variants(vname, N, H, dev)
    TQ = N // 128
    gvar.tile_visits = torch.zeros((B, H, TQ, TQ), dtype=torch.uint8, device=dev)
    x = inputs.prefill(B, H, H, N, d, seed)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    out, lse = af.fwd(q, k, v, scale=0.125, rope_theta=1e4, variant=gvar)
    torch.cuda.synchronize()
    assert af.device_status() == 0
    rows = inputs.sample_rows(B, H, N, 40, seed=seed, always=[(0, 0, 0), (1, 15, 4095),
                                                              (0, 3, 1024), (1, 8, 63)])
    rows = np.concatenate([rows, _slice_rows(1, 9, N)])
    o_ref, l_ref = oracle.forward_rows(f64(x["q"]), f64(x["k"]), f64(x["v"]), 0.125, 1e4, True,
                                       ovar, rows)
    oc, lc = out.cpu(), lse.cpu()
    check_out(torch.stack([oc[b, h, m] for b, h, m in rows]), o_ref)
    check_lse(torch.stack([lc[b, h, m] for b, h, m in rows]), l_ref)
    ref_vis = oracle.tile_visits(N, 128, 128, ovar)
    got = gvar.tile_visits.cpu().numpy()
    assert all(np.array_equal(got[b, h], ref_vis) for b in range(B) for h in range(H))


def test_timeout_path_reports_status():
    """A wait that can never complete gives up after its limit and sets the status word."""
    af.load().attnfuse_debug_wait_timeout(2_000_000, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert af.device_status(clear=True) == 5
    assert af.device_status(clear=True) == 0
    # the context is still usable
    test_tiny_config()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("rope_mode", [af.ROPE_FUSED, af.ROPE_PREROTATE])
@pytest.mark.parametrize("which", ["q", "k"])
def test_fp16_range_is_reported(d, rope_mode, which):
    """The rotating modes round Q' and K' to fp16: an element beyond 65504 saturates, and the
    call reports it through the device status word (ATTNFUSE_ERR_FP16_RANGE = 6), which a read
    clears. Position 0 rotates by angle 0, so a value of 70000 there reaches the rounding as it
    is. Without RoPE the bf16 operands are used as they are and nothing is reported."""
    dev = torch.device("cuda")
    N = 300
    x = inputs.prefill(1, 4, 2, N, d, seed=33)
    t = x[which].clone()
    t[0, 1, 0, 3] = 70000.0
    x[which] = t
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    assert af.device_status() == 0
    af.fwd(q, k, v, rope_theta=1e4, rope_mode=rope_mode)
    assert af.device_status() == 6
    assert af.device_status() == 0
    af.fwd(q, k, v, rope_theta=1e4, rope_mode=af.ROPE_NONE)
    assert af.device_status() == 0


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("rope_mode", [af.ROPE_NONE, af.ROPE_FUSED])
@pytest.mark.parametrize("N", [129, 256])
def test_many_units_with_an_empty_slot(d, rope_mode, N):
    """With one head per work unit (Hq == Hkv) and two query tiles, a unit's second slot has no
    rows; many such units per cluster (B * H >> the number of clusters) must not let that
    slot's bookkeeping run a unit ahead of its softmax."""
    _run(40, 4, 4, N, d, rope_mode, "causal", seed=N + d)
