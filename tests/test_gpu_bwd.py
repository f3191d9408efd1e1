"""GPU parity: the three-kernel backward (AttnFuse paper §4.4) through the C ABI vs the oracle.

Gradients are with respect to the un-rotated q and k, summed over GQA groups for dk and dv,
and must lie within 5e-2 * max|reference gradient| of the fp64 oracle's direct
differentiation; dBias (additive bias) is held to the same bar element by element. Covers
rope fused / none / pre-rotated, every mask and bias combinator of the forward (paper §3.1,
§4.3: the backward visits only active tiles), GQA ratios, d 64 and 128, ragged N, the
training-step workload (B=8, Hq=32, Hkv=8, d=128, N=2048 and 4096; dq on sampled rows, dk/dv
on whole GQA groups), the mask-variant workload (B=2, H=16, N=4096, d=64) and run-to-run
determinism (no atomics).
"""
import numpy as np
import pytest
import torch

import attention_attn_fwd_bwd_gb300 as af
from attention_attn_fwd_bwd_gb300 import inputs
from tests._helpers import check_grad, f64, variant_pair

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
    """B=8, Hq=32, Hkv=8, d=128, theta=5e5, causal, fused RoPE; dq on one whole (b, h) slice
    plus sampled rows, dk/dv on whole GQA groups (every row of those groups' key/value heads)."""
    import oracle

    B, Hq, Hkv, d = 8, 32, 8, 128
    x = inputs.prefill(B, Hq, Hkv, N, d, seed=4000 + N, with_dout=True)
    dq, dk, dv = _gpu_fwd_bwd(x, 5e5, af.ROPE_FUSED, True)
    q64, k64, v64, do64 = (f64(x[n]) for n in ("q", "k", "v", "dout"))
    var = oracle.Variant(mask=1)
    rows = inputs.sample_rows(B, Hq, N, 48, seed=N, always=[(0, 0, 0), (7, 31, N - 1), (3, 9, 128)])
    m = np.arange(N, dtype=np.int64)
    rows = np.concatenate([rows, np.stack([np.full_like(m, 6), np.full_like(m, 13), m], axis=1)])
    rdq = oracle.backward_dq_rows(q64, k64, v64, do64, d ** -0.5, 5e5, True, var, rows)
    dqc = dq.cpu()
    check_grad(torch.stack([dqc[b, h, m] for b, h, m in rows]), rdq, "dq rows")
    groups = [(0, 0), (7, 5)] if N == 2048 else [(5, 3)]
    _, _, _, rk, rv = oracle.backward(q64, k64, v64, do64, d ** -0.5, 5e5, True, var, groups=groups)
    dkc, dvc = dk.cpu(), dv.cpu()
    for b, h in groups:
        check_grad(dkc[b, h], rk[b, h], f"dk[{b},{h}]")
        check_grad(dvc[b, h], rv[b, h], f"dv[{b},{h}]")


def _run_variant_bwd(B, Hq, Hkv, N, d, rope_mode, vname, seed, theta=1e4):
    import oracle

    dev = torch.device("cuda")
    x = inputs.prefill(B, Hq, Hkv, N, d, seed, with_dout=True)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    gvar, ovar = variant_pair(vname, N, Hq, dev, seed, B=B)
    with_db = vname.startswith("addbias")
    scale = d ** -0.5
    out, lse = af.fwd(q, k, v, scale=scale, rope_theta=theta, rope_mode=rope_mode, variant=gvar)
    if with_db:
        gvar.dbias = torch.full((B, Hq, N, N), float("nan"), dtype=torch.float32, device=dev)
    dq, dk, dv = af.bwd(q, k, v, out, lse, do, scale=scale, rope_theta=theta,
                        rope_mode=rope_mode, variant=gvar)
    torch.cuda.synchronize()
    assert af.device_status() == 0
    ref = oracle.backward(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["dout"]), scale, theta,
                          rope_mode != af.ROPE_NONE, ovar, with_dbias=with_db)
    check_grad(dq, ref[2], "dq")
    check_grad(dk, ref[3], "dk")
    check_grad(dv, ref[4], "dv")
    if with_db:
        check_grad(gvar.dbias, ref[5], "dbias")


BWD_VARIANTS = ["window_100_c", "window_70", "alibi", "alibi_full", "addbias_f32",
                "addbias_bf16_bcast_c", "bs_64", "bs_64_c", "bs_128", "bs_128_c"]


@pytest.mark.parametrize("vname", BWD_VARIANTS)
@pytest.mark.parametrize("d", [64, 128])
def test_bwd_variants(vname, d):
    _run_variant_bwd(2, 4, 2, 517, d, af.ROPE_FUSED, vname, seed=41 + d)


@pytest.mark.parametrize("vname", ["window_70", "alibi", "addbias_f32_c", "bs_64_c"])
@pytest.mark.parametrize("rope_mode", [af.ROPE_NONE, af.ROPE_PREROTATE])
def test_bwd_variants_rope_modes(vname, rope_mode):
    _run_variant_bwd(1, 4, 4, 300, 128, rope_mode, vname, seed=43)


@pytest.mark.parametrize("vname", ["window_1_c", "window_129", "window_600_c", "bs_64"])
@pytest.mark.parametrize("N", [1, 64, 129])
def test_bwd_variant_edges(vname, N):
    """W = 1 (one visible key per row: dS = 0), windows wider than N, tiny and ragged N."""
    _run_variant_bwd(1, 2, 1, N, 64, af.ROPE_FUSED, vname, seed=44 + N)


def test_bwd_variant_prerotate_matches_fused():
    dev = torch.device("cuda")
    x = inputs.prefill(1, 4, 2, 300, 128, seed=45, with_dout=True)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    res = []
    for mode in (af.ROPE_FUSED, af.ROPE_PREROTATE):
        gvar, _ = variant_pair("bs_64_c", 300, 4, dev, 45)
        out, lse = af.fwd(q, k, v, rope_theta=5e5, rope_mode=mode, variant=gvar)
        res.append(af.bwd(q, k, v, out, lse, do, rope_theta=5e5, rope_mode=mode, variant=gvar))
    torch.cuda.synchronize()
    for u, w in zip(*res):
        assert torch.equal(u, w)


@pytest.mark.parametrize("vname", ["window_1024_c", "alibi", "bigbird"])
def test_bwd_mask_variant_workload(vname):
    """B=2, H=16, N=4096, d=64, theta=1e4, fused: window 1024 + causal, ALiBi + causal,
    BigBird 64-blocks (non-causal). dq on sampled rows, dk/dv on one whole head."""
    import oracle

    dev = torch.device("cuda")
    B, H, N, d = 2, 16, 4096, 64
    seed = 3100 + {"window_1024_c": 1, "alibi": 2, "bigbird": 3}[vname]
    x = inputs.prefill(B, H, H, N, d, seed, with_dout=True)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    gvar, ovar = variant_pair(vname, N, H, dev, seed)
    out, lse = af.fwd(q, k, v, rope_theta=1e4, variant=gvar)
    dq, dk, dv = af.bwd(q, k, v, out, lse, do, rope_theta=1e4, variant=gvar)
    torch.cuda.synchronize()
    assert af.device_status() == 0
    q64, k64, v64, do64 = (f64(x[n]) for n in ("q", "k", "v", "dout"))
    rows = inputs.sample_rows(B, H, N, 32, seed=seed, always=[(0, 0, 0), (1, 15, N - 1), (0, 7, 1023)])
    rdq = oracle.backward_dq_rows(q64, k64, v64, do64, d ** -0.5, 1e4, True, ovar, rows)
    dqc = dq.cpu()
    check_grad(torch.stack([dqc[b, h, m] for b, h, m in rows]), rdq, "dq rows")
    _, _, _, rk, rv = oracle.backward(q64, k64, v64, do64, d ** -0.5, 1e4, True, ovar, groups=[(1, 9)])
    check_grad(dk.cpu()[1, 9], rk[1, 9], "dk[1,9]")
    check_grad(dv.cpu()[1, 9], rv[1, 9], "dv[1,9]")


@pytest.mark.parametrize("vname,N,d,B,Hq,Hkv", [
    ("bigbird", 4096, 64, 1, 2, 2),          # the mask-variant workload's BigBird layout
    ("window_1024_c", 4096, 64, 1, 2, 2),    # its sliding window + causal
    ("causal", 2048, 128, 1, 8, 2),          # GQA 4:1, head dim 128
    ("bs_128_c", 1000, 128, 2, 4, 2),        # ragged N, 128-blocks with the causal restriction
    ("bs_64", 700, 64, 1, 3, 1),             # 64-blocks, GQA 3:1
])
def test_bwd_tile_visits_match_oracle(vname, N, d, B, Hq, Hkv):
    """Both backward kernels visit exactly the active tiles (paper §4.3): the dQ kernel's
    (query tile, key tile) record equals the oracle's tile-visit set for 128 x 128 tiles, and
    the dK/dV kernel's (64-row query block, key tile) record the set for 64 x 128 tiles, bit
    for bit and for every head. Extra visits (wasted work that still gives correct gradients)
    fail here."""
    import oracle

    dev = torch.device("cuda")
    x = inputs.prefill(B, Hq, Hkv, N, d, seed=N + 3, with_dout=True)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    gvar, ovar = variant_pair(vname, N, Hq, dev, seed=5, B=B)
    out, lse = af.fwd(q, k, v, rope_theta=1e4, rope_mode=af.ROPE_FUSED, variant=gvar)
    t128, t64 = -(-N // 128), -(-N // 64)
    gvar.bwd_dq_visits = torch.zeros((B, Hq, t128, t128), dtype=torch.uint8, device=dev)
    gvar.bwd_dkdv_visits = torch.zeros((B, Hq, t64, t128), dtype=torch.uint8, device=dev)
    af.bwd(q, k, v, out, lse, do, rope_theta=1e4, rope_mode=af.ROPE_FUSED, variant=gvar)
    torch.cuda.synchronize()
    assert af.device_status() == 0
    ref_q = oracle.tile_visits(N, 128, 128, ovar)
    ref_kv = oracle.tile_visits(N, 64, 128, ovar)
    got_q, got_kv = gvar.bwd_dq_visits.cpu().numpy(), gvar.bwd_dkdv_visits.cpu().numpy()
    for b in range(B):
        for h in range(Hq):
            assert np.array_equal(got_q[b, h], ref_q), f"dQ visits differ at b={b} h={h}"
            assert np.array_equal(got_kv[b, h], ref_kv), f"dK/dV visits differ at b={b} h={h}"
