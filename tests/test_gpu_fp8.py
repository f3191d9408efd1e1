"""GPU parity of the e4m3 forward (fp8 attention, named as future work in the AttnFuse paper
§9.1) against the fp64 oracle.

The inputs are e4m3 bytes with per-tensor scales (``inputs.prefill_e4m3``); the oracle
attends over exactly the decoded values scale * e4m3(byte) (``oracle.decode_e4m3``), so the
comparison measures only the kernel's arithmetic: exact e4m3 products summed in fp32 for the
scores, P rounded to bf16, V widened exactly to bf16, O rounded to bf16. That is the error
budget of the bf16 forward, and the tolerances are the same (O max-abs 2e-2 and mean-abs
2e-3, LSE 1e-3 relative). Covers every mask and bias kind, both normalisers, GQA ratios that
map to each unit shape, ragged N, the Llama-3-8B shape (one whole (b, h) slice plus sampled
rows), tile-visit sets and argument errors."""
import math

import numpy as np
import pytest
import torch

import attention_attn_fwd_bwd_gb300 as af
from attention_attn_fwd_bwd_gb300 import inputs
from tests._helpers import check_lse, check_out, variant_pair

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from attention_attn_fwd_bwd_gb300 import _build

    _build.build()
    af.load()
    assert af.device_status() == 0


def _decoded(x, name):
    import oracle

    return oracle.decode_e4m3(x[name].numpy()) * x[name + "_scale"]


def _run(B, Hq, Hkv, N, vname, seed, rows=None, norm=None, visits=False):
    import oracle

    dev = torch.device("cuda")
    x = inputs.prefill_e4m3(B, Hq, Hkv, N, 128, seed)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    gvar, ovar = variant_pair(vname, N, Hq, dev, seed, B=B)
    if norm == "relu":
        gvar.norm, ovar.norm = af.NORM_RELU, oracle.NORM_RELU
    TQ = -(-N // 128)
    if visits:
        gvar.tile_visits = torch.zeros((B, Hq, TQ, TQ), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(128)
    out, lse = af.fwd_fp8(q, k, v, x["q_scale"], x["k_scale"], x["v_scale"], scale=scale,
                          variant=gvar)
    torch.cuda.synchronize()
    assert af.device_status() == 0
    q64, k64, v64 = _decoded(x, "q"), _decoded(x, "k"), _decoded(x, "v")
    if rows is None:
        o_ref, l_ref = oracle.forward(q64, k64, v64, scale, 1e4, False, ovar)
        check_out(out, o_ref)
        if norm != "relu":
            check_lse(lse, l_ref)
    else:
        o_ref, l_ref = oracle.forward_rows(q64, k64, v64, scale, 1e4, False, ovar, rows)
        oc, lc = out.cpu(), lse.cpu()
        check_out(torch.stack([oc[b, h, m] for b, h, m in rows]), o_ref)
        check_lse(torch.stack([lc[b, h, m] for b, h, m in rows]), l_ref)
    if visits:
        ref_vis = oracle.tile_visits(N, 128, 128, ovar)
        got = gvar.tile_visits.cpu().numpy()
        assert all(np.array_equal(got[b, h], ref_vis) for b in range(B) for h in range(Hq))
    return out


@pytest.mark.parametrize("gqa", [(4, 1), (8, 2), (2, 2), (3, 1)])
@pytest.mark.parametrize("N", [1, 100, 128, 300, 1000])
def test_fp8_shapes_causal(gqa, N):
    _run(1, gqa[0], gqa[1], N, "causal", seed=500 + N + gqa[0])


@pytest.mark.parametrize("vname", ["full", "window_100_c", "window_70", "alibi", "alibi_full",
                                   "addbias_f32", "addbias_bf16_bcast_c", "bs_64", "bs_128_c"])
def test_fp8_variants(vname):
    _run(2, 4, 2, 517, vname, seed=600 + len(vname), visits=not vname.startswith("addbias"))


def test_fp8_relu_normaliser():
    _run(1, 4, 1, 333, "causal", seed=77, norm="relu")


def test_fp8_full_size_llama8b():
    """B=4, Hq=32, Hkv=8, N=4096, causal: one whole (b, h) slice plus sampled rows."""
    rows = inputs.sample_rows(4, 32, 4096, 40, seed=8, always=[(0, 0, 0), (3, 31, 4095)])
    m = np.arange(4096, dtype=np.int64)
    rows = np.concatenate([rows, np.stack([np.full_like(m, 2), np.full_like(m, 7), m], axis=1)])
    _run(4, 32, 8, 4096, "causal", seed=8000, rows=rows)


def test_fp8_float8_dtype_and_determinism():
    """torch.float8_e4m3fn tensors are accepted as the same bytes; two calls agree bitwise."""
    dev = torch.device("cuda")
    x = inputs.prefill_e4m3(1, 8, 2, 700, 128, 9)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    sc = (x["q_scale"], x["k_scale"], x["v_scale"])
    a, la = af.fwd_fp8(q, k, v, *sc)
    b, lb = af.fwd_fp8(q.view(torch.float8_e4m3fn), k.view(torch.float8_e4m3fn),
                       v.view(torch.float8_e4m3fn), *sc)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_fp8_argument_errors():
    dev = torch.device("cuda")
    x = inputs.prefill_e4m3(1, 2, 2, 64, 128, 3)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    with pytest.raises(af.AttnfuseError, match="scale"):
        af.fwd_fp8(q, k, v, 0.0, 1.0, 1.0)
    with pytest.raises(af.AttnfuseError, match="scale"):
        af.fwd_fp8(q, k, v, 1.0, float("inf"), 1.0)
    q64 = torch.zeros((1, 2, 64, 64), dtype=torch.uint8, device=dev)
    with pytest.raises(af.AttnfuseError, match="head dim 128"):
        af.fwd_fp8(q64, q64, q64, 1.0, 1.0, 1.0)
    with pytest.raises(TypeError):
        af.fwd_fp8(q.to(torch.int8), k, v, 1.0, 1.0, 1.0)
