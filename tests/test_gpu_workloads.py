"""GPU parity on the paper's other workloads (§6.1-§6.3): GPT-2-small geometry forwards
(B=4, H=12, d=64) for dense, causal, causal sliding window 256, causal + ALiBi and fused RoPE +
dense / causal / sliding window; decode at the Llama-3-8B (Hq=32, Hkv=8, d=128, L=4096) and
Mistral-7B (L=16384) head shapes."""
import math

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


CELLS = {
    "dense": (af.ROPE_NONE, dict(mask=0), dict(mask=0)),
    "causal": (af.ROPE_NONE, dict(mask=1), dict(mask=1)),
    "sw256": (af.ROPE_NONE, dict(mask=2, window=256, causal=True), dict(mask=2, window=256, causal=True)),
    "causal_alibi": (af.ROPE_NONE, dict(mask=1, bias=1), dict(mask=1, bias=1)),
    "rope_dense": (af.ROPE_FUSED, dict(mask=0), dict(mask=0)),
    "rope_causal": (af.ROPE_FUSED, dict(mask=1), dict(mask=1)),
    "rope_sw256": (af.ROPE_FUSED, dict(mask=2, window=256, causal=True), dict(mask=2, window=256, causal=True)),
}


def _gpt2(name, N, rows=None):
    import oracle

    B, H, d = 4, 12, 64
    dev = torch.device("cuda")
    mode, gkw, okw = CELLS[name]
    gkw, okw = dict(gkw), dict(okw)
    sl = inputs.alibi_slopes(H)
    if gkw.get("bias") == 1:
        gkw["alibi_slopes"] = torch.tensor(sl, dtype=torch.float32, device=dev)
        okw["slopes"] = sl.astype(np.float32).astype(np.float64)
    x = inputs.prefill(B, H, H, N, d, seed=6000 + N)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    out, lse = af.fwd(q, k, v, rope_theta=1e4, rope_mode=mode, variant=af.Variant(**gkw))
    torch.cuda.synchronize()
    assert af.device_status() == 0
    args = (f64(x["q"]), f64(x["k"]), f64(x["v"]), 1 / math.sqrt(d), 1e4, mode != af.ROPE_NONE,
            oracle.Variant(**okw))
    if rows is None:
        o, l = oracle.forward(*args)
        check_out(out, o)
        check_lse(lse, l)
    else:
        o, l = oracle.forward_rows(*args, rows)
        oc, lc = out.cpu(), lse.cpu()
        check_out(torch.stack([oc[b, h, m] for b, h, m in rows]), o)
        check_lse(torch.stack([lc[b, h, m] for b, h, m in rows]), l)


@pytest.mark.parametrize("name", sorted(CELLS))
def test_gpt2_small_geometry_n512(name):
    _gpt2(name, 512)


@pytest.mark.parametrize("name", ["dense", "causal_alibi", "rope_sw256"])
def test_gpt2_small_geometry_n4096_sampled(name):
    rows = inputs.sample_rows(4, 12, 4096, 32, seed=11, always=[(0, 0, 0), (3, 11, 4095), (2, 5, 255)])
    _gpt2(name, 4096, rows)


@pytest.mark.parametrize("L,B", [(4096, 8), (16384, 1), (16384, 8)])
def test_decode_llama8b_mistral7b_head_shapes(L, B):
    import oracle

    Hq, Hkv, d = 32, 8, 128
    x = inputs.decode(B, Hq, Hkv, L, d, seed=7000 + L + B)
    dev = torch.device("cuda")
    q, kc, vc = x["q"].to(dev), x["k_cache"].to(dev), x["v_cache"].to(dev)
    out, lse = af.decode(q, kc, vc, L - 1, rope_theta=5e5)
    torch.cuda.synchronize()
    assert af.device_status() == 0
    o, l = oracle.decode(f64(x["q"]), f64(x["k_cache"]), f64(x["v_cache"]), L - 1, d ** -0.5, 5e5)
    check_out(out, o)
    check_lse(lse, l)


def test_cuda_graph_capture_replays_bit_identically():
    """Forward, backward and decode are capturable in a CUDA graph (launches only, buffers
    preallocated); replays reproduce the eager results bit for bit."""
    dev = torch.device("cuda")
    x = inputs.prefill(2, 8, 2, 640, 128, seed=71, with_dout=True)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    out, lse = torch.empty_like(q), torch.empty((2, 8, 640), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsf = torch.empty(af.fwd_workspace_size(2, 8, 2, 640, 128, af.ROPE_FUSED), dtype=torch.uint8, device=dev)
    wsb = torch.empty(af.bwd_workspace_size(2, 8, 2, 640, 128, af.ROPE_FUSED), dtype=torch.uint8, device=dev)
    xd = inputs.decode(2, 32, 8, 3000, 128, seed=72)
    qd, kc, vc = (xd[n].to(dev) for n in ("q", "k_cache", "v_cache"))
    od, ld = torch.empty_like(qd), torch.empty((2, 32), dtype=torch.float32, device=dev)
    wsd = torch.empty(af.decode_workspace_size(2, 32, 8, 3000, 128, 0), dtype=torch.uint8, device=dev)

    def step():
        af.fwd(q, k, v, rope_theta=5e5, out=out, lse=lse, workspace=wsf)
        af.bwd(q, k, v, out, lse, do, rope_theta=5e5, dq=dq, dk=dk, dv=dv, workspace=wsb)
        af.decode(qd, kc, vc, 2999, rope_theta=5e5, out=od, lse=ld, workspace=wsd)

    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (out, lse, dq, dk, dv, od, ld)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in (out, lse, dq, dk, dv, od, ld):
        t.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert af.device_status() == 0
    for a, b in zip(eager, (out, lse, dq, dk, dv, od, ld)):
        assert torch.equal(a, b)
