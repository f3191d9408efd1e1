"""GPU parity on the golden fixtures (tests/golden/): the library's fused-RoPE forward,
backward (window + ALiBi) and decode, run through the C ABI on the fixtures' bf16-exact inputs,
must match the stored fp64 values within the usual tolerances (O max-abs 2e-2 / mean-abs 2e-3,
LSE 1e-3 relative, gradients 5e-2 of the largest reference gradient). The fixtures are tiny
(N = 5 to 7, below one 128-row tile): every tile is ragged and every row is a tail row."""
import pytest
import torch

import attention_attn_fwd_bwd_gb300 as af
from tests import _golden
from tests._helpers import check_grad, check_lse, check_out

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from attention_attn_fwd_bwd_gb300 import _build

    _build.build()
    af.load()
    assert af.device_status() == 0


def _dev(a):
    return torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).cuda().contiguous()


def test_golden_forward():
    p, a = _golden.load("fwd_rope_causal_d64.txt")
    q, k, v = _dev(a["q"]), _dev(a["k"]), _dev(a["v"])
    for mode in (af.ROPE_FUSED, af.ROPE_PREROTATE):
        out, lse = af.fwd(q, k, v, scale=p["scale"], rope_theta=p["theta"], rope_mode=mode,
                          variant=af.Variant(mask=af.MASK_CAUSAL))
        torch.cuda.synchronize()
        assert af.device_status() == 0
        check_out(out, a["out"])
        check_lse(lse, a["lse"])


def test_golden_backward():
    p, a = _golden.load("bwd_rope_window_alibi_d64.txt")
    q, k, v, do = _dev(a["q"]), _dev(a["k"]), _dev(a["v"]), _dev(a["dout"])
    var = af.Variant(mask=af.MASK_WINDOW, window=p["window"], causal=False, bias=af.BIAS_ALIBI,
                     alibi_slopes=torch.tensor(p["slopes"], dtype=torch.float32).cuda())
    out, lse = af.fwd(q, k, v, scale=p["scale"], rope_theta=p["theta"], rope_mode=af.ROPE_FUSED,
                      variant=var)
    check_out(out, a["out"])
    check_lse(lse, a["lse"])
    for mode in (af.ROPE_FUSED, af.ROPE_PREROTATE):
        dq, dk, dv = af.bwd(q, k, v, out, lse, do, scale=p["scale"], rope_theta=p["theta"],
                            rope_mode=mode, variant=var)
        torch.cuda.synchronize()
        assert af.device_status() == 0
        check_grad(dq, a["dq"], "dQ")
        check_grad(dk, a["dk"], "dK")
        check_grad(dv, a["dv"], "dV")


def test_golden_decode():
    p, a = _golden.load("decode_rope_d64.txt")
    q = _dev(a["q"])
    kc, vc = _dev(a["k_cache"]), _dev(a["v_cache"])
    for splits in (0, 1, 3):
        out, lse = af.decode(q, kc, vc, p["q_pos"], scale=p["scale"], rope_theta=p["theta"],
                             rope_mode=af.ROPE_FUSED, num_splits=splits)
        torch.cuda.synchronize()
        assert af.device_status() == 0
        check_out(out, a["out"])
        check_lse(lse, a["lse"])
