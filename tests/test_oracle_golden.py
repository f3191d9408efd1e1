"""Golden fixtures (tests/golden/): the fp64 oracle must reproduce the stored values to ~1e-13
(a change to its arithmetic is then deliberate: the fixtures are rewritten by
tests/golden/make_golden.py and the commit names the passage behind it), and the independent
brute-force restatement (tests/_bruteforce.py, math.fsum sums) must reproduce them to ~1e-12."""
import numpy as np
import pytest

from tests import _bruteforce as bf
from tests import _golden

ORC_TOL, BF_TOL = 1e-13, 1e-12


def _close(got, ref, tol, what):
    scale = max(1.0, np.abs(ref).max())
    err = np.abs(np.asarray(got) - ref).max()
    assert err <= tol * scale, f"{what}: {err:.3e} > {tol} * {scale:.3e}"


def test_inputs_are_bf16_exact():
    for name in _golden.FIXTURES:
        _, a = _golden.load(name)
        for key in ("q", "k", "v", "dout", "k_cache", "v_cache"):
            if key in a:
                x = a[key].astype(np.float32)
                assert np.array_equal(x.astype(np.float64), a[key]), (name, key)
                assert np.all((x.view(np.uint32) & 0xFFFF) == 0), (name, key)


def test_forward_fixture(orc):
    p, a = _golden.load("fwd_rope_causal_d64.txt")
    var = orc.Variant(mask=orc.MASK_CAUSAL)
    o, lse = orc.forward(a["q"], a["k"], a["v"], p["scale"], p["theta"], True, var)
    _close(o, a["out"], ORC_TOL, "oracle O")
    _close(lse, a["lse"], ORC_TOL, "oracle LSE")
    bo, blse = bf.forward(a["q"], a["k"], a["v"], p["scale"], p["theta"], True, {"mask": "causal"})
    _close(bo, a["out"], BF_TOL, "brute-force O")
    _close(blse, a["lse"], BF_TOL, "brute-force LSE")
    # first causal row sees only key 0: O_0 = v_0 for every query head of the group
    for h in range(p["Hq"]):
        _close(a["out"][0, h, 0], a["v"][0, 0, 0], 1e-15, "O_0 = v_0")


def test_backward_fixture(orc):
    p, a = _golden.load("bwd_rope_window_alibi_d64.txt")
    var = orc.Variant(mask=orc.MASK_WINDOW, window=p["window"], bias=orc.BIAS_ALIBI,
                      slopes=np.array(p["slopes"]))
    res = orc.backward(a["q"], a["k"], a["v"], a["dout"], p["scale"], p["theta"], True, var)
    spec = {"mask": "window", "window": p["window"], "bias": "alibi", "slopes": p["slopes"]}
    bo, blse = bf.forward(a["q"], a["k"], a["v"], p["scale"], p["theta"], True, spec)
    bdq, bdk, bdv, _ = bf.backward(a["q"], a["k"], a["v"], a["dout"], p["scale"], p["theta"],
                                   True, spec)
    for key, got, brute in zip(("out", "lse", "dq", "dk", "dv"), res, (bo, blse, bdq, bdk, bdv)):
        _close(got, a[key], ORC_TOL, f"oracle {key}")
        _close(brute, a[key], BF_TOL, f"brute-force {key}")


def test_decode_fixture(orc):
    p, a = _golden.load("decode_rope_d64.txt")
    o, lse = orc.decode(a["q"], a["k_cache"], a["v_cache"], p["q_pos"], p["scale"], p["theta"])
    _close(o, a["out"], ORC_TOL, "oracle O")
    _close(lse, a["lse"], ORC_TOL, "oracle LSE")
    bo, blse = bf.decode(a["q"], a["k_cache"], a["v_cache"], p["q_pos"], p["scale"], p["theta"])
    _close(bo, a["out"], BF_TOL, "brute-force O")
    _close(blse, a["lse"], BF_TOL, "brute-force LSE")
