"""Brute-force pins of the fp64 oracle: on tiny inputs, the oracle's forward, backward (with
dBias) and decode must agree with the plain-Python restatement in tests/_bruteforce.py, which
takes every sum with math.fsum, to ~1e-12. Cases cover every mask kind (with and without the
causal restriction), both bias kinds, RoPE on and off, GQA groups, ragged block-sparse rows and
a block row with no active block (fully masked rows: O = 0, LSE = -inf)."""
import zlib

import numpy as np
import pytest

from tests import _bruteforce as bf

TOL = 1e-12


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _orc_variant(orc, spec):
    kinds = {"full": 0, "causal": 1, "window": 2, "block_sparse": 3}
    kw = dict(mask=kinds[spec["mask"]], causal=spec.get("causal", False))
    if spec["mask"] == "window":
        kw["window"] = spec["window"]
    if spec["mask"] == "block_sparse":
        kw.update(bs_block=spec["block"], bs_row_ptr=np.array(spec["row_ptr"]),
                  bs_col_idx=np.array(spec["col_idx"]))
    if spec.get("bias") == "alibi":
        kw.update(bias=1, slopes=np.array(spec["slopes"]))
    elif spec.get("bias") == "additive":
        kw.update(bias=2, add_bias=spec["add_bias"])
    if spec.get("norm") == "relu":
        kw["norm"] = 1
    return orc.Variant(**kw)


def _close(got, ref, what):
    got, ref = np.asarray(got), np.asarray(ref)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: -inf pattern differs"
    assert np.all(got[~fin] == ref[~fin]), what
    if fin.any():
        scale = max(1.0, np.abs(ref[fin]).max())
        err = np.abs(got[fin] - ref[fin]).max()
        assert err <= TOL * scale, f"{what}: {err:.3e} > {TOL} * {scale:.3e}"


def _cases():
    rng = np.random.default_rng(7)
    # (name, B, Hq, Hkv, N, d, rope_on, theta, scale, spec)
    yield "full_rope", 1, 4, 2, 9, 8, True, 1e4, 0.35, {"mask": "full"}
    yield "causal_alibi_rope", 2, 2, 1, 9, 8, True, 5e5, 0.3, {
        "mask": "causal", "bias": "alibi", "slopes": [2.0 ** -4, 2.0 ** -8]}
    yield "window3_additive", 1, 2, 2, 10, 4, False, 1e4, 0.5, {
        "mask": "window", "window": 3, "bias": "additive", "add_bias": _rand(rng, 1, 2, 10, 10)}
    yield "window4_causal_rope", 1, 4, 1, 11, 8, True, 1e4, 0.25, {
        "mask": "window", "window": 4, "causal": True}
    # 150 rows in blocks of 64: block row 1 lists no block, so rows 64..127 see no key
    yield "block_sparse_rope", 1, 2, 1, 150, 4, True, 1e4, 0.5, {
        "mask": "block_sparse", "block": 64, "row_ptr": [0, 2, 2, 4], "col_idx": [0, 2, 1, 2]}
    yield "block_sparse_causal_additive", 1, 2, 1, 140, 4, True, 1e4, 0.5, {
        "mask": "block_sparse", "block": 64, "causal": True, "row_ptr": [0, 1, 3, 5],
        "col_idx": [0, 0, 1, 1, 2], "bias": "additive", "add_bias": _rand(rng, 1, 1, 140, 140)}


CASES = list(_cases())


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_forward_and_backward_match_brute_force(orc, case):
    name, B, Hq, Hkv, N, d, rope_on, theta, scale, spec = case
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    q, k, v = _rand(rng, B, Hq, N, d), _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    dout = _rand(rng, B, Hq, N, d)
    var = _orc_variant(orc, spec)
    with_db = spec.get("bias") == "additive"
    res = orc.backward(q, k, v, dout, scale, theta, rope_on, var, with_dbias=with_db)
    o, lse, dq, dk, dv = res[:5]
    bo, blse = bf.forward(q, k, v, scale, theta, rope_on, spec)
    _close(o, bo, "O")
    _close(lse, blse, "LSE")
    fo, flse = orc.forward(q, k, v, scale, theta, rope_on, var)
    _close(fo, bo, "forward O")
    _close(flse, blse, "forward LSE")
    bdq, bdk, bdv, bdb = bf.backward(q, k, v, dout, scale, theta, rope_on, spec)
    _close(dq, bdq, "dQ")
    _close(dk, bdk, "dK")
    _close(dv, bdv, "dV")
    if with_db:
        _close(res[5], bdb, "dBias")
    if spec["mask"] == "block_sparse" and spec["row_ptr"][1] == spec["row_ptr"][2]:
        assert np.all(np.isneginf(lse[:, :, 64:128])) and np.all(o[:, :, 64:128] == 0)


def test_decode_matches_brute_force(orc):
    rng = np.random.default_rng(11)
    B, Hq, Hkv, L, d = 2, 4, 2, 11, 8
    q, kc, vc = _rand(rng, B, Hq, d), _rand(rng, B, Hkv, L, d), _rand(rng, B, Hkv, L, d)
    for rope_q in (True, False):
        o, lse = orc.decode(q, kc, vc, L - 1, 0.35, 5e5, rope_q=rope_q)
        bo, blse = bf.decode(q, kc, vc, L - 1, 0.35, 5e5, rope_q=rope_q)
        _close(o, bo, "decode O")
        _close(lse, blse, "decode LSE")


def test_rope_matches_brute_force(orc):
    rng = np.random.default_rng(13)
    x = _rand(rng, 6, 8)
    pos = np.array([0, 1, 7, 100, 4095, 32767], np.float64)
    for inverse in (False, True):
        y = orc.rope(x, pos, 5e5, inverse=inverse)
        by = np.array([bf.rotate(list(x[r]), pos[r], 5e5, inverse) for r in range(6)])
        _close(y, by, "rope")


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_relu_forward_matches_brute_force(orc, case):
    """The relu_attention normaliser over every mask and bias kind: O agrees with the brute
    force to 1e-12 and no LSE is defined (NaN)."""
    name, B, Hq, Hkv, N, d, rope_on, theta, scale, spec = case
    spec = dict(spec, norm="relu")
    rng = np.random.default_rng(zlib.crc32(name.encode()) + 1)
    q, k, v = _rand(rng, B, Hq, N, d), _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    o, lse = orc.forward(q, k, v, scale, theta, rope_on, _orc_variant(orc, spec))
    bo, _ = bf.forward(q, k, v, scale, theta, rope_on, spec)
    _close(o, bo, "relu O")
    assert np.all(np.isnan(lse))
