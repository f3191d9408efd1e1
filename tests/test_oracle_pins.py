"""Pins for the fp64 oracle, independent of the oracle's own code.

Each test checks the oracle against something the pages or the mathematics fix:
closed forms, invariants, a textbook special case, an independent library routine
(torch's fp64 scaled_dot_product_attention and autograd), or finite differences.
AttnFuse paper sections cited per test.
"""
import cmath
import math

import numpy as np
import pytest
import torch

from attention_attn_fwd_bwd_gb300 import inputs

pytestmark = pytest.mark.filterwarnings("ignore")


def _rand(shape, seed):
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape)


# --------------------------------------------------------------------------------------------
# RoPE (paper §2 "Rotary Position Embeddings", §4.1 NeoX half-split)
# --------------------------------------------------------------------------------------------
def test_rope_complex_form(orc):
    """RoFormer's complex form: pair (i, i+d/2) as z = x_i + j x_{i+d/2}, rotated z e^{j p th_i}."""
    d, theta = 8, 10000.0
    x = _rand((5, d), 1)
    pos = np.array([0.0, 1.0, 7.0, 123.0, 32767.0])
    y = orc.rope(x, pos, theta)
    for r in range(5):
        for i in range(d // 2):
            th = theta ** (-2.0 * i / d)
            z = complex(x[r, i], x[r, i + d // 2]) * cmath.exp(1j * pos[r] * th)
            assert abs(y[r, i] - z.real) < 1e-12 and abs(y[r, i + d // 2] - z.imag) < 1e-12


def test_rope_d2_closed_form(orc):
    """d = 2: theta_0 = 1, so R_p is the plane rotation by p radians."""
    x = np.array([[0.3, -1.7]])
    for p in (0.0, 1.0, 2.5, 100.0):
        y = orc.rope(x, [p], 500000.0)
        c, s = math.cos(p), math.sin(p)
        assert np.allclose(y, [[0.3 * c + 1.7 * s, -1.7 * c + 0.3 * s]], atol=1e-14)


def test_rope_invariants(orc):
    d, theta = 128, 500000.0
    x = _rand((64, d), 2)
    pos = np.arange(64) * 511.0
    y = orc.rope(x, pos, theta)
    # norm preserving
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    # R_0 = identity
    assert np.array_equal(orc.rope(x, np.zeros(64), theta), x)
    # R^T R = I
    assert np.allclose(orc.rope(y, pos, theta, inverse=True), x, atol=1e-12)


def test_rope_relative_position(orc):
    """<R_m q, R_n k> depends only on m - n (paper §2)."""
    d, theta = 64, 10000.0
    q, k = _rand((1, d), 3), _rand((1, d), 4)
    for m, n in ((5, 2), (100, 37), (4000, 4000)):
        ref = (orc.rope(q, [m], theta) @ orc.rope(k, [n], theta).T).item()
        for c in (1, 17, 1000):
            got = (orc.rope(q, [m + c], theta) @ orc.rope(k, [n + c], theta).T).item()
            assert abs(got - ref) < 1e-10 * max(1.0, abs(ref))


# --------------------------------------------------------------------------------------------
# Forward: independent library routine (torch fp64 SDPA) for the post-rotation part
# --------------------------------------------------------------------------------------------
def _dense_mask(N, mask, causal=False, window=0, row_ptr=None, col_idx=None, blk=64):
    """Boolean [N, N] allowed-matrix built with numpy primitives (tril / kron)."""
    allow = np.ones((N, N), bool)
    if mask == 1 or causal:
        allow &= np.tril(np.ones((N, N), bool))
    if mask == 2:
        allow &= np.triu(np.ones((N, N), bool), -(window - 1)) & np.tril(np.ones((N, N), bool), window - 1)
    if mask == 3:
        nb = -(-N // blk)
        bm = np.zeros((nb, nb), bool)
        for r in range(nb):
            bm[r, col_idx[row_ptr[r]:row_ptr[r + 1]]] = True
        allow &= np.kron(bm, np.ones((blk, blk), bool))[:N, :N]
    return allow


def _sdpa(q, k, v, scale, allow, bias=None):
    """torch fp64 SDPA with GQA by repeat_interleave; returns O and LSE (via logsumexp)."""
    B, Hq, N, d = q.shape
    g = Hq // k.shape[1]
    qt = torch.tensor(q)
    kt = torch.tensor(k).repeat_interleave(g, dim=1)
    vt = torch.tensor(v).repeat_interleave(g, dim=1)
    am = torch.zeros(allow.shape, dtype=torch.float64)
    am[~torch.tensor(allow)] = float("-inf")
    if bias is not None:
        am = am + torch.tensor(bias)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=am, scale=scale)
    lse = torch.logsumexp(torch.einsum("bhmd,bhnd->bhmn", qt, kt) * scale + am, dim=-1)
    return o.numpy(), lse.numpy()


@pytest.mark.parametrize("mask,causal,window", [(0, 0, 0), (1, 0, 0), (2, 1, 5), (2, 0, 3)])
@pytest.mark.parametrize("gqa", [(2, 2), (4, 2), (4, 1)])
def test_forward_vs_sdpa(orc, mask, causal, window, gqa):
    Hq, Hkv = gqa
    B, N, d = 2, 19, 8
    q, k, v = _rand((B, Hq, N, d), 5), _rand((B, Hkv, N, d), 6), _rand((B, Hkv, N, d), 7)
    scale = 1 / math.sqrt(d)
    var = orc.Variant(mask=mask, causal=causal, window=window)
    o, lse = orc.forward(q, k, v, scale, 10000.0, False, var)
    ro, rl = _sdpa(q, k, v, scale, _dense_mask(N, mask, causal, window))
    assert np.allclose(o, ro, atol=1e-12)
    assert np.allclose(lse, rl, atol=1e-12)


def test_forward_rope_vs_sdpa_on_rotated(orc):
    """Fused-RoPE forward == SDPA on inputs rotated by the (separately pinned) rotation."""
    B, Hq, Hkv, N, d, theta = 1, 4, 2, 33, 16, 10000.0
    q, k, v = _rand((B, Hq, N, d), 8), _rand((B, Hkv, N, d), 9), _rand((B, Hkv, N, d), 10)
    pos = np.tile(np.arange(N, dtype=float), B * Hq)
    qr = orc.rope(q.reshape(-1, d), pos, theta).reshape(q.shape)
    kr = orc.rope(k.reshape(-1, d), np.tile(np.arange(N, dtype=float), B * Hkv), theta).reshape(k.shape)
    o, lse = orc.forward(q, k, v, 0.25, theta, True, orc.Variant(mask=1))
    ro, rl = _sdpa(qr, kr, v, 0.25, _dense_mask(N, 1))
    assert np.allclose(o, ro, atol=1e-12) and np.allclose(lse, rl, atol=1e-12)


def test_alibi_and_additive_vs_sdpa(orc):
    B, H, N, d = 1, 4, 21, 8
    q, k, v = _rand((B, H, N, d), 11), _rand((B, H, N, d), 12), _rand((B, H, N, d), 13)
    slopes = inputs.alibi_slopes(H)
    o, lse = orc.forward(q, k, v, 0.3, 1e4, False, orc.Variant(mask=1, bias=1, slopes=slopes))
    rel = np.arange(N)[None, :] - np.arange(N)[:, None]
    bias = slopes[:, None, None] * rel[None]
    ro, rl = _sdpa(q, k, v, 0.3, _dense_mask(N, 1), bias=bias[None])
    assert np.allclose(o, ro, atol=1e-12) and np.allclose(lse, rl, atol=1e-12)
    ab = _rand((1, H, N, N), 14)
    o2, l2 = orc.forward(q, k, v, 0.3, 1e4, False, orc.Variant(mask=0, bias=2, add_bias=ab))
    ro2, rl2 = _sdpa(q, k, v, 0.3, _dense_mask(N, 0), bias=ab)
    assert np.allclose(o2, ro2, atol=1e-12) and np.allclose(l2, rl2, atol=1e-12)


def test_block_sparse_vs_sdpa(orc):
    N, blk = 40, 8
    rp, ci = inputs.bigbird_csr(5, seed=3, n_random=1)
    q, k, v = _rand((1, 2, N, 8), 15), _rand((1, 2, N, 8), 16), _rand((1, 2, N, 8), 17)
    var = orc.Variant(mask=3, bs_block=blk, bs_row_ptr=rp, bs_col_idx=ci)
    o, lse = orc.forward(q, k, v, 0.5, 1e4, False, var)
    ro, rl = _sdpa(q, k, v, 0.5, _dense_mask(N, 3, row_ptr=rp, col_idx=ci, blk=blk))
    assert np.allclose(o, ro, atol=1e-12) and np.allclose(lse, rl, atol=1e-12)


# --------------------------------------------------------------------------------------------
# Forward: closed forms and special cases (paper §2 online softmax is exact; §3.1 combinators)
# --------------------------------------------------------------------------------------------
def test_zero_keys_closed_form(orc):
    """K = 0 => all scores 0: causal O_m = mean(v_0..v_m), LSE_m = ln(m+1)."""
    N, d = 50, 8
    v = _rand((1, 1, N, d), 18)
    o, lse = orc.forward(_rand((1, 1, N, d), 19), np.zeros((1, 1, N, d)), v, 1.0, 1e4, True,
                         orc.Variant(mask=1))
    assert np.allclose(lse[0, 0], np.log(np.arange(1, N + 1)), atol=1e-13)
    assert np.allclose(o[0, 0], np.cumsum(v[0, 0], axis=0) / np.arange(1, N + 1)[:, None], atol=1e-13)


def test_alibi_geometric_closed_form(orc):
    """K = 0 with ALiBi: weights e^{-slope j}; LSE_m = ln((1 - e^{-s(m+1)}) / (1 - e^{-s}))."""
    N, H = 40, 2
    slopes = np.array([0.5, 0.0625])
    o, lse = orc.forward(_rand((1, H, N, 4), 20), np.zeros((1, H, N, 4)), np.ones((1, H, N, 4)),
                         1.0, 1e4, False, orc.Variant(mask=1, bias=1, slopes=slopes))
    m = np.arange(N)
    for h, s in enumerate(slopes):
        assert np.allclose(lse[0, h], np.log((1 - np.exp(-s * (m + 1))) / (1 - np.exp(-s))), atol=1e-13)
    assert np.allclose(o, 1.0, atol=1e-13)  # rows of P sum to 1


def test_probability_rows_sum_to_one(orc):
    """V constant => O = that constant for every row and variant (sum_n P_mn = 1)."""
    B, Hq, Hkv, N, d = 1, 4, 2, 37, 8
    q, k = _rand((B, Hq, N, d), 21) * 3, _rand((B, Hkv, N, d), 22) * 3
    for var in (orc.Variant(mask=0), orc.Variant(mask=1), orc.Variant(mask=2, window=4, causal=True)):
        o, _ = orc.forward(q, k, np.full((B, Hkv, N, d), 2.5), 0.5, 1e4, True, var)
        assert np.allclose(o, 2.5, atol=1e-12)


def test_first_causal_row_is_v0(orc):
    B, H, N, d = 1, 2, 17, 8
    q, k, v = _rand((B, H, N, d), 23), _rand((B, H, N, d), 24), _rand((B, H, N, d), 25)
    for var in (orc.Variant(mask=1), orc.Variant(mask=1, bias=1, slopes=np.array([0.5, 0.25]))):
        o, _ = orc.forward(q, k, v, 0.3, 1e4, True, var)
        assert np.allclose(o[:, :, 0], v[:, :, 0], atol=1e-14)


def test_window_special_cases(orc):
    B, H, N, d = 1, 2, 23, 8
    q, k, v = _rand((B, H, N, d), 26), _rand((B, H, N, d), 27), _rand((B, H, N, d), 28)
    oc, lc = orc.forward(q, k, v, 0.3, 1e4, True, orc.Variant(mask=1))
    ow, lw = orc.forward(q, k, v, 0.3, 1e4, True, orc.Variant(mask=2, window=N, causal=True))
    assert np.array_equal(oc, ow) and np.array_equal(lc, lw)  # window >= N reproduces causal
    o1, l1 = orc.forward(q, k, v, 0.3, 1e4, False, orc.Variant(mask=2, window=1))
    assert np.allclose(o1, v, atol=1e-14)  # W = 1: each row sees only itself
    assert np.allclose(l1, 0.3 * np.einsum("bhnd,bhnd->bhn", q, k), atol=1e-13)


def test_block_sparse_special_cases(orc):
    N, blk = 48, 16
    nb = N // blk
    q, k, v = _rand((1, 2, N, 8), 29), _rand((1, 2, N, 8), 30), _rand((1, 2, N, 8), 31)
    full_rp = np.arange(nb + 1, dtype=np.int32) * nb
    full_ci = np.tile(np.arange(nb, dtype=np.int32), nb)
    of, lf = orc.forward(q, k, v, 0.3, 1e4, True, orc.Variant(mask=0))
    ob, lb = orc.forward(q, k, v, 0.3, 1e4, True,
                         orc.Variant(mask=3, bs_block=blk, bs_row_ptr=full_rp, bs_col_idx=full_ci))
    assert np.array_equal(of, ob) and np.array_equal(lf, lb)  # every block active == FULL
    tri_rp = np.cumsum([0] + [r + 1 for r in range(nb)]).astype(np.int32)
    tri_ci = np.concatenate([np.arange(r + 1) for r in range(nb)]).astype(np.int32)
    oc, lc = orc.forward(q, k, v, 0.3, 1e4, True, orc.Variant(mask=1))
    ot, lt = orc.forward(q, k, v, 0.3, 1e4, True,
                         orc.Variant(mask=3, causal=True, bs_block=blk, bs_row_ptr=tri_rp, bs_col_idx=tri_ci))
    assert np.array_equal(oc, ot) and np.array_equal(lc, lt)  # causal block pattern + causal == CAUSAL


def test_gqa_equals_repeated_mha(orc):
    B, Hq, Hkv, N, d = 2, 6, 2, 15, 8
    q, k, v = _rand((B, Hq, N, d), 32), _rand((B, Hkv, N, d), 33), _rand((B, Hkv, N, d), 34)
    o, lse = orc.forward(q, k, v, 0.4, 1e4, True, orc.Variant(mask=1))
    kr, vr = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
    o2, l2 = orc.forward(q, kr, vr, 0.4, 1e4, True, orc.Variant(mask=1))
    assert np.array_equal(o, o2) and np.array_equal(lse, l2)


def test_forward_rows_matches_full(orc):
    B, Hq, Hkv, N, d = 2, 4, 2, 29, 16
    q, k, v = _rand((B, Hq, N, d), 35), _rand((B, Hkv, N, d), 36), _rand((B, Hkv, N, d), 37)
    var = orc.Variant(mask=2, window=7, causal=True)
    o, lse = orc.forward(q, k, v, 0.3, 1e4, True, var)
    rows = inputs.sample_rows(B, Hq, N, 20, seed=1, always=[(0, 0, 0), (1, 3, N - 1)])
    ro, rl = orc.forward_rows(q, k, v, 0.3, 1e4, True, var, rows)
    for i, (b, h, m) in enumerate(rows):
        assert np.array_equal(ro[i], o[b, h, m]) and rl[i] == lse[b, h, m]


def test_fully_masked_row(orc):
    """A row with no allowed key gives O = 0 and LSE = -inf (block-sparse with an empty row)."""
    N, blk = 16, 8
    rp = np.array([0, 0, 1], np.int32)
    ci = np.array([0], np.int32)
    o, lse = orc.forward(_rand((1, 1, N, 4), 38), _rand((1, 1, N, 4), 39), _rand((1, 1, N, 4), 40),
                         1.0, 1e4, False, orc.Variant(mask=3, bs_block=blk, bs_row_ptr=rp, bs_col_idx=ci))
    assert np.all(o[0, 0, :blk] == 0) and np.all(np.isneginf(lse[0, 0, :blk]))
    assert np.all(np.isfinite(lse[0, 0, blk:]))


# --------------------------------------------------------------------------------------------
# Backward (paper §4.4): finite differences and torch autograd
# --------------------------------------------------------------------------------------------
def _variants(orc, H, N):
    rp, ci = inputs.bigbird_csr(-(-N // 4), seed=5, n_random=1)
    return [
        orc.Variant(mask=0),
        orc.Variant(mask=1),
        orc.Variant(mask=2, window=3, causal=True),
        orc.Variant(mask=1, bias=1, slopes=inputs.alibi_slopes(H)),
        orc.Variant(mask=0, bias=2, add_bias=_rand((1, H, N, N), 41)),
        orc.Variant(mask=3, bs_block=4, bs_row_ptr=rp, bs_col_idx=ci),
        orc.Variant(mask=2, window=3, bias=1, slopes=inputs.alibi_slopes(H)),
        orc.Variant(mask=3, bs_block=4, bs_row_ptr=rp, bs_col_idx=ci, causal=True,
                    bias=2, add_bias=_rand((1, 1, N, N), 75)),
    ]


@pytest.mark.parametrize("vi", range(8))
@pytest.mark.parametrize("rope_on", [False, True])
def test_backward_finite_differences(orc, vi, rope_on):
    B, Hq, Hkv, N, d, theta, scale = 1, 2, 1, 9, 4, 100.0, 0.7
    var = _variants(orc, Hq, N)[vi]
    q, k, v = _rand((B, Hq, N, d), 42), _rand((B, Hkv, N, d), 43), _rand((B, Hkv, N, d), 44)
    do = _rand((B, Hq, N, d), 45)
    _, _, dq, dk, dv = orc.backward(q, k, v, do, scale, theta, rope_on, var)

    def loss(qq, kk, vv):
        o, _ = orc.forward(qq, kk, vv, scale, theta, rope_on, var)
        return float(np.sum(o * do))

    h = 1e-6
    for x, gx, idx in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(x)
        for i in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[i] += h
            xm[i] -= h
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[idx], args_m[idx] = xp, xm
            num[i] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.allclose(gx, num, atol=1e-6 * max(1.0, np.abs(num).max()), rtol=1e-6)


def test_backward_vs_torch_autograd(orc):
    B, Hq, Hkv, N, d = 2, 4, 2, 23, 8
    q, k, v = _rand((B, Hq, N, d), 46), _rand((B, Hkv, N, d), 47), _rand((B, Hkv, N, d), 48)
    do = _rand((B, Hq, N, d), 49)
    o, lse, dq, dk, dv = orc.backward(q, k, v, do, 0.35, 1e4, False, orc.Variant(mask=1))
    qt, kt, vt = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    ot = torch.nn.functional.scaled_dot_product_attention(
        qt, kt.repeat_interleave(2, 1), vt.repeat_interleave(2, 1), is_causal=True, scale=0.35)
    ot.backward(torch.tensor(do))
    assert np.allclose(o, ot.detach().numpy(), atol=1e-12)
    for a, b in ((dq, qt), (dk, kt), (dv, vt)):
        assert np.allclose(a, b.grad.numpy(), atol=1e-11)


@pytest.mark.parametrize("rope_on", [False, True])
@pytest.mark.parametrize("causal", [False, True])
def test_dbias_finite_differences(orc, rope_on, causal):
    """dBias (the gradient with respect to an additive bias, §3.1 additive_bias) against central
    differences of the forward in the bias itself."""
    B, H, N, d, theta, scale = 1, 2, 7, 4, 100.0, 0.6
    q, k, v = _rand((B, H, N, d), 60), _rand((B, H, N, d), 61), _rand((B, H, N, d), 62)
    do = _rand((B, H, N, d), 63)
    ab = _rand((B, H, N, N), 64)
    var = orc.Variant(mask=1 if causal else 0, bias=2, add_bias=ab)
    *_, db = orc.backward(q, k, v, do, scale, theta, rope_on, var, with_dbias=True)
    h = 1e-6
    num = np.zeros_like(ab)
    for i in np.ndindex(ab.shape):
        ap, am = ab.copy(), ab.copy()
        ap[i] += h
        am[i] -= h
        op, _ = orc.forward(q, k, v, scale, theta, rope_on, orc.Variant(mask=var.mask, bias=2, add_bias=ap))
        om, _ = orc.forward(q, k, v, scale, theta, rope_on, orc.Variant(mask=var.mask, bias=2, add_bias=am))
        num[i] = (np.sum(op * do) - np.sum(om * do)) / (2 * h)
    assert np.allclose(db, num, atol=1e-7, rtol=1e-6)


def test_dbias_vs_torch_autograd(orc):
    """dBias equals the autograd gradient of torch's fp64 SDPA with respect to a float mask."""
    B, H, N, d = 2, 3, 13, 8
    q, k, v = _rand((B, H, N, d), 65), _rand((B, H, N, d), 66), _rand((B, H, N, d), 67)
    do = _rand((B, H, N, d), 68)
    ab = _rand((B, H, N, N), 69)
    var = orc.Variant(mask=1, bias=2, add_bias=ab)
    _, _, dq, dk, dv, db = orc.backward(q, k, v, do, 0.4, 1e4, False, var, with_dbias=True)
    qt, kt, vt = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    bt = torch.tensor(ab, requires_grad=True)
    am = torch.zeros(N, N, dtype=torch.float64)
    am[~torch.tensor(_dense_mask(N, 1))] = float("-inf")
    ot = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=am + bt, scale=0.4)
    ot.backward(torch.tensor(do))
    assert np.allclose(db, bt.grad.numpy(), atol=1e-12)
    for a, t in ((dq, qt), (dk, kt), (dv, vt)):
        assert np.allclose(a, t.grad.numpy(), atol=1e-11)


def test_dbias_rows_sum_to_zero_and_masked_zero(orc):
    """sum_n dS_mn = sum_n P_mn dP_mn - D_m = 0 (softmax Jacobian rows), and dBias is exactly 0
    wherever the mask forbids (m, n) (§4.3: masked pairs carry no gradient)."""
    B, H, N, d = 1, 2, 24, 8
    rp, ci = inputs.bigbird_csr(6, seed=7, n_random=1)
    ab = _rand((1, H, N, N), 70)
    for var in (orc.Variant(mask=2, window=5, causal=True, bias=2, add_bias=ab),
                orc.Variant(mask=3, bs_block=4, bs_row_ptr=rp, bs_col_idx=ci, bias=2, add_bias=ab)):
        q, k, v = _rand((B, H, N, d), 71), _rand((B, H, N, d), 72), _rand((B, H, N, d), 73)
        do = _rand((B, H, N, d), 74)
        *_, db = orc.backward(q, k, v, do, 0.5, 1e4, True, var, with_dbias=True)
        assert np.allclose(db.sum(-1), 0.0, atol=1e-12)
        allow = _dense_mask(N, var.mask, var.causal, var.window, row_ptr=rp, col_idx=ci, blk=4)
        assert np.all(db[:, :, ~allow] == 0.0)


def test_backward_groups_and_rows(orc):
    B, Hq, Hkv, N, d = 2, 4, 2, 17, 8
    q, k, v = _rand((B, Hq, N, d), 50), _rand((B, Hkv, N, d), 51), _rand((B, Hkv, N, d), 52)
    do = _rand((B, Hq, N, d), 53)
    var = orc.Variant(mask=1)
    full = orc.backward(q, k, v, do, 0.3, 1e4, True, var)
    part = orc.backward(q, k, v, do, 0.3, 1e4, True, var, groups=[(1, 0)])
    assert np.array_equal(part[3][1, 0], full[3][1, 0]) and np.array_equal(part[4][1, 0], full[4][1, 0])
    assert np.array_equal(part[2][1, 0:2], full[2][1, 0:2])
    rows = np.array([(0, 3, 16), (1, 0, 0), (1, 2, 9)])
    dqr = orc.backward_dq_rows(q, k, v, do, 0.3, 1e4, True, var, rows)
    for i, (b, h, m) in enumerate(rows):
        assert np.allclose(dqr[i], full[2][b, h, m], atol=1e-13)


# --------------------------------------------------------------------------------------------
# Decode (paper §4.2) and tile visits (§4.3)
# --------------------------------------------------------------------------------------------
def test_decode_equals_last_prefill_row(orc):
    B, Hq, Hkv, L, d, theta = 1, 8, 2, 40, 16, 5e5
    q, k, v = _rand((B, Hq, L, d), 54), _rand((B, Hkv, L, d), 55), _rand((B, Hkv, L, d), 56)
    o, lse = orc.forward(q, k, v, 0.25, theta, True, orc.Variant(mask=1))
    krot = orc.rope(k.reshape(-1, d), np.tile(np.arange(L, dtype=float), B * Hkv), theta).reshape(k.shape)
    od, ld = orc.decode(q[:, :, -1], krot, v, L - 1, 0.25, theta, rope_q=True)
    assert np.allclose(od, o[:, :, -1], atol=1e-12) and np.allclose(ld, lse[:, :, -1], atol=1e-12)


def test_decode_vs_sdpa(orc):
    B, Hq, Hkv, L, d = 2, 8, 2, 33, 16
    q, k, v = _rand((B, Hq, d), 57), _rand((B, Hkv, L, d), 58), _rand((B, Hkv, L, d), 59)
    od, ld = orc.decode(q, k, v, 1000, 0.25, 1e4, rope_q=False)
    ro, rl = _sdpa(q[:, :, None], k, v, 0.25, np.ones((1, L), bool))
    assert np.allclose(od, ro[:, :, 0], atol=1e-12) and np.allclose(ld, rl[:, :, 0], atol=1e-12)


def test_tile_visits(orc):
    N = 1000
    T = -(-N // 128)
    vis = orc.tile_visits(N, 128, 128, orc.Variant(mask=1))
    assert vis.sum() == T * (T + 1) // 2 and np.array_equal(vis, np.tril(np.ones((T, T), np.uint8)))
    vw = orc.tile_visits(4096, 128, 128, orc.Variant(mask=2, window=1024, causal=True))
    # tile (i, j) visited iff j <= i and the window reaches it: 128 j + 127 > 128 i - 1024
    ii, jj = np.meshgrid(np.arange(32), np.arange(32), indexing="ij")
    assert np.array_equal(vw, ((jj <= ii) & (128 * jj + 127 > 128 * ii - 1024)).astype(np.uint8))
    rp, ci = inputs.bigbird_csr(64, seed=3003)
    vb = orc.tile_visits(4096, 64, 64, orc.Variant(mask=3, bs_block=64, bs_row_ptr=rp, bs_col_idx=ci))
    dense = np.zeros((64, 64), np.uint8)
    for r in range(64):
        dense[r, ci[rp[r]:rp[r + 1]]] = 1
    assert np.array_equal(vb, dense)
    assert orc.allowed_pairs(4096, orc.Variant(mask=3, bs_block=64, bs_row_ptr=rp, bs_col_idx=ci)) == len(ci) * 64 * 64
    assert orc.allowed_pairs(N, orc.Variant(mask=1)) == N * (N + 1) // 2


@pytest.mark.parametrize("BM,BN", [(256, 128), (128, 256), (64, 128)])
def test_tile_visits_rectangular_tiles(orc, BM, BN):
    """Query and key tiles of different heights. A causal (window) tile pair is visited iff the
    key tile's first key is at or before the query tile's last row (and its last key is still
    inside the first row's window): interval bounds, not the element loop of the oracle."""
    N, W = 1000, 300
    TQ, TK = -(-N // BM), -(-N // BN)
    i, j = np.meshgrid(np.arange(TQ), np.arange(TK), indexing="ij")
    m_lo, m_hi = BM * i, np.minimum(BM * i + BM - 1, N - 1)
    n_lo, n_hi = BN * j, np.minimum(BN * j + BN - 1, N - 1)
    vis = orc.tile_visits(N, BM, BN, orc.Variant(mask=1))
    assert vis.shape == (TQ, TK)
    assert np.array_equal(vis, (n_lo <= m_hi).astype(np.uint8))
    vw = orc.tile_visits(N, BM, BN, orc.Variant(mask=2, window=W, causal=True))
    assert np.array_equal(vw, ((n_lo <= m_hi) & (n_hi > m_lo - W)).astype(np.uint8))


def test_bigbird_layout_structure():
    rp, ci = inputs.bigbird_csr(64, seed=3003)
    for r in range(64):
        cols = ci[rp[r]:rp[r + 1]]
        assert np.all(np.diff(cols) > 0)
        if r < 2:
            assert len(cols) == 64
        else:
            assert {0, 1, r}.issubset(set(cols.tolist()))
            assert len(cols) == len({0, 1} | {c for c in (r - 1, r, r + 1) if c < 64}) + 3


def test_relu_attention_closed_forms(orc):
    """relu_attention (this build's reading of the paper's §3.1 normaliser: weights
    max(s, 0) / N, N the number of keys). Pins that separate it from nearby mistakes:
    - every score positive and equal (q = k = u, no RoPE): causal row m is
      (scale |u|^2 / N) * sum_{n<=m} v_n, divided by N, not by the m + 1 visible keys;
    - every score negative (q = -u): O = 0 exactly (the relu is applied);
    - positive homogeneity: O(a q) = a O(q) for a > 0, which no exponential satisfies."""
    rng = np.random.default_rng(11)
    B, H, N, d, scale = 1, 2, 12, 8, 0.3
    u = rng.standard_normal(d)
    k = np.broadcast_to(u, (B, H, N, d)).copy()
    v = rng.standard_normal((B, H, N, d))
    var = orc.Variant(mask=orc.MASK_CAUSAL, norm=orc.NORM_RELU)
    o, lse = orc.forward(k.copy(), k, v, scale, 1e4, False, var)
    c = scale * float(u @ u) / N
    assert np.allclose(o, c * np.cumsum(v, axis=2), rtol=0, atol=1e-12)
    assert np.all(np.isnan(lse))
    o_neg, _ = orc.forward(-k, k, v, scale, 1e4, False, var)
    assert np.array_equal(o_neg, np.zeros_like(o_neg))
    q = rng.standard_normal((B, H, N, d))
    kk = rng.standard_normal((B, H, N, d))
    for rope_on in (False, True):
        o1, _ = orc.forward(q, kk, v, scale, 1e4, rope_on, orc.Variant(mask=orc.MASK_FULL, norm=orc.NORM_RELU))
        o3, _ = orc.forward(3.0 * q, kk, v, scale, 1e4, rope_on, orc.Variant(mask=orc.MASK_FULL, norm=orc.NORM_RELU))
        assert np.allclose(o3, 3.0 * o1, rtol=0, atol=1e-12)
        assert not np.allclose(o1, 0.0)


def test_decode_e4m3_closed_forms_and_library():
    """E4M3 (OCP 8-bit floating point): 1.0 = 0 0111 000, the largest finite value 448 =
    0 1111 110, the smallest subnormal 2^-9 = 0 0000 001, the smallest normal 2^-6, sign bit,
    NaN at x 1111 111; and all 256 codes against torch's float8_e4m3fn widening (an
    independent library routine)."""
    import oracle

    d = oracle.decode_e4m3
    assert d(0x38) == 1.0 and d(0xB8) == -1.0
    assert d(0x7E) == 448.0 and d(0xFE) == -448.0
    assert d(0x01) == 2.0 ** -9 and d(0x07) == 7 * 2.0 ** -9
    assert d(0x08) == 2.0 ** -6 and d(0x0F) == 2.0 ** -6 * 1.875
    assert d(0x00) == 0.0 and np.signbit(d(0x80))
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    b = np.arange(256)
    ref = torch.tensor(b, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = d(b)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    fin = ~np.isnan(ref)
    assert np.array_equal(ref[fin], got[fin])
