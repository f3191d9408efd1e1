"""Brute-force restatement of the attention definition, for pinning the fp64 oracle on tiny
inputs. Plain Python: every sum is math.fsum (exactly rounded), rotations use math.cos /
math.sin of p * theta_i. It shares no code with oracle/attn_oracle.c or the CUDA library.

What it computes (AttnFuse paper):
  - RoPE, NeoX half-split pairs (i, i + d/2), theta_i = theta^(-2i/d), position p = token
    index (§4.1): x'_i = x_i cos - x_{i+d/2} sin, x'_{i+d/2} = x_{i+d/2} cos + x_i sin;
  - score s = scale * <q'_m, k'_n> plus the bias combinator (ALiBi slope_h * (n - m), or an
    additive bias[b, h, m, n]) (§2, §3.1);
  - the mask combinators (causal n <= m; window |m - n| < W, with n <= m when causal;
    block-sparse: block (m // blk, n // blk) listed in the CSR, with n <= m when causal) (§3.1,
    §4.3);
  - softmax over the allowed keys with LSE = max + ln(sum exp(s - max)); O = P V; a row with
    no allowed key has O = 0 and LSE = -inf (§2, §4.4);
  - the backward by direct differentiation: D = rowsum(dO * O), dS = P (dP - D), dQ' =
    scale dS K', dK' = scale dS^T Q', dV = P^T dO, then dQ = R^T dQ', dK = R^T dK', dK and
    dV summed over the query heads of a group, dBias = dS (§4.4);
  - the decode step: one query row at q_pos against a cache whose keys are already rotated
    (§4.2);
  - relu_attention (§3.1 names it without a definition; this build's reading): weights
    max(s, 0) / N over the allowed keys, N the number of keys, O = sum of weight * v, no LSE.

A mask is described by a plain dict: {"mask": "full" | "causal" | "window" | "block_sparse",
"causal": bool, "window": W, "block": blk, "row_ptr": [...], "col_idx": [...], "bias":
"none" | "alibi" | "additive", "slopes": [...], "add_bias": array broadcastable to
[B, Hq, N, N], "norm": "softmax" | "relu"}.
"""
import math

import numpy as np


def _angles(p, d, theta):
    return [p * theta ** (-2.0 * i / d) for i in range(d // 2)]


def rotate(x, p, theta, inverse=False):
    """R_p x (or R_p^T x) of one vector x (a list of d floats)."""
    d = len(x)
    h = d // 2
    y = list(x)
    for i, a in enumerate(_angles(p, d, theta)):
        c, s = math.cos(a), math.sin(a)
        if inverse:
            s = -s
        y[i] = x[i] * c - x[i + h] * s
        y[i + h] = x[i + h] * c + x[i] * s
    return y


def _allowed(m, n, spec):
    kind = spec["mask"]
    if kind == "full":
        ok = True
    elif kind == "causal":
        return n <= m
    elif kind == "window":
        ok = abs(m - n) < spec["window"]
    elif kind == "block_sparse":
        blk = spec["block"]
        rp, ci = spec["row_ptr"], spec["col_idx"]
        r = m // blk
        ok = (n // blk) in ci[rp[r]:rp[r + 1]]
    else:
        raise ValueError(kind)
    if spec.get("causal", False):
        ok = ok and n <= m
    return ok


def _bias(b, h, m, n, spec, add_bias):
    kind = spec.get("bias", "none")
    if kind == "alibi":
        return spec["slopes"][h] * (n - m)
    if kind == "additive":
        return float(add_bias[b, h, m, n])
    return 0.0


def _dot(a, b):
    return math.fsum(x * y for x, y in zip(a, b))


def _prepare(q, k, scale, theta, rope_on, spec):
    """Rotated rows, the allowed-key lists and the scores of every (b, h, m)."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    add_bias = None
    if spec.get("bias") == "additive":
        add_bias = np.broadcast_to(np.asarray(spec["add_bias"], np.float64), (B, Hq, N, N))
    qr = [[[rotate(list(q[b, h, m]), m, theta) if rope_on else list(q[b, h, m])
            for m in range(N)] for h in range(Hq)] for b in range(B)]
    kr = [[[rotate(list(k[b, j, n]), n, theta) if rope_on else list(k[b, j, n])
            for n in range(N)] for j in range(Hkv)] for b in range(B)]
    rows = {}
    for b in range(B):
        for h in range(Hq):
            for m in range(N):
                keys = [n for n in range(N) if _allowed(m, n, spec)]
                s = [scale * _dot(qr[b][h][m], kr[b][h // g][n]) + _bias(b, h, m, n, spec, add_bias)
                     for n in keys]
                rows[b, h, m] = (keys, s)
    return qr, kr, rows


def _softmax(s):
    """(P, LSE) of one row of scores over its allowed keys."""
    if not s:
        return [], -math.inf
    mx = max(s)
    lse = mx + math.log(math.fsum(math.exp(x - mx) for x in s))
    return [math.exp(x - lse) for x in s], lse


def forward(q, k, v, scale, theta, rope_on, spec):
    """O [B, Hq, N, d] and LSE [B, Hq, N]."""
    q, k, v = (np.asarray(a, np.float64) for a in (q, k, v))
    B, Hq, N, d = q.shape
    g = Hq // k.shape[1]
    _, _, rows = _prepare(q, k, scale, theta, rope_on, spec)
    out = np.zeros((B, Hq, N, d))
    lse = np.zeros((B, Hq, N))
    relu = spec.get("norm", "softmax") == "relu"
    for (b, h, m), (keys, s) in rows.items():
        if relu:
            p, lse[b, h, m] = [max(x, 0.0) / N for x in s], math.nan
        else:
            p, lse[b, h, m] = _softmax(s)
        for c in range(d):
            out[b, h, m, c] = math.fsum(pi * v[b, h // g, n, c] for pi, n in zip(p, keys))
    return out, lse


def backward(q, k, v, dout, scale, theta, rope_on, spec):
    """(dQ, dK, dV, dBias) with dBias [B, Hq, N, N] = dS (zero where not allowed)."""
    q, k, v, dout = (np.asarray(a, np.float64) for a in (q, k, v, dout))
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    qr, kr, rows = _prepare(q, k, scale, theta, rope_on, spec)
    out, _ = forward(q, k, v, scale, theta, rope_on, spec)
    dbias = np.zeros((B, Hq, N, N))
    dq = np.zeros_like(q)
    # per (b, kv head, key n): the terms of dK' and dV, summed once over (h, m) with fsum
    dk_terms = {}
    dv_terms = {}
    for (b, h, m), (keys, s) in rows.items():
        p, _ = _softmax(s)
        D = _dot(dout[b, h, m], out[b, h, m])
        dq_terms = [[] for _ in range(d)]
        for pi, n in zip(p, keys):
            dP = _dot(dout[b, h, m], v[b, h // g, n])
            dS = pi * (dP - D)
            dbias[b, h, m, n] = dS
            for c in range(d):
                dq_terms[c].append(scale * dS * kr[b][h // g][n][c])
                dk_terms.setdefault((b, h // g, n, c), []).append(scale * dS * qr[b][h][m][c])
                dv_terms.setdefault((b, h // g, n, c), []).append(pi * dout[b, h, m, c])
        dqr = [math.fsum(t) for t in dq_terms]
        dq[b, h, m] = rotate(dqr, m, theta, inverse=True) if rope_on else dqr
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for j in range(Hkv):
            for n in range(N):
                dkr = [math.fsum(dk_terms.get((b, j, n, c), [])) for c in range(d)]
                dk[b, j, n] = rotate(dkr, n, theta, inverse=True) if rope_on else dkr
                for c in range(d):
                    dv[b, j, n, c] = math.fsum(dv_terms.get((b, j, n, c), []))
    return dq, dk, dv, dbias


def decode(q, kc, vc, q_pos, scale, theta, rope_q=True):
    """One query row per (b, h) at position q_pos; keys of the cache are used as stored."""
    q, kc, vc = (np.asarray(a, np.float64) for a in (q, kc, vc))
    B, Hq, d = q.shape
    Hkv, L = kc.shape[1], kc.shape[2]
    g = Hq // Hkv
    out = np.zeros((B, Hq, d))
    lse = np.zeros((B, Hq))
    for b in range(B):
        for h in range(Hq):
            qr = rotate(list(q[b, h]), q_pos, theta) if rope_q else list(q[b, h])
            s = [scale * _dot(qr, kc[b, h // g, n]) for n in range(L)]
            p, lse[b, h] = _softmax(s)
            for c in range(d):
                out[b, h, c] = math.fsum(pi * vc[b, h // g, n, c] for n, pi in enumerate(p))
    return out, lse
