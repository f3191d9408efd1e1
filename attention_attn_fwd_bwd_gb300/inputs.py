"""Seeded synthetic workloads shared by the tests, the oracle checks and the benchmark.

This module only draws data; it holds none of the attention arithmetic. Recipe:
``torch.Generator('cpu').manual_seed(seed)``, ``torch.randn`` in fp32, round to bf16 (RNE).
Prefill draw order is Q, K, V, dO; decode draw order is q, K cache, V cache. The decode
K cache is drawn i.i.d. N(0, 1) and treated as already rotated: a rotation maps an isotropic
Gaussian vector to an isotropic Gaussian vector, so the drawn cache has exactly the
distribution of a rotated one.

The block-sparse layout is the BigBird pattern (AttnFuse paper §4.3 evaluates on it): for
block row i of Nb blocks, the window blocks {i-1, i, i+1}, global block columns {0, 1} for
every row, global block rows {0, 1} that see every column, plus ``n_random`` random columns
per row drawn without replacement from those not yet active (numpy PCG64, rows in order).
"""
from __future__ import annotations

import numpy as np
import torch


def randn_bf16(shape, gen: torch.Generator) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def prefill(B, Hq, Hkv, N, d, seed, with_dout=False):
    """bf16 CPU tensors q [B,Hq,N,d], k, v [B,Hkv,N,d] (and dout [B,Hq,N,d])."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    out = {
        "q": randn_bf16((B, Hq, N, d), g),
        "k": randn_bf16((B, Hkv, N, d), g),
        "v": randn_bf16((B, Hkv, N, d), g),
    }
    if with_dout:
        out["dout"] = randn_bf16((B, Hq, N, d), g)
    return out


def prefill_e4m3(B, Hq, Hkv, N, d, seed):
    """e4m3 inputs for the fp8 forward: q, k, v are drawn exactly as in ``prefill`` (fp32
    N(0, 1), same generator order), each scaled so that its largest magnitude maps to 448 (the
    largest finite e4m3 value) and rounded to e4m3 by torch's float8_e4m3fn conversion.
    Returns raw bytes as torch.uint8 CPU tensors under "q", "k", "v" and the per-tensor
    dequantisation scales (python floats) under "q_scale", "k_scale", "v_scale": the intended
    value of a byte x is scale * e4m3(x)."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    out = {}
    for name, shape in (("q", (B, Hq, N, d)), ("k", (B, Hkv, N, d)), ("v", (B, Hkv, N, d))):
        x = torch.randn(*shape, generator=g, dtype=torch.float32)
        amax = float(x.abs().max()) if x.numel() else 1.0
        sc = float(np.float32(max(amax, 1e-6) / 448.0))
        out[name] = (x / sc).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        out[name + "_scale"] = sc
    return out


def decode(B, Hq, Hkv, L, d, seed):
    """bf16 CPU tensors q [B,Hq,d], k_cache, v_cache [B,Hkv,L,d]."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    return {
        "q": randn_bf16((B, Hq, d), g),
        "k_cache": randn_bf16((B, Hkv, L, d), g),
        "v_cache": randn_bf16((B, Hkv, L, d), g),
    }


def alibi_slopes(H):
    """Per-head ALiBi slopes 2^(-8 (h+1) / H), h = 0..H-1 (geometric sequence of Press et al.)."""
    return np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], dtype=np.float64)


def bigbird_csr(Nb, seed, n_window=3, n_global=2, n_random=3):
    """CSR (row_ptr [Nb+1], col_idx) int32 of a BigBird block layout over Nb x Nb blocks."""
    rng = np.random.Generator(np.random.PCG64(int(seed)))
    half = n_window // 2
    rows = []
    for i in range(Nb):
        if i < n_global:
            active = set(range(Nb))
        else:
            active = {j for j in range(i - half, i + half + 1) if 0 <= j < Nb}
            active |= set(range(min(n_global, Nb)))
            free = np.array(sorted(set(range(Nb)) - active), dtype=np.int64)
            if free.size:
                pick = rng.choice(free, size=min(n_random, free.size), replace=False)
                active |= {int(x) for x in pick}
        rows.append(sorted(active))
    row_ptr = np.zeros(Nb + 1, np.int32)
    for i, r in enumerate(rows):
        row_ptr[i + 1] = row_ptr[i] + len(r)
    col_idx = np.array([c for r in rows for c in r], np.int32)
    return row_ptr, col_idx


def sample_rows(B, H, N, count, seed, always=()):
    """int64 [count, 3] of (b, h, m): a seeded sample of query rows, plus the given rows."""
    rng = np.random.Generator(np.random.PCG64(int(seed)))
    rows = [tuple(r) for r in always]
    while len(rows) < count:
        rows.append((int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(N))))
    return np.array(rows[:max(count, len(always))], np.int64)
