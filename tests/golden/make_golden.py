"""Write the golden fixtures of this directory from the fp64 oracle.

The AttnFuse pages print no worked numeric example, so the stored expected values come from the
oracle (oracle/, which this script alone calls) on small bf16-exact inputs drawn here with
numpy's PCG64. Each fixture names the passages that define what it holds. The fixtures pin the
oracle against silent change (tests/test_oracle_golden.py re-derives them with the oracle and,
independently, with the brute-force restatement in tests/_bruteforce.py), and the CUDA library
is checked against them on a GPU (tests/test_gpu_golden.py).

Run from the repository root: python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402


def bf16_exact(x):
    """Round float64 values to the nearest bf16 (ties to even), returned as float64."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def draw(seed, *shapes):
    rng = np.random.Generator(np.random.PCG64(seed))
    return [bf16_exact(rng.standard_normal(s)) for s in shapes]


def write(name, header, params, arrays):
    path = os.path.join(HERE, name)
    with open(path, "w") as f:
        for line in header:
            f.write(f"# {line}\n")
        f.write("# written by tests/golden/make_golden.py from the fp64 oracle; inputs are bf16-exact\n")
        f.write("%params " + json.dumps(params, sort_keys=True) + "\n")
        for key, a in arrays:
            a = np.asarray(a, np.float64)
            f.write(f"@{key} " + " ".join(str(n) for n in a.shape) + "\n")
            flat = [repr(float(x)) for x in a.ravel()]
            for i in range(0, len(flat), 8):
                f.write(" ".join(flat[i:i + 8]) + "\n")
    print("wrote", path)


def main():
    # 1. forward: RoPE + causal, GQA group of 2
    B, Hq, Hkv, N, d, theta, scale = 1, 2, 1, 5, 64, 1e4, 0.125
    q, k, v = draw(101, (B, Hq, N, d), (B, Hkv, N, d), (B, Hkv, N, d))
    o, lse = oracle.forward(q, k, v, scale, theta, True, oracle.Variant(mask=oracle.MASK_CAUSAL))
    write("fwd_rope_causal_d64.txt",
          ["Fused RoPE + causal attention forward: O and LSE.",
           "RoPE: NeoX half-split pairs, theta_i = theta^(-2i/d), position = token index (AttnFuse paper §4.1).",
           "Causal combinator: key n visible from query m iff n <= m (§3.1).",
           "Softmax attention O = softmax(scale Q'K'^T) V over the visible keys, LSE = max + ln(sum) (§2, §4.4).",
           "GQA: query head h reads key/value head h // (Hq / Hkv)."],
          dict(B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, theta=theta, scale=scale, mask="causal", rope=True),
          [("q", q), ("k", k), ("v", v), ("out", o), ("lse", lse)])

    # 2. forward + backward: RoPE + sliding window 3 (non-causal) + ALiBi
    B, Hq, Hkv, N, d, theta, scale, W = 1, 2, 1, 6, 64, 1e4, 0.125, 3
    slopes = [2.0 ** -4, 2.0 ** -8]  # 2^(-8 (h + 1) / Hq), exact in fp32
    q, k, v, do = draw(202, (B, Hq, N, d), (B, Hkv, N, d), (B, Hkv, N, d), (B, Hq, N, d))
    var = oracle.Variant(mask=oracle.MASK_WINDOW, window=W, bias=oracle.BIAS_ALIBI,
                         slopes=np.array(slopes))
    o, lse, dq, dk, dv = oracle.backward(q, k, v, do, scale, theta, True, var)
    write("bwd_rope_window_alibi_d64.txt",
          ["Fused RoPE + sliding window + ALiBi attention: forward (O, LSE) and backward (dQ, dK, dV).",
           "RoPE as in §4.1; gradients are taken with respect to the un-rotated q and k (dQ = R^T dQ').",
           "Sliding window combinator: key n visible from query m iff |m - n| < W (§3.1).",
           "ALiBi combinator: s += slope_h (n - m), applied after the scale (§3.1).",
           "Backward by direct differentiation: D = rowsum(dO O), dS = P (dP - D), dQ' = scale dS K',",
           "dK' = scale dS^T Q', dV = P^T dO, dK and dV summed over the query heads of a group (§4.4)."],
          dict(B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, theta=theta, scale=scale, mask="window", window=W,
               causal=False, bias="alibi", slopes=slopes, rope=True),
          [("q", q), ("k", k), ("v", v), ("dout", do), ("out", o), ("lse", lse), ("dq", dq),
           ("dk", dk), ("dv", dv)])

    # 3. decode: one query row at q_pos against a pre-rotated cache
    B, Hq, Hkv, L, d, theta, scale = 1, 2, 1, 7, 64, 5e5, 0.125
    q, kc, vc = draw(303, (B, Hq, d), (B, Hkv, L, d), (B, Hkv, L, d))
    o, lse = oracle.decode(q, kc, vc, L - 1, scale, theta, rope_q=True)
    write("decode_rope_d64.txt",
          ["Decode step: q rotated at q_pos, keys of the cache used as stored (already rotated) (§4.2).",
           "Every cached key 0..L-1 is visible; O and LSE as in the forward (§2, §4.4)."],
          dict(B=B, Hq=Hq, Hkv=Hkv, L=L, d=d, theta=theta, scale=scale, q_pos=L - 1, rope=True),
          [("q", q), ("k_cache", kc), ("v_cache", vc), ("out", o), ("lse", lse)])


if __name__ == "__main__":
    oracle.build()
    main()
