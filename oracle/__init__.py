"""fp64 CPU oracle for the fused RoPE + variant attention path — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import
this package. It wraps ``attn_oracle.c`` (plain loops, OpenMP over heads) through ctypes and
shares nothing with the CUDA library. Every function takes and returns numpy float64 arrays in
contiguous [B, H, N, d] layout; bf16 inputs are widened exactly before they reach it.

What each function computes, with the passage of the AttnFuse paper it follows, is documented
in ``attn_oracle.c``.

Parity status: every function here is pinned by ``tests/test_oracle_*.py`` (closed forms,
invariants, brute force on tiny inputs, an independent library routine and finite differences).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liborc.so")
_lock = threading.Lock()
_lib = None

MASK_FULL, MASK_CAUSAL, MASK_WINDOW, MASK_BLOCK_SPARSE = 0, 1, 2, 3
BIAS_NONE, BIAS_ALIBI, BIAS_ADDITIVE = 0, 1, 2
NORM_SOFTMAX, NORM_RELU = 0, 1


def build(force: bool = False) -> str:
    """Compile attn_oracle.c with gcc (-O2, OpenMP) into oracle/_build/liborc.so."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Variant(ctypes.Structure):
    _fields_ = [
        ("mask", ctypes.c_int32),
        ("causal", ctypes.c_int32),
        ("window", ctypes.c_int32),
        ("bs_block", ctypes.c_int32),
        ("bs_row_ptr", ctypes.c_void_p),
        ("bs_col_idx", ctypes.c_void_p),
        ("bias", ctypes.c_int32),
        ("norm", ctypes.c_int32),
        ("slopes", ctypes.c_void_p),
        ("add_bias", ctypes.c_void_p),
        ("add_bias_strides", ctypes.c_int64 * 4),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I, I64, D = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            VP = ctypes.POINTER(_Variant)
            lib.orc_rope.argtypes = [P, P, I64, I, P, D, I]
            lib.orc_fwd.argtypes = [P, P, P, I, I, I, I64, I, D, D, I, VP, P, P]
            lib.orc_fwd_rows.argtypes = [P, P, P, I, I, I, I64, I, D, D, I, VP, I64, P, P, P]
            lib.orc_bwd.argtypes = [P, P, P, P, I, I, I, I64, I, D, D, I, VP, I64, P, P, P, P, P, P, P]
            lib.orc_bwd_dq_rows.argtypes = [P, P, P, P, I, I, I, I64, I, D, D, I, VP, I64, P, P]
            lib.orc_decode.argtypes = [P, P, P, I, I, I, I64, I, I64, D, D, I, P, P]
            lib.orc_tile_visits.argtypes = [I64, I, I, VP, P]
            lib.orc_allowed_pairs.argtypes = [I64, VP]
            lib.orc_allowed_pairs.restype = I64
            for f in ("orc_rope", "orc_fwd", "orc_fwd_rows", "orc_bwd", "orc_bwd_dq_rows",
                      "orc_decode", "orc_tile_visits"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


class Variant:
    """Combinator set (paper §3.1): a mask kind plus an optional bias, as plain data.

    mask: MASK_FULL / MASK_CAUSAL / MASK_WINDOW / MASK_BLOCK_SPARSE; causal: extra n <= m;
    window: W; bs_row_ptr / bs_col_idx: CSR of active blocks (block edge bs_block);
    bias: BIAS_NONE / BIAS_ALIBI (slopes, one per query head) / BIAS_ADDITIVE (add_bias,
    any array broadcastable to [B, Hq, N, N]); norm: NORM_SOFTMAX or NORM_RELU (relu_attention,
    O_m = (1/N) sum_n max(s_mn, 0) v_n over the allowed keys; forward only, LSE is NaN).
    """

    def __init__(self, mask=MASK_CAUSAL, causal=False, window=0, bs_block=64, bs_row_ptr=None,
                 bs_col_idx=None, bias=BIAS_NONE, slopes=None, add_bias=None, norm=0):
        self.norm = norm
        self.mask, self.causal, self.window, self.bs_block = mask, bool(causal), window, bs_block
        self.bs_row_ptr = None if bs_row_ptr is None else np.ascontiguousarray(bs_row_ptr, np.int32)
        self.bs_col_idx = None if bs_col_idx is None else np.ascontiguousarray(bs_col_idx, np.int32)
        self.bias = bias
        self.slopes = None if slopes is None else np.ascontiguousarray(slopes, np.float64)
        self.add_bias = None if add_bias is None else np.asarray(add_bias, np.float64)

    def _c(self, shape4=None):
        v = _Variant()
        v.mask, v.causal, v.window, v.bs_block = self.mask, int(self.causal), self.window, self.bs_block
        keep = []
        if self.mask == MASK_BLOCK_SPARSE:
            v.bs_row_ptr = self.bs_row_ptr.ctypes.data
            v.bs_col_idx = self.bs_col_idx.ctypes.data
        v.bias = self.bias
        v.norm = self.norm
        if self.bias == BIAS_ALIBI:
            v.slopes = self.slopes.ctypes.data
        if self.bias == BIAS_ADDITIVE:
            ab = self.add_bias
            while ab.ndim < 4:
                ab = ab[None]
            if shape4 is not None:
                ab = np.broadcast_to(ab, shape4)
            keep.append(ab)
            v.add_bias = ab.ctypes.data
            for i in range(4):
                v.add_bias_strides[i] = ab.strides[i] // 8
        return v, keep


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return a.ctypes.data if a is not None else None


def rope(x, pos, theta, inverse=False):
    """Rotate rows of x [..., d] (row r at position pos[r]) by RoPE; inverse: R^T."""
    x = _f64(x)
    d = x.shape[-1]
    rows = x.size // d
    pos = _f64(np.broadcast_to(np.asarray(pos, np.float64), (rows,)))
    y = np.empty_like(x)
    rc = _load().orc_rope(x.ctypes.data, y.ctypes.data, rows, d, pos.ctypes.data, float(theta),
                          int(inverse))
    if rc:
        raise ValueError("orc_rope failed")
    return y


def forward(q, k, v, scale, theta, rope_on, variant: Variant):
    """O [B,Hq,N,d] and LSE [B,Hq,N] for the whole problem."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    out = np.zeros_like(q)
    lse = np.zeros((B, Hq, N))
    cv, keep = variant._c((B, Hq, N, N))
    rc = _load().orc_fwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, B, Hq, Hkv, N, d,
                         float(scale), float(theta), int(rope_on), ctypes.byref(cv),
                         out.ctypes.data, lse.ctypes.data)
    if rc:
        raise RuntimeError(f"orc_fwd failed ({rc})")
    return out, lse


def forward_rows(q, k, v, scale, theta, rope_on, variant: Variant, rows):
    """O and LSE of selected rows; rows: int array [R, 3] of (b, h, m)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    rows = np.ascontiguousarray(rows, np.int64).reshape(-1, 3)
    out = np.zeros((rows.shape[0], d))
    lse = np.zeros(rows.shape[0])
    cv, keep = variant._c((B, Hq, N, N))
    rc = _load().orc_fwd_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, B, Hq, Hkv, N, d,
                              float(scale), float(theta), int(rope_on), ctypes.byref(cv),
                              rows.shape[0], rows.ctypes.data, out.ctypes.data, lse.ctypes.data)
    if rc:
        raise RuntimeError(f"orc_fwd_rows failed ({rc})")
    return out, lse


def backward(q, k, v, dout, scale, theta, rope_on, variant: Variant, groups=None,
             with_dbias=False):
    """(O, LSE, dQ, dK, dV), plus dBias [B, Hq, N, N] (the gradient with respect to an additive
    bias, before any broadcast is summed out) when with_dbias. groups: optional [G, 2] list of
    (b, kv_head) to compute."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    out = np.zeros_like(q)
    lse = np.zeros((B, Hq, N))
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dbias = np.zeros((B, Hq, N, N)) if with_dbias else None
    g = None
    if groups is not None:
        g = np.ascontiguousarray(groups, np.int64).reshape(-1, 2)
    cv, keep = variant._c((B, Hq, N, N))
    rc = _load().orc_bwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, B, Hq,
                         Hkv, N, d, float(scale), float(theta), int(rope_on), ctypes.byref(cv),
                         0 if g is None else g.shape[0], _ptr(g), out.ctypes.data,
                         lse.ctypes.data, dq.ctypes.data, dk.ctypes.data, dv.ctypes.data,
                         _ptr(dbias))
    if rc:
        raise RuntimeError(f"orc_bwd failed ({rc})")
    if with_dbias:
        return out, lse, dq, dk, dv, dbias
    return out, lse, dq, dk, dv


def backward_dq_rows(q, k, v, dout, scale, theta, rope_on, variant: Variant, rows):
    """dQ of selected rows; rows: [R, 3] of (b, h, m)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    rows = np.ascontiguousarray(rows, np.int64).reshape(-1, 3)
    dq = np.zeros((rows.shape[0], d))
    cv, keep = variant._c((B, Hq, N, N))
    rc = _load().orc_bwd_dq_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data,
                                 B, Hq, Hkv, N, d, float(scale), float(theta), int(rope_on),
                                 ctypes.byref(cv), rows.shape[0], rows.ctypes.data,
                                 dq.ctypes.data)
    if rc:
        raise RuntimeError(f"orc_bwd_dq_rows failed ({rc})")
    return dq


def decode(q, kc, vc, q_pos, scale, theta, rope_q=True):
    """Decode step: q [B,Hq,d], caches [B,Hkv,L,d] (keys already rotated) -> (O, LSE)."""
    q, kc, vc = _f64(q), _f64(kc), _f64(vc)
    B, Hq, d = q.shape
    Hkv, L = kc.shape[1], kc.shape[2]
    out = np.zeros_like(q)
    lse = np.zeros((B, Hq))
    rc = _load().orc_decode(q.ctypes.data, kc.ctypes.data, vc.ctypes.data, B, Hq, Hkv, L, d,
                            int(q_pos), float(scale), float(theta), int(rope_q),
                            out.ctypes.data, lse.ctypes.data)
    if rc:
        raise RuntimeError(f"orc_decode failed ({rc})")
    return out, lse


def decode_e4m3(x):
    """Values of e4m3 bytes (the fp8 forward's operand format) as float64, from the OCP 8-bit
    floating-point definition of E4M3: byte s eeee mmm encodes (-1)^s 2^(e-7) (1 + m/8) for
    e > 0 and (-1)^s 2^(-6) (m/8) for e = 0 (subnormals); eeee mmm = 1111 111 is NaN and there
    are no infinities. The pages name fp8 attention as future work without fixing a format;
    E4M3 is the plainest reading (the tensor cores' fp8 operand format with the wider range
    of mantissa). x: any integer array of bytes (0..255)."""
    b = np.asarray(x).astype(np.int64) & 0xFF
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    mag = np.where(e > 0, np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64)), np.ldexp(m / 8.0, -6))
    out = sign * mag
    return np.where((b & 0x7F) == 0x7F, np.nan, out)


def tile_visits(N, BM, BN, variant: Variant):
    """uint8 [ceil(N/BM), ceil(N/BN)]: 1 where the tile holds at least one allowed pair."""
    TQ, TK = -(-N // BM), -(-N // BN)
    out = np.zeros((TQ, TK), np.uint8)
    cv, keep = variant._c()
    rc = _load().orc_tile_visits(N, BM, BN, ctypes.byref(cv), out.ctypes.data)
    if rc:
        raise RuntimeError("orc_tile_visits failed")
    return out


def allowed_pairs(N, variant: Variant) -> int:
    """Number of allowed (m, n) pairs of one head."""
    cv, keep = variant._c()
    return int(_load().orc_allowed_pairs(N, ctypes.byref(cv)))
