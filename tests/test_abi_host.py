"""C-ABI boundary checks that need no GPU: every symbol declared in include/attnfuse.h is
exported by libattnfuse.so, and argument validation returns the documented status codes
before any CUDA call is made. No compute is launched."""
import ctypes
import os
import re

import pytest

import attention_attn_fwd_bwd_gb300 as af

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, WS_SMALL = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    from attention_attn_fwd_bwd_gb300 import _build

    _build.build()
    return af.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "attnfuse.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attnfuse_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n


def _st(*v):
    return (ctypes.c_int64 * len(v))(*v)


FAKE = ctypes.c_void_p(0x100000)  # 16-byte aligned, never dereferenced on these paths
STR = _st(4 * 1024 * 128, 1024 * 128, 128, 1)


def _fwd(lib, q=FAKE, qs=STR, B=1, Hq=4, Hkv=4, N=1024, d=128, scale=0.1, mode=1, var=None,
         ws=FAKE, ws_bytes=1 << 30):
    return lib.attnfuse_fwd(q, qs, FAKE, STR, FAKE, STR, FAKE, STR, None, B, Hq, Hkv, N, d, scale,
                            1e4, mode, var, ws, ws_bytes, None)


def test_fwd_validation(lib):
    assert _fwd(lib, d=96) == UNSUPPORTED
    assert _fwd(lib, Hq=6, Hkv=4) == UNSUPPORTED
    assert _fwd(lib, q=None) == INVALID
    assert b"q is NULL" in lib.attnfuse_last_error()
    assert _fwd(lib, q=ctypes.c_void_p(0x100001)) == INVALID
    assert _fwd(lib, qs=_st(4 * 1024 * 128, 1024 * 128, 128, 2)) == INVALID
    assert _fwd(lib, qs=_st(4 * 1024 * 128, 1024 * 128, 130, 1)) == INVALID
    assert _fwd(lib, scale=0.0) == INVALID
    assert _fwd(lib, mode=7) == INVALID
    assert _fwd(lib, ws=None, ws_bytes=0) == WS_SMALL
    assert _fwd(lib, ws_bytes=1024) == WS_SMALL
    v = af.CVariant()
    v.mask = 3
    v.bs_block = 64
    assert _fwd(lib, var=ctypes.byref(v)) == INVALID  # CSR pointers missing
    v.bs_block = 32
    assert _fwd(lib, var=ctypes.byref(v)) == UNSUPPORTED
    v = af.CVariant()
    v.mask = 2
    v.window = 0
    assert _fwd(lib, var=ctypes.byref(v)) == INVALID
    v = af.CVariant()
    v.mask = 1
    v.bias = 1
    assert _fwd(lib, var=ctypes.byref(v)) == INVALID  # ALiBi slopes missing


def test_workspace_sizes(lib):
    n = ctypes.c_size_t()
    assert lib.attnfuse_fwd_workspace_size(4, 32, 8, 4096, 128, 0, ctypes.byref(n)) == OK
    assert n.value == 0
    assert lib.attnfuse_fwd_workspace_size(4, 32, 8, 4096, 128, 1, ctypes.byref(n)) == OK
    # (cos, sin) fp32 table, then (head dim 128) the rotated keys K' in fp16 and one flag per
    # 64-key block
    assert n.value == 4096 * 64 * 8 + 4 * 8 * 4096 * 128 * 2 + 4 * 8 * 64 * 4
    assert lib.attnfuse_fwd_workspace_size(4, 32, 8, 4096, 128, 2, ctypes.byref(n)) == OK
    assert n.value == 4096 * 64 * 8 + 4 * 32 * 4096 * 128 * 2 + 4 * 8 * 4096 * 128 * 2
    assert lib.attnfuse_fwd_workspace_size(1, 2, 2, 10, 64, 1, ctypes.byref(n)) == OK
    # the table always covers 128 positions; K' (10 x 64 fp16 per head, 256-byte aligned) and
    # one flag per 64 keys (256-byte aligned)
    assert n.value == 128 * 32 * 8 + 2 * 10 * 64 * 2 + 256
    # e4m3 forward: the widened V (bf16)
    assert lib.attnfuse_fwd_fp8_workspace_size(4, 32, 8, 4096, 128, ctypes.byref(n)) == OK
    assert n.value == 4 * 8 * 4096 * 128 * 2
    assert lib.attnfuse_fwd_fp8_workspace_size(4, 32, 8, 4096, 64, ctypes.byref(n)) == UNSUPPORTED
    assert lib.attnfuse_bwd_workspace_size(8, 32, 8, 2048, 128, 1, ctypes.byref(n)) == OK
    assert n.value == 2048 * 64 * 8 + 8 * 32 * 2048 * 4
    assert lib.attnfuse_decode_workspace_size(1, 64, 8, 32768, 128, 8, ctypes.byref(n)) == OK
    assert n.value == 64 * 8 * 128 * 4 + 2 * 2048  # acc + (max, sum), 256-byte aligned


def test_decode_and_bwd_validation(lib):
    q_st, c_st, o_st = _st(64 * 128, 128, 1), _st(8 * 32768 * 128, 32768 * 128, 128, 1), _st(64 * 128, 128, 1)
    args = lambda Hq, Hkv, mode, ws_bytes: lib.attnfuse_decode(
        FAKE, q_st, FAKE, c_st, FAKE, c_st, FAKE, o_st, None, 1, Hq, Hkv, 32768, 128, 32767,
        0.088, 5e5, mode, 8, FAKE, ws_bytes, None)
    assert args(64, 1, 1, 1 << 30) == UNSUPPORTED  # g = 64 > 32
    assert args(64, 8, 2, 1 << 30) == UNSUPPORTED  # decode rotates q only
    assert args(64, 8, 1, 100) == WS_SMALL
    rc = lib.attnfuse_decode_noalloc(FAKE, q_st, FAKE, c_st, FAKE, c_st, FAKE, o_st, None, 8, 64, 8,
                                     32768, 128, 32767, 0.088, 5e5, 1, 128, None)
    assert rc == WS_SMALL and b"4194304" in lib.attnfuse_last_error()
    s = STR
    bwd = lambda v: lib.attnfuse_bwd(FAKE, s, FAKE, s, FAKE, s, FAKE, s, FAKE, FAKE, s, FAKE, s,
                                     FAKE, s, FAKE, s, 1, 4, 4, 1024, 128, 0.1, 1e4, 1,
                                     ctypes.byref(v), FAKE, 1 << 30, None)
    v = af.CVariant()
    v.mask = 2
    v.window = 16
    v.dbias = FAKE
    v.dbias_strides[:] = [4 * 1024 * 1024, 1024 * 1024, 1024, 1]
    assert bwd(v) == INVALID  # dbias without an additive bias
    v.bias = 2
    v.add_bias = FAKE
    v.dbias_strides[:] = [4 * 1024 * 1024, 1024 * 1024, -1024, 1]
    assert bwd(v) == INVALID  # negative dbias stride
    v.dbias_strides[:] = [4 * 1024 * 1024, 1024 * 1024, 1024, 2]
    assert bwd(v) == INVALID  # dbias key stride must be 1
    v.bs_block, v.mask = 96, 3
    assert bwd(v) == UNSUPPORTED  # block edge


def test_version(lib):
    assert lib.attnfuse_version() >= 100


def test_rope_entry_points_validation(lib):
    x_st = _st(4 * 1024 * 64, 1024 * 64, 64, 1)
    pre = lambda x=FAKE, out=FAKE, d=64, theta=1e4, ws=FAKE, ws_bytes=1 << 20: \
        lib.attnfuse_rope_prerotate(x, x_st, out, 1, 4, 1024, d, theta, ws, ws_bytes, None)
    assert pre(d=96) == UNSUPPORTED
    assert pre(x=None) == INVALID
    assert pre(out=ctypes.c_void_p(0x100008)) == INVALID  # output must be 16-byte aligned
    assert pre(theta=0.0) == INVALID
    assert pre(ws_bytes=1024) == WS_SMALL  # the (cos, sin) table of 1024 x 32 pairs
    table = lambda t=FAKE, nbytes=1 << 20, N=1024, d=64, theta=1e4: \
        lib.attnfuse_rope_table(t, nbytes, N, d, theta, None)
    assert table(N=0) == UNSUPPORTED
    assert table(d=32) == UNSUPPORTED
    assert table(theta=-1.0) == INVALID
    assert table(t=None) == WS_SMALL
    assert table(nbytes=1024 * 32 * 8 - 1) == WS_SMALL


def test_rope_auto_mode_rule(lib):
    m = ctypes.c_int()
    auto = lambda N, d, bwd: (lib.attnfuse_rope_auto_mode(N, d, bwd, ctypes.byref(m)), m.value)
    FUSED, PRE = af.ROPE_FUSED, af.ROPE_PREROTATE
    # head dim 128: fusion wins for the forward below the measured crossover (14900); the
    # backward pre-rotates at every N
    assert auto(256, 128, 0) == (OK, FUSED) and auto(14899, 128, 0) == (OK, FUSED)
    assert auto(14900, 128, 0) == (OK, PRE) and auto(256, 128, 1) == (OK, PRE)
    # head dim 64: fusion wins below the measured crossovers (forward 1850, backward 258)
    assert auto(1849, 64, 0) == (OK, FUSED) and auto(1850, 64, 0) == (OK, PRE)
    assert auto(257, 64, 1) == (OK, FUSED) and auto(258, 64, 1) == (OK, PRE)
    assert lib.attnfuse_rope_auto_mode(0, 64, 0, ctypes.byref(m)) == INVALID
    assert lib.attnfuse_rope_auto_mode(512, 80, 0, ctypes.byref(m)) == UNSUPPORTED
    assert lib.attnfuse_rope_auto_mode(512, 64, 0, None) == INVALID
    n = ctypes.c_int()
    assert lib.attnfuse_decode_auto_splits(0, 8, 32768, ctypes.byref(n)) == INVALID
    assert lib.attnfuse_decode_auto_splits(1, 8, 32768, None) == INVALID
