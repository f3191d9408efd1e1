"""attnfuse_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (a runtime whose device memory is fully pre-reserved by its own allocator, a host
without an allocator to hand out scratch, a path where a cudaMalloc is not allowed) get the
split-KV partials in a fixed array inside the library. This file is collected last so that a
run stopping at its first failure has already run every other test; it passes both alone in a
fresh process and after the other tests.
"""
import ctypes

import pytest
import torch

import attention_attn_fwd_bwd_gb300 as af
import oracle
from attention_attn_fwd_bwd_gb300 import inputs
from tests._helpers import check_lse, check_out, f64

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def _noalloc(q, kc, vc, q_pos, theta, splits, out=None, lse=None):
    """Call the C entry point directly with raw pointers; returns (status, out, lse)."""
    lib = af.load()
    B, Hq, d = q.shape
    Hkv, L = kc.shape[1], kc.shape[2]
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
    st = lambda t, n: (ctypes.c_int64 * n)(*t.stride())
    rc = lib.attnfuse_decode_noalloc(
        ctypes.c_void_p(q.data_ptr()), st(q, 3), ctypes.c_void_p(kc.data_ptr()), st(kc, 4),
        ctypes.c_void_p(vc.data_ptr()), st(vc, 4), ctypes.c_void_p(out.data_ptr()), st(out, 3),
        ctypes.c_void_p(lse.data_ptr()), B, Hq, Hkv, L, d, q_pos, d ** -0.5, theta,
        af.ROPE_FUSED, splits, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, out, lse


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from attention_attn_fwd_bwd_gb300 import _build

    _build.build()
    af.load()


def test_noalloc_decode_matches_workspace_decode_twice():
    dev = torch.device("cuda")
    # two different problems in a row: the shared scratch keeps the first call's contents
    for seed, (B, Hq, Hkv, L, splits) in ((61, (2, 16, 2, 3000, 0)), (62, (1, 64, 8, 32768, 19))):
        x = inputs.decode(B, Hq, Hkv, L, 128, seed)
        q, kc, vc = (x[n].to(dev) for n in ("q", "k_cache", "v_cache"))
        ref_o, ref_l = af.decode(q, kc, vc, L - 1, rope_theta=5e5, num_splits=splits)
        rc, out, lse = _noalloc(q, kc, vc, L - 1, 5e5, splits)
        torch.cuda.synchronize()
        assert rc == 0, af.load().attnfuse_last_error().decode()
        assert af.device_status() == 0
        check_out(out.cpu(), ref_o.cpu())
        check_lse(lse.cpu(), ref_l.cpu())
        # and against the fp64 oracle on the same inputs
        oo, ol = oracle.decode(f64(x["q"]), f64(x["k_cache"]), f64(x["v_cache"]), L - 1,
                               128 ** -0.5, 5e5, True)
        check_out(out.cpu(), oo)
        check_lse(lse.cpu(), ol)


def test_noalloc_decode_allocates_no_device_memory():
    """After the first call on a device (which looks up the array's address), calls change
    neither torch's allocator statistics nor the device's free memory."""
    dev = torch.device("cuda")
    B, Hq, Hkv, L = 1, 64, 8, 32768
    x = inputs.decode(B, Hq, Hkv, L, 128, 64)
    q, kc, vc = (x[n].to(dev) for n in ("q", "k_cache", "v_cache"))
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    rc, _, _ = _noalloc(q, kc, vc, L - 1, 5e5, 0, out, lse)  # set-up call
    torch.cuda.synchronize()
    assert rc == 0, af.load().attnfuse_last_error().decode()
    alloc0, free0 = torch.cuda.memory_allocated(dev), torch.cuda.mem_get_info(dev)[0]
    for _ in range(2):
        rc, _, _ = _noalloc(q, kc, vc, L - 1, 5e5, 0, out, lse)
        assert rc == 0, af.load().attnfuse_last_error().decode()
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated(dev) == alloc0
    assert torch.cuda.mem_get_info(dev)[0] == free0
    assert af.device_status() == 0


def test_noalloc_decode_rejects_too_large():
    dev = torch.device("cuda")
    x = inputs.decode(8, 64, 8, 4096, 128, 63)
    q, kc, vc = (x[n].to(dev) for n in ("q", "k_cache", "v_cache"))
    rc, _, _ = _noalloc(q, kc, vc, 4095, 5e5, 32)  # 8*64*32 rows of partials: 17 MB > 4 MiB
    assert rc == 3  # ATTNFUSE_ERR_WORKSPACE_TOO_SMALL
    assert b"4194304" in af.load().attnfuse_last_error()
