"""The Python binding rejects, before any launch, tensors that the C ABI cannot check through
a bare pointer: another element type, another rank or shape, a CPU tensor (its address would
reach a kernel), a block-sparse row_ptr shorter than the layout's block rows. No GPU needed:
every case here fails in the binding."""
import pytest
import torch

import attention_attn_fwd_bwd_gb300 as af

B, Hq, Hkv, N, d = 1, 4, 2, 200, 64


def _qkv(dtype=torch.bfloat16):
    return (torch.zeros(B, Hq, N, d, dtype=dtype), torch.zeros(B, Hkv, N, d, dtype=dtype),
            torch.zeros(B, Hkv, N, d, dtype=dtype))


def test_forward_rejects_wrong_dtype_rank_and_device():
    q, k, v = _qkv(torch.float32)
    with pytest.raises(TypeError, match="q: dtype"):
        af.fwd(q, k, v)
    q, k, v = _qkv()
    with pytest.raises(ValueError, match=r"expected \[B, Hq, N, d\]"):
        af.fwd(q[0], k, v)
    with pytest.raises(ValueError, match="q: on cpu"):
        af.fwd(q, k, v)


def test_backward_and_decode_reject_cpu_and_wrong_types():
    q, k, v = _qkv()
    lse = torch.zeros(B, Hq, N)
    with pytest.raises(ValueError, match="q: on cpu"):
        af.bwd(q, k, v, q, lse, q)
    with pytest.raises(TypeError, match="q: dtype"):
        af.bwd(q.float(), k, v, q, lse, q)
    qd = torch.zeros(B, Hq, d, dtype=torch.bfloat16)
    cache = torch.zeros(B, Hkv, 64, d, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match=r"expected \[B, Hq, d\]"):
        af.decode(q, cache, cache, 63)
    with pytest.raises(ValueError, match="q: on cpu"):
        af.decode(qd, cache, cache, 63)
    with pytest.raises(TypeError, match="x: dtype"):
        af.rope_prerotate(q.half(), 1e4)


def test_variant_tensors_are_checked():
    dev = torch.device("cpu")
    v = af.Variant(mask=af.MASK_CAUSAL, bias=af.BIAS_ALIBI, alibi_slopes=torch.ones(Hq, dtype=torch.float64))
    with pytest.raises(TypeError, match="alibi_slopes: dtype"):
        v.check(dev, B, Hq, N)
    v = af.Variant(mask=af.MASK_BLOCK_SPARSE, bs_block=64,
                   bs_row_ptr=torch.zeros(5, dtype=torch.int64), bs_col_idx=torch.zeros(1, dtype=torch.int32))
    with pytest.raises(TypeError, match="bs_row_ptr: dtype"):
        v.check(dev, B, Hq, N)
    with pytest.raises(ValueError, match="bs_row_ptr and bs_col_idx are required"):
        af.Variant(mask=af.MASK_BLOCK_SPARSE).check(dev, B, Hq, N)
    v = af.Variant(mask=af.MASK_FULL, bias=af.BIAS_ADDITIVE, add_bias=torch.zeros(3, N, N))
    with pytest.raises(ValueError, match="does not broadcast"):
        v.check(dev, B, Hq, N)
    v = af.Variant(mask=af.MASK_FULL, bias=af.BIAS_ADDITIVE, add_bias=torch.zeros(N, N, dtype=torch.int32))
    with pytest.raises(TypeError, match="add_bias: dtype"):
        v.check(dev, B, Hq, N)
    v = af.Variant(mask=af.MASK_CAUSAL, dbias=torch.zeros(B, Hq, N, N - 1))
    with pytest.raises(ValueError, match="dbias: shape"):
        v.check(dev, B, Hq, N)


class _FakeStream:
    def __init__(self, device, handle):
        self.device, self.cuda_stream = device, handle


def test_calls_run_on_the_tensors_device_and_its_stream(monkeypatch):
    """The C ABI works on the current device; the binding makes the tensors' device current
    and takes that device's stream, so tensors on cuda:1 never reach a launch on cuda:0."""
    seen = {}

    class _Dev:
        def __init__(self, device):
            seen["device"] = device

        def __enter__(self):
            seen["entered"] = True

        def __exit__(self, *exc):
            return False

    monkeypatch.setattr(torch.cuda, "device", _Dev)
    monkeypatch.setattr(torch.cuda, "current_stream",
                        lambda device=None: _FakeStream(device, 1234))
    dev1 = torch.device("cuda", 1)
    ctx, st = af._launch_context(dev1)
    with ctx:
        pass
    assert seen == {"device": dev1, "entered": True}
    assert st.value == 1234
    # an explicit stream of another device is refused
    with pytest.raises(ValueError, match="stream is on cuda:0"):
        af._launch_context(dev1, _FakeStream(torch.device("cuda", 0), 99))
    ctx, st = af._launch_context(dev1, _FakeStream(dev1, 77))
    assert st.value == 77


def test_reuse_table_needs_the_callers_workspace():
    """ROPE_REUSE_TABLE reads the (cos, sin) table from the caller's workspace: a missing or
    too small workspace is refused instead of replaced by a new (table-less) buffer."""
    with pytest.raises(ValueError, match="ROPE_REUSE_TABLE.*got none"):
        af._workspace(4096, torch.device("cuda", 0), None, reuse_table=True)
    small = torch.zeros(100, dtype=torch.uint8)
    with pytest.raises(ValueError, match="ROPE_REUSE_TABLE.*got 100 bytes"):
        af._workspace(4096, torch.device("cuda", 0), small, reuse_table=True)
