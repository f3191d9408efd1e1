"""attnfuse-gb300: fused RoPE + variant attention for NVIDIA GB300 (sm_103a).

Thin Python binding over the C ABI declared in ``include/attnfuse.h`` (ctypes; argument
marshalling only — every step of the computation runs in the library's CUDA kernels).
PyTorch supplies device memory and streams. There is no CPU fallback: every call raises
if ``libattnfuse.so`` is missing or fails to load.

Low-level functions carry the C names (``attnfuse_fwd`` ...) and take raw pointers; the
torch-level helpers ``fwd``, ``bwd``, ``decode`` and ``rope_prerotate`` allocate outputs and
workspace with torch and call them on the current CUDA stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "ROPE_NONE", "ROPE_FUSED", "ROPE_PREROTATE", "MASK_FULL", "MASK_CAUSAL", "MASK_WINDOW",
    "MASK_BLOCK_SPARSE", "BIAS_NONE", "BIAS_ALIBI", "BIAS_ADDITIVE", "AttnfuseError", "Variant",
    "load", "library_path", "fwd", "bwd", "decode", "rope_prerotate", "device_status",
    "fwd_workspace_size", "bwd_workspace_size", "decode_workspace_size",
]

ROPE_NONE, ROPE_FUSED, ROPE_PREROTATE, ROPE_AUTO = 0, 1, 2, 3
ROPE_REUSE_TABLE = 0x100
MASK_FULL, MASK_CAUSAL, MASK_WINDOW, MASK_BLOCK_SPARSE = 0, 1, 2, 3
BIAS_NONE, BIAS_ALIBI, BIAS_ADDITIVE = 0, 1, 2
NORM_SOFTMAX, NORM_RELU = 0, 1
_STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE_TOO_SMALL",
           4: "CUDA_ERROR", 5: "TIMEOUT", 6: "FP16_RANGE"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libattnfuse.so")
_lock = threading.Lock()
_lib = None


class AttnfuseError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"attnfuse error {code} ({_STATUS.get(code, '?')}): {msg}")
        self.code = code


class CVariant(ctypes.Structure):
    """Mirror of the C struct attnfuse_variant."""
    _fields_ = [
        ("mask", ctypes.c_int32),
        ("causal", ctypes.c_int32),
        ("window", ctypes.c_int32),
        ("bs_block", ctypes.c_int32),
        ("bs_row_ptr", ctypes.c_void_p),
        ("bs_col_idx", ctypes.c_void_p),
        ("bias", ctypes.c_int32),
        ("add_bias_is_bf16", ctypes.c_int32),
        ("alibi_slopes", ctypes.c_void_p),
        ("add_bias", ctypes.c_void_p),
        ("add_bias_strides", ctypes.c_int64 * 4),
        ("tile_visits", ctypes.c_void_p),
        ("dbias", ctypes.c_void_p),
        ("dbias_strides", ctypes.c_int64 * 4),
        ("normalizer", ctypes.c_int32),
        ("bwd_dq_visits", ctypes.c_void_p),
        ("bwd_dkdv_visits", ctypes.c_void_p),
    ]


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libattnfuse.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise AttnfuseError(4, f"{_LIB_PATH} not built; run __graft_entry__.build() or "
                                   f"python -m attention_attn_fwd_bwd_gb300._build")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        ST = ctypes.POINTER(ctypes.c_int64)
        VP = ctypes.POINTER(CVariant)
        sig = {
            "attnfuse_last_error": ([], ctypes.c_char_p),
            "attnfuse_version": ([], I),
            "attnfuse_device_status": ([P, I, ctypes.POINTER(I)], I),
            "attnfuse_fwd_workspace_size": ([I, I, I, I, I, I, ctypes.POINTER(S)], I),
            "attnfuse_fwd": ([P, ST, P, ST, P, ST, P, ST, P, I, I, I, I, I, F, F, I, VP, P, S, P], I),
            "attnfuse_bwd_workspace_size": ([I, I, I, I, I, I, ctypes.POINTER(S)], I),
            "attnfuse_bwd": ([P, ST, P, ST, P, ST, P, ST, P, P, ST, P, ST, P, ST, P, ST,
                              I, I, I, I, I, F, F, I, VP, P, S, P], I),
            "attnfuse_decode_workspace_size": ([I, I, I, I, I, I, ctypes.POINTER(S)], I),
            "attnfuse_decode": ([P, ST, P, ST, P, ST, P, ST, P, I, I, I, I, I, I, F, F, I, I,
                                 P, S, P], I),
            "attnfuse_decode_auto_splits": ([I, I, I, ctypes.POINTER(I)], I),
            "attnfuse_decode_noalloc": ([P, ST, P, ST, P, ST, P, ST, P, I, I, I, I, I, I, F, F, I,
                                         I, P], I),
            "attnfuse_rope_prerotate": ([P, ST, P, I, I, I, I, F, P, S, P], I),
            "attnfuse_debug_wait_timeout": ([ctypes.c_uint64, P], I),
            "attnfuse_rope_table": ([P, S, I, I, F, P], I),
            "attnfuse_rope_auto_mode": ([I, I, I, ctypes.POINTER(I)], I),
            "attnfuse_fwd_fp8_workspace_size": ([I, I, I, I, I, ctypes.POINTER(S)], I),
            "attnfuse_fwd_host_workspace_size": ([I, I, I, I, I, I, I, ctypes.POINTER(S)], I),
            "attnfuse_fwd_host": ([P, P, P, P, P, I, I, I, I, I, F, F, I, VP, I, P, S, P], I),
            "attnfuse_fwd_fp8": ([P, ST, P, ST, P, ST, P, ST, P, I, I, I, I, I, F, F, F, F, VP,
                                  P, S, P], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(rc):
    if rc != 0:
        raise AttnfuseError(rc, load().attnfuse_last_error().decode())


def _strides(t, n):
    arr = (ctypes.c_int64 * n)(*t.stride())
    return arr


def _launch_context(device, stream=None):
    """(context manager, stream handle) for a call whose tensors live on `device`.

    The C ABI works on the current CUDA device (its status word, tensor maps and launches), so
    every call runs with the tensors' device made current and, unless the caller passes one,
    on that device's current stream. A stream of another device is rejected."""
    import torch

    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif stream.device != device:
        raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
    return torch.cuda.device(device), ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(t, name, dtypes, shape=None, device=None, contiguous=False, ndim=None, dims=""):
    """Reject what the C ABI cannot see through a bare pointer: a tensor that is not on the
    CUDA device of the call (its address would reach a kernel), of another element type, of
    another shape, or (where the call takes no strides) not contiguous."""
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: expected {dims}, got shape {tuple(t.shape)}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {' or '.join(str(x) for x in dtypes)}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.device.type != "cuda" or (device is not None and t.device != device):
        raise ValueError(f"{name}: on {t.device}, expected {device or 'a CUDA device'}")


# ------------------------------------------------------------------------------------------
# C names (raw pointers)
# ------------------------------------------------------------------------------------------
def __getattr__(name):
    if name.startswith("attnfuse_"):
        return getattr(load(), name)
    raise AttributeError(name)


# ------------------------------------------------------------------------------------------
# torch-level helpers
# ------------------------------------------------------------------------------------------
class Variant:
    """Combinator set (paper §3.1). Tensors must live on the device of the attention inputs.

    mask: MASK_*; causal: also require n <= m; window: W for MASK_WINDOW; bs_row_ptr /
    bs_col_idx: int32 CSR block layout (block edge bs_block, 64 or 128); bias: BIAS_*;
    alibi_slopes: fp32 [Hq]; add_bias: fp32 or bf16 tensor broadcastable to [B, Hq, N, N];
    tile_visits: uint8 [B, Hq, ceil(N/128), ceil(N/128)] (debug record of computed tiles);
    bwd_dq_visits / bwd_dkdv_visits: the backward's records, uint8 [B, Hq, ceil(N/128),
    ceil(N/128)] (dQ kernel) and [B, Hq, ceil(N/64), ceil(N/128)] (dK/dV kernel, 64-row blocks);
    dbias: fp32 [B, Hq, N, N] output of the backward with an additive bias (its gradient before
    any broadcast is summed out); norm: NORM_SOFTMAX or NORM_RELU (relu_attention: O_m =
    (1/N) sum_n max(s_mn, 0) v_n, forward only, no LSE).
    """

    def __init__(self, mask=MASK_CAUSAL, causal=False, window=0, bs_block=64, bs_row_ptr=None,
                 bs_col_idx=None, bias=BIAS_NONE, alibi_slopes=None, add_bias=None,
                 tile_visits=None, dbias=None, norm=NORM_SOFTMAX, bwd_dq_visits=None,
                 bwd_dkdv_visits=None):
        self.norm = norm
        self.bwd_dq_visits, self.bwd_dkdv_visits = bwd_dq_visits, bwd_dkdv_visits
        self.mask, self.causal, self.window, self.bs_block = mask, causal, window, bs_block
        self.bs_row_ptr, self.bs_col_idx = bs_row_ptr, bs_col_idx
        self.bias, self.alibi_slopes, self.add_bias = bias, alibi_slopes, add_bias
        self.tile_visits = tile_visits
        self.dbias = dbias

    def check(self, device, B, Hq, N):
        """Validate the variant's tensors for a call on `device` with B, Hq and N (lengths
        the kernels index by; the values of a block-sparse layout are the caller's to keep in
        range, since reading them here would synchronise the stream)."""
        import torch

        if self.mask == MASK_BLOCK_SPARSE:
            if self.bs_row_ptr is None or self.bs_col_idx is None:
                raise ValueError("block-sparse variant: bs_row_ptr and bs_col_idx are required")
            if self.bs_block in (64, 128):
                rows = -(-N // self.bs_block)
                if self.bs_row_ptr.numel() < rows + 1:
                    raise ValueError(f"bs_row_ptr: {self.bs_row_ptr.numel()} entries, "
                                     f"the layout has {rows} block rows (needs {rows + 1})")
            _need(self.bs_row_ptr, "bs_row_ptr", (torch.int32,), device=device, contiguous=True)
            _need(self.bs_col_idx, "bs_col_idx", (torch.int32,), device=device, contiguous=True)
        if self.alibi_slopes is not None:
            if self.alibi_slopes.numel() < Hq:
                raise ValueError(f"alibi_slopes: {self.alibi_slopes.numel()} entries for {Hq} heads")
            _need(self.alibi_slopes, "alibi_slopes", (torch.float32,), device=device, contiguous=True)
        if self.add_bias is not None:
            if self.add_bias.dim() > 4:
                raise ValueError("add_bias: at most 4 dimensions ([B, Hq, N, N])")
            full = (B, Hq, N, N)[4 - self.add_bias.dim():]
            for have, want in zip(self.add_bias.shape, full):
                if have not in (1, want):
                    raise ValueError(f"add_bias: shape {tuple(self.add_bias.shape)} does not "
                                     f"broadcast to {(B, Hq, N, N)}")
            _need(self.add_bias, "add_bias", (torch.float32, torch.bfloat16), device=device)
        if self.tile_visits is not None:
            t = -(-N // 128)
            _need(self.tile_visits, "tile_visits", (torch.uint8,), (B, Hq, t, t), device, True)
        if self.dbias is not None:
            _need(self.dbias, "dbias", (torch.float32,), (B, Hq, N, N), device)
        if self.bwd_dq_visits is not None:
            t = -(-N // 128)
            _need(self.bwd_dq_visits, "bwd_dq_visits", (torch.uint8,), (B, Hq, t, t), device, True)
        if self.bwd_dkdv_visits is not None:
            _need(self.bwd_dkdv_visits, "bwd_dkdv_visits", (torch.uint8,),
                  (B, Hq, -(-N // 64), -(-N // 128)), device, True)

    def c_struct(self):
        v = CVariant()
        v.mask, v.causal, v.window, v.bs_block = self.mask, int(bool(self.causal)), self.window, self.bs_block
        if self.bs_row_ptr is not None:
            v.bs_row_ptr, v.bs_col_idx = self.bs_row_ptr.data_ptr(), self.bs_col_idx.data_ptr()
        v.bias = self.bias
        v.normalizer = self.norm
        if self.alibi_slopes is not None:
            v.alibi_slopes = self.alibi_slopes.data_ptr()
        if self.add_bias is not None:
            import torch

            ab = self.add_bias
            while ab.dim() < 4:
                ab = ab.unsqueeze(0)
            v.add_bias = ab.data_ptr()
            v.add_bias_is_bf16 = int(ab.dtype == torch.bfloat16)
            for i in range(4):
                v.add_bias_strides[i] = ab.stride(i) if ab.size(i) > 1 else 0
        if self.tile_visits is not None:
            v.tile_visits = self.tile_visits.data_ptr()
        if self.bwd_dq_visits is not None:
            v.bwd_dq_visits = self.bwd_dq_visits.data_ptr()
        if self.bwd_dkdv_visits is not None:
            v.bwd_dkdv_visits = self.bwd_dkdv_visits.data_ptr()
        if self.dbias is not None:
            v.dbias = self.dbias.data_ptr()
            for i in range(4):
                v.dbias_strides[i] = self.dbias.stride(i)
        return v


def rope_auto_mode(N, d, backward=False):
    """The mode ROPE_AUTO resolves to (ROPE_FUSED or ROPE_PREROTATE) for N and head dim d."""
    m = ctypes.c_int()
    _check(load().attnfuse_rope_auto_mode(N, d, int(bool(backward)), ctypes.byref(m)))
    return m.value


def fwd_workspace_size(B, Hq, Hkv, N, d, rope_mode):
    n = ctypes.c_size_t()
    _check(load().attnfuse_fwd_workspace_size(B, Hq, Hkv, N, d, rope_mode, ctypes.byref(n)))
    return n.value


def fwd_fp8_workspace_size(B, Hq, Hkv, N, d):
    n = ctypes.c_size_t()
    _check(load().attnfuse_fwd_fp8_workspace_size(B, Hq, Hkv, N, d, ctypes.byref(n)))
    return n.value


def bwd_workspace_size(B, Hq, Hkv, N, d, rope_mode):
    n = ctypes.c_size_t()
    _check(load().attnfuse_bwd_workspace_size(B, Hq, Hkv, N, d, rope_mode, ctypes.byref(n)))
    return n.value


def decode_workspace_size(B, Hq, Hkv, L, d, num_splits):
    n = ctypes.c_size_t()
    _check(load().attnfuse_decode_workspace_size(B, Hq, Hkv, L, d, num_splits, ctypes.byref(n)))
    return n.value


def _workspace(nbytes, device, workspace=None, reuse_table=False):
    """The caller's workspace if it holds nbytes, else a new one. With ROPE_REUSE_TABLE the
    (cos, sin) table must already sit in the caller's workspace, so a missing or too small one
    is an error (a new buffer would hold no table)."""
    import torch

    have = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if reuse_table and (workspace is None or have < nbytes):
        raise ValueError(f"ROPE_REUSE_TABLE needs the workspace that holds the table "
                         f"({nbytes} bytes); got {'none' if workspace is None else f'{have} bytes'}")
    if nbytes == 0:
        return None
    if workspace is not None:
        _need(workspace, "workspace", (workspace.dtype,), device=device)
        if have >= nbytes:
            return workspace
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def fwd(q, k, v, scale=None, rope_theta=10000.0, rope_mode=ROPE_FUSED, variant=None,
        out=None, lse=None, with_lse=True, workspace=None, stream=None):
    """Forward: q [B,Hq,N,d], k/v [B,Hkv,N,d] bf16 CUDA tensors -> (out, lse)."""
    import torch

    bf16, f32 = (torch.bfloat16,), (torch.float32,)
    _need(q, "q", bf16, ndim=4, dims="[B, Hq, N, d]")
    B, Hq, N, d = q.shape
    dev = q.device
    _need(k, "k", bf16, ndim=4, dims="[B, Hkv, N, d]")
    Hkv = k.shape[1]
    _need(k, "k", bf16, (B, Hkv, N, d), dev)
    _need(v, "v", bf16, (B, Hkv, N, d), dev)
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", bf16, (B, Hq, N, d), dev)
    relu = variant is not None and variant.norm == NORM_RELU
    if relu and lse is not None:
        raise ValueError("relu_attention has no LSE: pass lse=None")
    if with_lse and lse is None and not relu:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", f32, (B, Hq, N), dev, contiguous=True)
    if variant is not None:
        variant.check(dev, B, Hq, N)
    ws_n = fwd_workspace_size(B, Hq, Hkv, N, d, rope_mode & 0xFF)
    ws = _workspace(ws_n, dev, workspace, bool(rope_mode & ROPE_REUSE_TABLE))
    cv = (variant or Variant()).c_struct()
    ctx, st = _launch_context(dev, stream)
    with ctx:
        _check(load().attnfuse_fwd(
            _ptr(q), _strides(q, 4), _ptr(k), _strides(k, 4), _ptr(v), _strides(v, 4),
            _ptr(out), _strides(out, 4), _ptr(lse), B, Hq, Hkv, N, d, float(scale),
            float(rope_theta), rope_mode, ctypes.byref(cv), _ptr(ws), ws_n, st))
    return out, lse


def fwd_host_workspace_size(B, Hq, Hkv, N, d, rope_mode, chunk_b):
    n = ctypes.c_size_t()
    _check(load().attnfuse_fwd_host_workspace_size(B, Hq, Hkv, N, d, rope_mode, chunk_b,
                                                   ctypes.byref(n)))
    return n.value


def fwd_host(q, k, v, scale=None, rope_theta=10000.0, rope_mode=ROPE_FUSED, variant=None,
             out=None, lse=None, with_lse=True, chunk_b=1, workspace=None, device=None,
             stream=None, sync=True):
    """Forward on CPU tensors (contiguous bf16; pinned memory lets the copies overlap): the
    batch is copied in, attended and copied out in chunks of chunk_b elements, the copies of
    one chunk overlapping the forward of the next. Returns CPU (out, lse); with sync=False the
    results are valid once the device stream has reached this point."""
    import torch

    bf16, f32 = (torch.bfloat16,), (torch.float32,)
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
            raise ValueError(f"{name}: expected a CPU tensor")
        if t.dtype not in bf16:
            raise TypeError(f"{name}: dtype {t.dtype}, expected torch.bfloat16")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name}: expected a contiguous [B, H, N, d] tensor")
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (B, Hkv, N, d) or tuple(v.shape) != (B, Hkv, N, d):
        raise ValueError("k, v: expected [B, Hkv, N, d] matching q")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if scale is None:
        scale = d ** -0.5
    pin = q.is_pinned()
    if out is None:
        out = torch.empty((B, Hq, N, d), dtype=torch.bfloat16, pin_memory=pin)
    relu = variant is not None and variant.norm == NORM_RELU
    if with_lse and lse is None and not relu:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, pin_memory=pin)
    for t, name, dt, shape in ((out, "out", bf16, (B, Hq, N, d)), (lse, "lse", f32, (B, Hq, N))):
        if t is None:
            continue
        if t.device.type != "cpu" or t.dtype not in dt or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name}: expected a contiguous CPU {dt[0]} tensor of shape {shape}")
    if variant is not None:
        variant.check(dev, B, Hq, N)
    ws_n = fwd_host_workspace_size(B, Hq, Hkv, N, d, rope_mode, chunk_b)
    ws = _workspace(ws_n, dev, workspace)
    cv = (variant or Variant()).c_struct()
    ctx, st = _launch_context(dev, stream)
    with ctx:
        _check(load().attnfuse_fwd_host(
            _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, N, d, float(scale),
            float(rope_theta), rope_mode, ctypes.byref(cv), int(chunk_b), _ptr(ws), ws_n, st))
        if sync:
            torch.cuda.current_stream(dev).synchronize() if stream is None else stream.synchronize()
    return out, lse


def fwd_fp8(q, k, v, q_scale, k_scale, v_scale, scale=None, variant=None, out=None, lse=None,
            with_lse=True, workspace=None, stream=None):
    """e4m3 forward (head dim 128): q [B,Hq,N,128], k/v [B,Hkv,N,128] as torch.uint8 (raw
    e4m3 bytes) or torch.float8_e4m3fn CUDA tensors; attends over q_scale*q, k_scale*k and
    v_scale*v; returns (out bf16, lse fp32). No RoPE: q and k are used as given."""
    import torch

    f8 = tuple(t for t in (torch.uint8, getattr(torch, "float8_e4m3fn", None)) if t is not None)
    bf16, f32 = (torch.bfloat16,), (torch.float32,)
    _need(q, "q", f8, ndim=4, dims="[B, Hq, N, d]")
    B, Hq, N, d = q.shape
    dev = q.device
    _need(k, "k", f8, ndim=4, dims="[B, Hkv, N, d]")
    Hkv = k.shape[1]
    _need(k, "k", f8, (B, Hkv, N, d), dev)
    _need(v, "v", f8, (B, Hkv, N, d), dev)
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty((B, Hq, N, d), dtype=torch.bfloat16, device=dev)
    _need(out, "out", bf16, (B, Hq, N, d), dev)
    relu = variant is not None and variant.norm == NORM_RELU
    if relu and lse is not None:
        raise ValueError("relu_attention has no LSE: pass lse=None")
    if with_lse and lse is None and not relu:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    if lse is not None:
        _need(lse, "lse", f32, (B, Hq, N), dev, contiguous=True)
    if variant is not None:
        variant.check(dev, B, Hq, N)
    ws_n = fwd_fp8_workspace_size(B, Hq, Hkv, N, d)
    ws = _workspace(ws_n, dev, workspace)
    cv = (variant or Variant()).c_struct()
    ctx, st = _launch_context(dev, stream)
    with ctx:
        _check(load().attnfuse_fwd_fp8(
            _ptr(q), _strides(q, 4), _ptr(k), _strides(k, 4), _ptr(v), _strides(v, 4),
            _ptr(out), _strides(out, 4), _ptr(lse), B, Hq, Hkv, N, d, float(scale),
            float(q_scale), float(k_scale), float(v_scale), ctypes.byref(cv), _ptr(ws), ws_n, st))
    return out, lse


def bwd(q, k, v, out, lse, dout, scale=None, rope_theta=10000.0, rope_mode=ROPE_FUSED,
        variant=None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward (paper §4.4): returns (dq, dk, dv) w.r.t. the un-rotated q, k and v."""
    import torch

    bf16, f32 = (torch.bfloat16,), (torch.float32,)
    _need(q, "q", bf16, ndim=4, dims="[B, Hq, N, d]")
    B, Hq, N, d = q.shape
    dev = q.device
    _need(k, "k", bf16, ndim=4, dims="[B, Hkv, N, d]")
    Hkv = k.shape[1]
    _need(k, "k", bf16, (B, Hkv, N, d), dev)
    _need(v, "v", bf16, (B, Hkv, N, d), dev)
    _need(out, "out", bf16, (B, Hq, N, d), dev)
    _need(lse, "lse", f32, (B, Hq, N), dev, contiguous=True)
    _need(dout, "dout", bf16, (B, Hq, N, d), dev)
    if scale is None:
        scale = d ** -0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _need(dq, "dq", bf16, (B, Hq, N, d), dev)
    _need(dk, "dk", bf16, (B, Hkv, N, d), dev)
    _need(dv, "dv", bf16, (B, Hkv, N, d), dev)
    if variant is not None:
        variant.check(dev, B, Hq, N)
    ws_n = bwd_workspace_size(B, Hq, Hkv, N, d, rope_mode & 0xFF)
    ws = _workspace(ws_n, dev, workspace, bool(rope_mode & ROPE_REUSE_TABLE))
    cv = (variant or Variant()).c_struct()
    ctx, st = _launch_context(dev, stream)
    with ctx:
        _check(load().attnfuse_bwd(
            _ptr(q), _strides(q, 4), _ptr(k), _strides(k, 4), _ptr(v), _strides(v, 4),
            _ptr(out), _strides(out, 4), _ptr(lse), _ptr(dout), _strides(dout, 4),
            _ptr(dq), _strides(dq, 4), _ptr(dk), _strides(dk, 4), _ptr(dv), _strides(dv, 4),
            B, Hq, Hkv, N, d, float(scale), float(rope_theta), rope_mode, ctypes.byref(cv),
            _ptr(ws), ws_n, st))
    return dq, dk, dv


def decode(q, k_cache, v_cache, q_pos, scale=None, rope_theta=10000.0, rope_mode=ROPE_FUSED,
           num_splits=0, out=None, lse=None, with_lse=True, workspace=None, stream=None):
    """Split-KV decode (paper §4.2): q [B,Hq,d], caches [B,Hkv,L,d] -> (out [B,Hq,d], lse)."""
    import torch

    bf16 = (torch.bfloat16,)
    _need(q, "q", bf16, ndim=3, dims="[B, Hq, d]")
    B, Hq, d = q.shape
    dev = q.device
    _need(k_cache, "k_cache", bf16, ndim=4, dims="[B, Hkv, L, d]")
    Hkv, L = k_cache.shape[1], k_cache.shape[2]
    _need(k_cache, "k_cache", bf16, (B, Hkv, L, d), dev)
    _need(v_cache, "v_cache", bf16, (B, Hkv, L, d), dev)
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", bf16, (B, Hq, d), dev)
    if with_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", (torch.float32,), (B, Hq), dev, contiguous=True)
    ws_n = decode_workspace_size(B, Hq, Hkv, L, d, num_splits)
    ws = _workspace(ws_n, dev, workspace)
    ctx, st = _launch_context(dev, stream)
    with ctx:
        _check(load().attnfuse_decode(
            _ptr(q), _strides(q, 3), _ptr(k_cache), _strides(k_cache, 4), _ptr(v_cache),
            _strides(v_cache, 4), _ptr(out), _strides(out, 3), _ptr(lse), B, Hq, Hkv, L, d,
            int(q_pos), float(scale), float(rope_theta), rope_mode, int(num_splits), _ptr(ws),
            ws_n, st))
    return out, lse


def decode_auto_splits(B, Hkv, L):
    n = ctypes.c_int()
    _check(load().attnfuse_decode_auto_splits(B, Hkv, L, ctypes.byref(n)))
    return n.value


def rope_prerotate(x, rope_theta, out=None, workspace=None, stream=None):
    """x [B,H,N,d] bf16 -> R_n x (contiguous)."""
    import torch

    _need(x, "x", (torch.bfloat16,), ndim=4, dims="[B, H, N, d]")
    B, H, N, d = x.shape
    out = torch.empty((B, H, N, d), dtype=x.dtype, device=x.device) if out is None else out
    _need(out, "out", (torch.bfloat16,), (B, H, N, d), x.device, contiguous=True)
    ws_n = fwd_workspace_size(B, H, H, N, d, ROPE_FUSED)
    ws = _workspace(ws_n, x.device, workspace)
    ctx, st = _launch_context(x.device, stream)
    with ctx:
        _check(load().attnfuse_rope_prerotate(_ptr(x), _strides(x, 4), _ptr(out), B, H, N, d,
                                              float(rope_theta), _ptr(ws), ws_n, st))
    return out


def device_status(clear=True, stream=None, device=None):
    """Synchronise and return the device status of `device` (default: the stream's device,
    else the current device): 0 OK, 5 TIMEOUT (a kernel gave up waiting), 6 FP16_RANGE (a
    rotating-mode forward saturated an fp16 Q' / K' element or met a non-finite input)."""
    import torch

    if device is None:
        device = stream.device if stream is not None else torch.device("cuda", torch.cuda.current_device())
    code = ctypes.c_int()
    ctx, st = _launch_context(device, stream)
    with ctx:
        _check(load().attnfuse_device_status(st, int(clear), ctypes.byref(code)))
    return code.value
