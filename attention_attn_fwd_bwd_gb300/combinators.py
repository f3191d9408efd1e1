"""Composable front end: attention variants from the paper's combinators (AttnFuse paper §3.1).

The paper lets a researcher define a variant by composing ten building blocks and compiles
each composition into one fused kernel. Here the CUDA kernels already cover every composition
of the mask and bias combinators, so composing only fills in the arguments of one C-ABI call:
the variant descriptor (attnfuse_variant), the scale and the rope mode.

    attn = attention(rope(theta=5e5), scaled_dot_product(), causal(), alibi(), softmax())
    out = attn(q, k, v)  # q [B, Hq, N, d], k / v [B, Hkv, N, d], bf16 CUDA tensors

The call is differentiable through torch.autograd: its backward runs the library's backward
(dq, dk, dv and, for a full-size additive bias that requires grad, dBias).

Rules of composition (what one library call can express):
  - masks: at most one of full / causal / sliding_window / block_sparse, except that causal
    may restrict sliding_window or block_sparse;
  - biases: at most one of alibi / additive_bias;
  - rope: optional (mode "auto" picks fused or pre-rotated by the measured crossover N*);
  - normaliser: softmax (the default). relu_attention is named by the paper but given no
    semantics, so composing it raises NotImplementedError.
This module only marshals arguments; every step of the computation runs in the library.
"""
from __future__ import annotations

import math

import attention_attn_fwd_bwd_gb300 as af

_ROPE_MODES = {"auto": af.ROPE_AUTO, "fused": af.ROPE_FUSED, "prerotate": af.ROPE_PREROTATE}


class Combinator:
    """One building block: a kind and its parameters."""

    def __init__(self, kind, **params):
        self.kind = kind
        self.params = params

    def __repr__(self):
        args = ", ".join(f"{k}={v!r}" for k, v in self.params.items() if not hasattr(v, "shape"))
        return f"{self.kind}({args})"


def scaled_dot_product(scale=None):
    """s = scale * <q, k>; scale defaults to 1 / sqrt(d)."""
    return Combinator("scaled_dot_product", scale=scale)


def rope(theta=10000.0, mode="auto"):
    """Rotary position embedding of q and k (NeoX half-split pairs), theta_i = theta^(-2i/d).
    mode: "auto", "fused" (rotated on chip) or "prerotate" (a separate rotation pass)."""
    if mode not in _ROPE_MODES:
        raise ValueError(f"rope mode {mode!r}: one of {sorted(_ROPE_MODES)}")
    return Combinator("rope", theta=float(theta), mode=mode)


def causal():
    """Key n visible from query m iff n <= m."""
    return Combinator("causal")


def sliding_window(window):
    """Key n visible from query m iff |m - n| < window (with causal: m - window < n <= m)."""
    if int(window) < 1:
        raise ValueError("window must be >= 1")
    return Combinator("sliding_window", window=int(window))


def full():
    """Every key visible from every query."""
    return Combinator("full")


def block_sparse(row_ptr, col_idx, block=64):
    """Blocks (m // block, n // block) listed in a CSR layout (int32 device tensors, shared by
    every batch and head) are visible; block 64 or 128."""
    if block not in (64, 128):
        raise ValueError("block must be 64 or 128")
    return Combinator("block_sparse", row_ptr=row_ptr, col_idx=col_idx, block=block)


def alibi(slopes=None):
    """s += slope_h * (n - m); slopes: fp32 [Hq] device tensor, default 2^(-8 (h + 1) / Hq)."""
    return Combinator("alibi", slopes=slopes)


def additive_bias(bias):
    """s += bias[b, h, m, n]; bias: fp32 or bf16 device tensor broadcastable to [B, Hq, N, N]."""
    return Combinator("additive_bias", bias=bias)


def softmax():
    """Softmax over the visible keys (the online softmax of the kernels)."""
    return Combinator("softmax")


def relu_attention():
    """ReLU normaliser instead of softmax. The paper names it among its ten combinators without
    a definition; this library reads it as O_m = (1/N) sum_n max(s_mn, 0) v_n over the visible
    keys, N the sequence length. Forward only (no LSE, no gradient); head dim 128."""
    return Combinator("relu_attention")


class Attention:
    """A composed variant; call it on (q, k, v)."""

    def __init__(self, *combinators):
        kinds = [c.kind for c in combinators]
        for c in combinators:
            if not isinstance(c, Combinator):
                raise TypeError(f"not a combinator: {c!r}")
        for k in set(kinds):
            if kinds.count(k) > 1:
                raise ValueError(f"{k} given twice")
        if "relu_attention" in kinds and "softmax" in kinds:
            raise ValueError("one normaliser per variant (softmax or relu_attention)")
        by = {c.kind: c for c in combinators}
        masks = [k for k in ("full", "sliding_window", "block_sparse") if k in by]
        if len(masks) > 1:
            raise ValueError(f"one mask combinator per variant, got {masks}")
        if "full" in by and "causal" in by:
            raise ValueError("full and causal contradict each other")
        if "alibi" in by and "additive_bias" in by:
            raise ValueError("one bias combinator per variant (alibi or additive_bias)")
        self.combinators = combinators
        self.by = by
        self.scale = by["scaled_dot_product"].params["scale"] if "scaled_dot_product" in by else None
        r = by.get("rope")
        self.rope_theta = r.params["theta"] if r else 10000.0
        self.rope_mode = _ROPE_MODES[r.params["mode"]] if r else af.ROPE_NONE
        self.bias = by["additive_bias"].params["bias"] if "additive_bias" in by else None

    def variant(self, Hq, device):
        """The af.Variant (attnfuse_variant) of this composition for Hq query heads."""
        import torch

        by = self.by
        causal_ = "causal" in by
        if "sliding_window" in by:
            v = af.Variant(mask=af.MASK_WINDOW, window=by["sliding_window"].params["window"],
                           causal=causal_)
        elif "block_sparse" in by:
            p = by["block_sparse"].params
            v = af.Variant(mask=af.MASK_BLOCK_SPARSE, bs_block=p["block"], causal=causal_,
                           bs_row_ptr=p["row_ptr"], bs_col_idx=p["col_idx"])
        elif causal_:
            v = af.Variant(mask=af.MASK_CAUSAL)
        else:
            v = af.Variant(mask=af.MASK_FULL)
        if "alibi" in by:
            slopes = by["alibi"].params["slopes"]
            if slopes is None:
                slopes = torch.tensor([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)],
                                      dtype=torch.float32, device=device)
            v.bias, v.alibi_slopes = af.BIAS_ALIBI, slopes
        elif self.bias is not None:
            v.bias, v.add_bias = af.BIAS_ADDITIVE, self.bias
        if "relu_attention" in by:
            v.norm = af.NORM_RELU
        return v

    def __call__(self, q, k, v):
        return _AttnFunction.apply(q, k, v, self.bias, self)

    def __repr__(self):
        return "attention(" + ", ".join(map(repr, self.combinators)) + ")"


def attention(*combinators):
    """Compose combinators into a callable attention variant (the paper's @attention)."""
    return Attention(*combinators)


def _autograd_function():
    import torch

    class _Fn(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q, k, v, bias, spec):
            scale = spec.scale if spec.scale is not None else 1.0 / math.sqrt(q.shape[-1])
            var = spec.variant(q.shape[1], q.device)
            out, lse = af.fwd(q, k, v, scale=scale, rope_theta=spec.rope_theta,
                              rope_mode=spec.rope_mode, variant=var)
            if lse is None:  # relu_attention: forward only
                lse = torch.empty(0, device=q.device)
                ctx.relu = True
            else:
                ctx.relu = False
            ctx.save_for_backward(q, k, v, out, lse)
            ctx.spec, ctx.scale, ctx.bias = spec, scale, bias
            return out

        @staticmethod
        def backward(ctx, dout):
            q, k, v, out, lse = ctx.saved_tensors
            if ctx.relu:
                raise NotImplementedError("relu_attention has no backward in this library")
            spec, bias = ctx.spec, ctx.bias
            var = spec.variant(q.shape[1], q.device)
            dbias = None
            if bias is not None and ctx.needs_input_grad[3]:
                B, Hq, N = q.shape[0], q.shape[1], q.shape[2]
                if tuple(bias.shape) != (B, Hq, N, N):
                    raise NotImplementedError(
                        "gradient of a broadcast additive bias: pass the full [B, Hq, N, N] bias")
                dbias = torch.empty((B, Hq, N, N), dtype=torch.float32, device=q.device)
                var.dbias = dbias
            dq, dk, dv = af.bwd(q, k, v, out, lse, dout.contiguous(), scale=ctx.scale,
                                rope_theta=spec.rope_theta, rope_mode=spec.rope_mode, variant=var)
            if dbias is not None and dbias.dtype != bias.dtype:
                dbias = dbias.to(bias.dtype)
            return dq, dk, dv, dbias, None

    return _Fn


class _LazyFunction:
    _fn = None

    def apply(self, *args):
        if _LazyFunction._fn is None:
            _LazyFunction._fn = _autograd_function()
        return _LazyFunction._fn.apply(*args)


_AttnFunction = _LazyFunction()
